"""fp64 CPU oracle for exact softmax attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline
leg and ``--impl reference`` arm may import this package.  It shares no code
with the CUDA path.  See ``oracle/attention.py`` for the definitions followed.
"""
from .attention import (  # noqa: F401
    PANEL_ROWS,
    backward,
    backward_rows,
    backward_varlen,
    decode_mask,
    forward,
    forward_decode,
    forward_rows,
    forward_varlen,
    softmax_rows,
    visible_mask,
)
