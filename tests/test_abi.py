"""Host-side checks of the C ABI: the library builds, loads and exports every
symbol include/fa.h declares, and argument validation rejects bad calls
before touching the GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

from io_aware_attention_flash_gb300 import _binding
from io_aware_attention_flash_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    return sorted(set(re.findall(r"^FA_API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return _binding.lib()


def test_header_declares_the_abi():
    names = _declared_symbols()
    assert {"fa_fwd", "fa_bwd", "fa_fwd_varlen", "fa_bwd_varlen", "fa_bwd_workspace_bytes",
            "fa_bwd_varlen_workspace_bytes", "fa_get_device_error", "fa_status_string"} <= set(names)
    assert set(names) == set(_binding.SIGNATURES), "binding and header disagree"


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_symbols():
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr), name


def test_only_abi_symbols_are_exported(lib):
    # -fvisibility=hidden: the dynamic symbol table holds the fa_* entry points only.
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(_declared_symbols()) <= exported
    assert all(s.startswith("fa_") or s.startswith("_") for s in exported), sorted(exported)[:20]


def test_status_strings(lib):
    for code in range(0, 11):
        assert lib.fa_status_string(code)
    assert lib.fa_status_string(3).decode().startswith("head dim")


FAKE = 0x10000  # aligned host-looking address; validation fails before it is used
NUL = None


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, scale=0.125, causal=0):
    return lib.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, None)


def test_fwd_validation(lib):
    assert _fwd(lib, d=96) == 3
    assert _fwd(lib, d=256) == 3
    assert _fwd(lib, N=0) == 4
    assert _fwd(lib, B=-1) == 4
    assert _fwd(lib, H=0) == 4
    assert _fwd(lib, q=NUL) == 1
    assert _fwd(lib, lse=NUL) == 1
    assert _fwd(lib, k=FAKE + 8) == 2
    assert _fwd(lib, o=FAKE + 2) == 2
    assert _fwd(lib, scale=float("inf")) == 9
    assert _fwd(lib, scale=float("nan")) == 9


def test_bwd_validation(lib):
    ws = lib.fa_bwd_workspace_bytes(1, 2, 100, 64)
    # D: 1*2*100 floats -> 800 -> 1024; dQ accum: 100 rows -> 128, 128*2*64*4 = 65536
    assert ws == 1024 + 65536

    def bwd(ws_ptr=FAKE, ws_bytes=ws, d=64, dq=FAKE):
        return lib.fa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dq, FAKE, FAKE, ws_ptr, ws_bytes,
                          1, 2, 100, d, 0.125, 1, None)

    assert bwd(ws_bytes=ws - 1) == 8
    assert bwd(ws_ptr=NUL) == 8
    assert bwd(ws_ptr=FAKE + 4) == 2
    assert bwd(d=32) == 3
    assert bwd(dq=NUL) == 1


def test_varlen_validation(lib):
    ws = lib.fa_bwd_varlen_workspace_bytes(1000, 3, 500, 4, 128)
    assert ws == (3 * 4 * 500 * 4 + 255) // 256 * 256 + 1024 * 4 * 128 * 4
    f = lib.fa_fwd_varlen
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, NUL, 3, 500, 1000, 4, 128, 0.1, 1, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 500, 1000, 4, 128, 0.1, 1, None) == 4
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 3, 0, 1000, 4, 128, 0.1, 1, None) == 4
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 3, 500, 1000, 4, 80, 0.1, 1, None) == 3


def test_valid_arguments_without_gpu_report_cuda_or_arch(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU tests cover valid calls")
    assert _fwd(lib) in (5, 6, 10)


def test_noalloc_limit_matches_header_and_rejects_on_host(lib):
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    m = re.search(r"#define FA_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == _binding.NOALLOC_SCRATCH_BYTES
    # 33.8 MB of workspace needed: rejected before any CUDA call
    assert lib.fa_bwd_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                              1, 16, 4096, 128, 0.1, 1, None) == 11


def test_decode_validation(lib):
    ws = lib.fa_decode_workspace_bytes(2, 4, 3, 1000, 128)
    assert ws > 0 and ws % 256 == 0
    assert lib.fa_decode_workspace_bytes(2, 4, 0, 1000, 128) == 0
    assert lib.fa_decode_workspace_bytes(2, 4, 9, 1000, 128) == 0
    assert lib.fa_decode_workspace_bytes(2, 4, 3, 0, 128) == 0
    assert lib.fa_decode_workspace_bytes(2, 4, 3, 1000, 96) == 0
    # one query per partial more costs more workspace; a longer cache never less
    assert lib.fa_decode_workspace_bytes(2, 4, 4, 1000, 128) > ws
    assert lib.fa_decode_workspace_bytes(2, 4, 3, 5000, 128) >= ws

    def dec(Nq=3, Nk=1000, d=128, ws_ptr=FAKE, ws_bytes=ws, q=FAKE):
        return lib.fa_fwd_decode(q, FAKE, FAKE, FAKE, FAKE, ws_ptr, ws_bytes, 2, 4, Nq, Nk, d, 0.1, 1, None)

    assert dec(Nq=0) == 4
    assert dec(Nq=9) == 4
    assert dec(Nk=0) == 4
    assert dec(d=96) == 3
    assert dec(q=NUL) == 1
    assert dec(ws_ptr=NUL) == 1
    assert dec(ws_ptr=FAKE + 8) == 2
    assert dec(ws_bytes=ws - 1) == 8
