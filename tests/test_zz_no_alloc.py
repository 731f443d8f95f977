"""fa_bwd_noalloc — the backward for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace: a plugin inside a
host framework that owns all device memory, or a latency-critical path where
allocation is not allowed.  fa_bwd_noalloc serves them from a static device
array inside the library.  This test calls it through the C ABI twice in a
row on the same inputs and compares each result with the ordinary fa_bwd
(caller workspace) within the gradient tolerance the other tests use.  A
second call that re-used stale accumulator contents from the first would
double dQ and fail.  The file is named to be collected last, and it needs no
state from other tests.
"""
import ctypes

import torch

from io_aware_attention_flash_gb300 import workloads as wl
from tests.gpu_util import GRAD_RTOL, f64, gpu, rel_fro, require_gpu

pytestmark = gpu


def test_noalloc_backward_matches_workspace_backward_twice():
    fa = require_gpu()
    lib = fa.load_library()
    B, N, H, d = 2, 1000, 4, 128        # needs ~4.1 MB of scratch
    causal = True
    scale = d ** -0.5
    q, k, v, do = (t.cuda() for t in wl.make_inputs(B, N, H, d, seed=77))
    o, lse = fa.attention_forward(q, k, v, causal)
    ref = fa.attention_backward(q, k, v, o, do, lse, causal)   # the existing entry point, with a workspace
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        status = lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                    lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                    B, H, N, d, scale, int(causal), stream)
        assert status == 0, fa.FaError("fa_bwd_noalloc", status)
        torch.cuda.synchronize()
        assert fa.fa_get_device_error() == 0
        for got, want in zip((dq, dk, dv), ref):
            assert rel_fro(f64(got), f64(want)) <= GRAD_RTOL


def test_noalloc_rejects_problems_beyond_its_scratch():
    fa = require_gpu()
    lib = fa.load_library()
    x = torch.zeros(1, 128, 1, 128, device="cuda", dtype=torch.bfloat16)
    lse = torch.zeros(1, 1, 128, device="cuda")
    B, H, N, d = 1, 16, 4096, 128       # workspace 33.8 MB > 32 MiB
    assert fa.fa_bwd_workspace_bytes(B, H, N, d) > fa._binding.NOALLOC_SCRATCH_BYTES
    status = lib.fa_bwd_noalloc(x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                lse.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), B, H, N, d, 0.1, 1, None)
    assert status == 11  # FA_ERR_SCRATCH_LIMIT, rejected before anything is enqueued
    assert fa.fa_get_device_error() == 0
