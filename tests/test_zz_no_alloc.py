"""fa_bwd_noalloc — the backward for callers that cannot allocate device memory.

Some callers have no way to hand the library a workspace: a plugin inside a
host framework that owns all device memory, or a latency-critical path where
allocation is not allowed.  fa_bwd_noalloc serves them from a static device
array inside the library.  This test calls it through the C ABI twice in a
row on the same inputs and compares each result with the ordinary fa_bwd
(caller workspace): dK and dV bit for bit (no reduction order is involved in
them), dQ to 1e-3 (its fp32 accumulation order varies from run to run, so a
few outputs may round to a neighbouring bf16 value; a stale accumulator or a
dropped contribution is far larger).  Each result is also checked against
the fp64 oracle, and the second call must not change the device memory in
use (torch's allocator and the driver's free-memory count).  The file is
named to be collected last, and it needs no state from other tests.
"""
import ctypes

import torch

import oracle
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
    oref = oracle.backward(*(f64(t) for t in (q, k, v, do)), scale, causal)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = [tuple(torch.empty_like(t) for t in (q, k, v)) for _ in range(2)]
    torch.cuda.synchronize()
    in_use = []
    for dq, dk, dv in outs:
        status = lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                    lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                    B, H, N, d, scale, int(causal), stream)
        assert status == 0, fa.FaError("fa_bwd_noalloc", status)
        torch.cuda.synchronize()
        # Device memory in use after each call, taken before any other work
        # that could allocate (the first call may load the library's kernels;
        # the second must not move either figure).
        in_use.append((torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]))
    assert in_use[1] == in_use[0], in_use
    assert fa.fa_get_device_error() == 0
    for dq, dk, dv in outs:
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
        assert rel_fro(f64(dq), f64(ref[0])) <= 1e-3
        for got, want in zip((dq, dk, dv), oref):
            assert rel_fro(f64(got), want) <= GRAD_RTOL


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
