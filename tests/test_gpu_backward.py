"""Backward parity: CUDA path vs the fp64 oracle on the same seeded bf16
inputs.  The CUDA backward consumes the CUDA forward's O and LSE (as a caller
would); the oracle recomputes everything from Q, K, V, dO."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_attention_flash_gb300 import workloads as wl
from tests.gpu_util import GRAD_RTOL, assert_no_device_error, f64, gpu, rel_fro, require_gpu

pytestmark = gpu

SHAPES = [
    (1, 1, 1, 64), (1, 2, 127, 64), (2, 3, 129, 128), (1, 2, 256, 128), (2, 2, 300, 64), (1, 3, 513, 128),
    (1, 2, 1000, 64),
]


def _run(fa, q, k, v, do, causal, scale=None):
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention_forward(qc, kc, vc, causal, scale)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, doc, lse, causal, scale)
    torch.cuda.synchronize()
    assert_no_device_error(fa)
    return f64(dq), f64(dk), f64(dv)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", SHAPES)
def test_backward_matches_oracle(B, H, N, d, causal):
    fa = require_gpu()
    q, k, v, do = wl.make_inputs(B, N, H, d, seed=2 * N + d)
    dq, dk, dv = _run(fa, q, k, v, do, causal)
    DQ, DK, DV = oracle.backward(f64(q), f64(k), f64(v), f64(do), d ** -0.5, causal)
    for name, got, ref in (("dq", dq, DQ), ("dk", dk, DK), ("dv", dv, DV)):
        assert rel_fro(got, ref) <= GRAD_RTOL, (name, rel_fro(got, ref))


@pytest.mark.parametrize("name", ["tiny", "small", "small_noncausal"])
def test_backward_small_workloads_full(name):
    fa = require_gpu()
    w = wl.WORKLOADS[name]
    q, k, v, do = wl.workload_inputs(w, seed=0)
    dq, dk, dv = _run(fa, q, k, v, do, w.causal)
    DQ, DK, DV = oracle.backward(f64(q), f64(k), f64(v), f64(do), w.scale, w.causal)
    for nm, got, ref in (("dq", dq, DQ), ("dk", dk, DK), ("dv", dv, DV)):
        assert rel_fro(got, ref) <= GRAD_RTOL, (nm, rel_fro(got, ref))


@pytest.mark.parametrize("name", ["mid_n4096_d128", "long_n32768"])
def test_backward_full_size_sampled(name):
    """Full-size workload in the benchmark's launch configuration.  Sampled
    dQ rows anywhere; dK/dV rows from the tail of the sequence (causal: few
    query rows see them) and a few from the start for one head; invariants
    that hold at any size on every head."""
    fa = require_gpu()
    w = wl.WORKLOADS[name]
    q, k, v, do = wl.workload_inputs(w, seed=0)
    dq, dk, dv = _run(fa, q, k, v, do, w.causal)
    qd, kd, vd, dod = f64(q), f64(k), f64(v), f64(do)
    rng = np.random.default_rng(7)
    for b, h in [(0, 0), (w.B - 1, w.H - 1)]:
        rows = np.unique(np.concatenate([[0, 127, 128, w.N - 1], rng.integers(0, w.N, 24)]))
        keys = np.unique(np.concatenate([[w.N - 1, w.N - 128, w.N - 129], rng.integers(w.N - 256, w.N, 12)]))
        DQ, DK, DV = oracle.backward_rows(qd, kd, vd, dod, w.scale, w.causal, b, h, rows, keys)
        assert rel_fro(dq[b, rows, h], DQ) <= GRAD_RTOL
        assert rel_fro(dk[b, keys, h], DK) <= GRAD_RTOL
        assert rel_fro(dv[b, keys, h], DV) <= GRAD_RTOL
    if w.N <= 4096:
        keys = np.array([0, 1, 127, 128, 1000])
        _, DK, DV = oracle.backward_rows(qd, kd, vd, dod, w.scale, w.causal, 0, 1, [], keys)
        assert rel_fro(dk[0, keys, 1], DK) <= GRAD_RTOL
        assert rel_fro(dv[0, keys, 1], DV) <= GRAD_RTOL
    # Rows of P sum to one: sum_j dV_j = sum_i dO_i.  Rows of dS sum to zero:
    # sum_j dK_j = 0.  Both per (batch, head), at full size.
    sdv, sdo = dv.sum(axis=1), dod.sum(axis=1)
    assert np.abs(sdv - sdo).max() <= 2e-2 * np.abs(sdo).max() + 1e-2 * np.sqrt(w.N)
    sdk = dk.sum(axis=1)
    assert np.abs(sdk).max() <= 2e-2 * np.abs(dk).max() * np.sqrt(w.N)
    assert np.isfinite(dq).all() and np.isfinite(dk).all() and np.isfinite(dv).all()


@pytest.mark.slow
def test_backward_long_first_key_tile():
    """long_n32768 (B=1, H=8, N=32768, causal): dK and dV of the first key
    tile (keys 0-127) of one head against the oracle.  These are the heaviest
    key tiles of the launch: their loop runs all 256 query tiles, wrapping
    the Q/dO ring and the dQ staging many times, and every query row of the
    sequence contributes to them (the oracle's cost is the full N x N
    attention of the head)."""
    fa = require_gpu()
    w = wl.WORKLOADS["long_n32768"]
    q, k, v, do = wl.workload_inputs(w, seed=0)
    dq, dk, dv = _run(fa, q, k, v, do, w.causal)
    h = 5
    one = (slice(None), slice(None), slice(h, h + 1), slice(None))
    keys = np.arange(128)
    _, DK, DV = oracle.backward_rows(f64(q[one]), f64(k[one]), f64(v[one]), f64(do[one]), w.scale, w.causal,
                                     0, 0, [], keys)
    assert rel_fro(dk[0, keys, h], DK) <= GRAD_RTOL
    assert rel_fro(dv[0, keys, h], DV) <= GRAD_RTOL


def test_backward_repeatable_and_workspace_reuse():
    """dQ is accumulated by unordered reduce-adds: results vary only by rounding order;
    a dirty reused workspace must not leak into the result."""
    fa = require_gpu()
    B, N, H, d = 1, 640, 2, 128
    q, k, v, do = wl.make_inputs(B, N, H, d, seed=99)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention_forward(qc, kc, vc, True)
    ws = torch.full((fa.fa_bwd_workspace_bytes(B, H, N, d),), 0x7F, device="cuda", dtype=torch.uint8)
    r1 = fa.attention_backward(qc, kc, vc, o, doc, lse, True, workspace=ws)
    r2 = fa.attention_backward(qc, kc, vc, o, doc, lse, True, workspace=ws)
    for a, b in zip(r1, r2):
        assert rel_fro(f64(a), f64(b)) <= 1e-2
    DQ, DK, DV = oracle.backward(f64(q), f64(k), f64(v), f64(do), d ** -0.5, True)
    for got, ref in zip(r2, (DQ, DK, DV)):
        assert rel_fro(f64(got), ref) <= GRAD_RTOL


def test_backward_calls_back_to_back_share_a_workspace():
    """Two backward calls on different inputs, queued with no synchronisation
    in between and one workspace: the second call's pre-pass zeroes the fp32
    accumulator that the first call's conversion reads, and each call's main
    kernel may start before its pre-pass has finished (programmatic dependent
    launch).  Both results against the oracle."""
    fa = require_gpu()
    B, N, H, d = 1, 515, 3, 128
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), device="cuda", dtype=torch.uint8)
    runs = []
    for seed in (21, 22):
        q, k, v, do = wl.make_inputs(B, N, H, d, seed=seed)
        qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
        o, lse = fa.attention_forward(qc, kc, vc, True)
        runs.append(((q, k, v, do), fa.attention_backward(qc, kc, vc, o, doc, lse, True, workspace=ws)))
    torch.cuda.synchronize()
    assert_no_device_error(fa)
    for (q, k, v, do), grads in runs:
        ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), d ** -0.5, True)
        for got, r in zip(grads, ref):
            assert rel_fro(f64(got), r) <= GRAD_RTOL


def test_backward_with_main_kernel_events():
    """With the main kernel's own timing events requested, the backward's
    kernels are launched one after another without overlap; same results,
    and the events bracket a positive time."""
    fa = require_gpu()
    B, N, H, d = 2, 384, 2, 64
    q, k, v, do = wl.make_inputs(B, N, H, d, seed=31)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention_forward(qc, kc, vc, False)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fa.fa_set_kernel_events(e0, e1)
    grads = fa.attention_backward(qc, kc, vc, o, doc, lse, False)
    torch.cuda.synchronize()
    assert_no_device_error(fa)
    assert e0.elapsed_time(e1) > 0
    ref = oracle.backward(f64(q), f64(k), f64(v), f64(do), d ** -0.5, False)
    for got, r in zip(grads, ref):
        assert rel_fro(f64(got), r) <= GRAD_RTOL


def test_autograd_function():
    fa = require_gpu()
    B, N, H, d = 1, 300, 2, 64
    q, k, v, do = wl.make_inputs(B, N, H, d, seed=4)
    tq, tk, tv = (t.cuda().requires_grad_() for t in (q, k, v))
    out = fa.flash_attention(tq, tk, tv, causal=True)
    out.backward(do.cuda())
    DQ, DK, DV = oracle.backward(f64(q), f64(k), f64(v), f64(do), d ** -0.5, True)
    assert rel_fro(f64(tq.grad), DQ) <= GRAD_RTOL
    assert rel_fro(f64(tk.grad), DK) <= GRAD_RTOL
    assert rel_fro(f64(tv.grad), DV) <= GRAD_RTOL


def test_concurrent_streams_with_separate_workspaces():
    """Two problems of different shapes (d = 128 causal and d = 64
    non-causal), each forward and backward on a stream of its own with its
    own workspace, queued interleaved with no synchronisation: the library's
    per-device state (shared-memory limits, error word) is shared by both
    streams, their kernels may overlap on the GPU, and each result must still
    match the oracle."""
    fa = require_gpu()
    from io_aware_attention_flash_gb300 import _binding as bnd

    probs = [(1, 2, 384, 128, True, 31), (2, 3, 200, 64, False, 32)]
    bufs = []
    for B, H, N, d, causal, seed in probs:
        q, k, v, do = wl.make_inputs(B, N, H, d, seed=seed)
        dev = [t.cuda() for t in (q, k, v, do)]
        o = torch.empty_like(dev[0])
        lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
        grads = [torch.empty_like(t) for t in dev[:3]]
        ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), device="cuda", dtype=torch.uint8)
        bufs.append(((q, k, v, do), dev, o, lse, grads, ws, causal, d))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for (_, (qc, kc, vc, doc), o, lse, g, ws, causal, d), s in zip(bufs, streams):
        bnd.fa_fwd(qc, kc, vc, o, lse, causal, stream=s)
    for (_, (qc, kc, vc, doc), o, lse, g, ws, causal, d), s in zip(bufs, streams):
        bnd.fa_bwd(qc, kc, vc, o, doc, lse, g[0], g[1], g[2], ws, causal, stream=s)
    torch.cuda.synchronize()
    assert_no_device_error(fa)
    for (q, k, v, do), _, o, lse, g, ws, causal, d in bufs:
        O, L = oracle.forward(f64(q), f64(k), f64(v), d ** -0.5, causal)
        assert np.abs(f64(o) - O).max() <= 1e-2
        DQ, DK, DV = oracle.backward(f64(q), f64(k), f64(v), f64(do), d ** -0.5, causal)
        for got, ref in zip(g, (DQ, DK, DV)):
            assert rel_fro(f64(got), ref) <= GRAD_RTOL
