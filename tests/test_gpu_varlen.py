"""Packed variable-length batches (cu_seqlens): parity with the fp64 oracle,
no attention across sequence boundaries, no writes outside a sequence."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_attention_flash_gb300 import workloads as wl
from tests.gpu_util import GRAD_RTOL, LSE_ATOL, O_ATOL, assert_no_device_error, f64, gpu, rel_fro, require_gpu

pytestmark = gpu


def _run(fa, cu, q, k, v, do, causal, max_len):
    cu_d = cu.cuda()
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention_forward_varlen(qc, kc, vc, cu_d, max_len, causal)
    dq, dk, dv = fa.attention_backward_varlen(qc, kc, vc, o, doc, lse, cu_d, max_len, causal)
    torch.cuda.synchronize()
    assert_no_device_error(fa)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_varlen_ragged_lengths_full(causal, d):
    fa = require_gpu()
    lengths = [1, 5, 127, 128, 129, 300, 64, 257]
    cu, q, k, v, do = wl.make_varlen_inputs(len(lengths), 0, 0, 3, d, seed=d, lengths=lengths)
    max_len = max(lengths)
    o, lse, dq, dk, dv = _run(fa, cu, q, k, v, do, causal, max_len)
    O, L = oracle.forward_varlen(f64(q), f64(k), f64(v), cu.numpy(), d ** -0.5, causal)
    DQ, DK, DV = oracle.backward_varlen(f64(q), f64(k), f64(v), f64(do), cu.numpy(), d ** -0.5, causal)
    assert np.abs(f64(o) - O).max() <= O_ATOL
    lse = f64(lse)
    for s, n in enumerate(lengths):
        assert np.abs(lse[s, :, :n] - L[s, :, :n]).max() <= LSE_ATOL
    for nm, got, ref in (("dq", dq, DQ), ("dk", dk, DK), ("dv", dv, DV)):
        assert rel_fro(f64(got), ref) <= GRAD_RTOL, nm


def test_varlen_empty_sequence_and_untouched_lse_tail():
    fa = require_gpu()
    lengths = [70, 0, 200]
    cu, q, k, v, do = wl.make_varlen_inputs(3, 0, 0, 2, 128, seed=1, lengths=lengths)
    max_len = 256
    cu_d = cu.cuda()
    lse = torch.full((3, 2, max_len), 12345.0, device="cuda")
    o = torch.empty_like(q.cuda())
    fa.fa_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), o, lse, cu_d, max_len, True)
    torch.cuda.synchronize()
    assert_no_device_error(fa)
    lse = f64(lse)
    assert (lse[0, :, 70:] == 12345.0).all() and (lse[1] == 12345.0).all() and (lse[2, :, 200:] == 12345.0).all()
    O, L = oracle.forward_varlen(f64(q), f64(k), f64(v), cu.numpy(), 128 ** -0.5, True)
    assert np.abs(f64(o) - O).max() <= O_ATOL


def test_varlen16_workload_sampled():
    """The 16-sequence packed workload (lengths uniform in [64, 4096]) at full
    size; the oracle checks every sequence's forward on sampled rows of one
    head, every sequence's backward on one head, and the shortest and longest
    sequence's backward on two more heads."""
    fa = require_gpu()
    w = wl.WORKLOADS["varlen16"]
    cu, q, k, v, do = wl.workload_inputs(w, seed=0)
    lengths = (cu[1:] - cu[:-1]).tolist()
    max_len = max(lengths)
    o, lse, dq, dk, dv = _run(fa, cu, q, k, v, do, w.causal, max_len)
    o, lse, dq, dk, dv = (f64(t) for t in (o, lse, dq, dk, dv))
    qd, kd, vd, dod = f64(q), f64(k), f64(v), f64(do)
    cun = cu.numpy()
    rng = np.random.default_rng(3)
    for s in range(len(lengths)):
        a, n = cun[s], lengths[s]
        h = int(rng.integers(w.H))
        rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 8)]))
        O, L = oracle.forward_rows(qd[None, a:a + n], kd[None, a:a + n], vd[None, a:a + n], w.scale, True, 0, h, rows)
        assert np.abs(o[a + rows, h] - O).max() <= O_ATOL
        assert np.abs(lse[s, h, rows] - L).max() <= LSE_ATOL
    checks = [(s, int(rng.integers(w.H))) for s in range(len(lengths))]
    checks += [(s, h) for s in (int(np.argmin(lengths)), int(np.argmax(lengths))) for h in (0, w.H - 1)]
    for s, h in checks:
        sl = slice(cun[s], cun[s] + lengths[s])
        DQ, DK, DV = oracle.backward(qd[None, sl, h:h + 1], kd[None, sl, h:h + 1], vd[None, sl, h:h + 1],
                                     dod[None, sl, h:h + 1], w.scale, True)
        assert rel_fro(dq[sl, h], DQ[0, :, 0]) <= GRAD_RTOL, (s, h)
        assert rel_fro(dk[sl, h], DK[0, :, 0]) <= GRAD_RTOL, (s, h)
        assert rel_fro(dv[sl, h], DV[0, :, 0]) <= GRAD_RTOL, (s, h)
