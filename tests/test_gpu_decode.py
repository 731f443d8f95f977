"""Decode parity: the split-KV CUDA path vs the fp64 oracle's one-shot decode
definition, on the same seeded bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_attention_flash_gb300 import workloads as wl
from tests.gpu_util import LSE_ATOL, O_ATOL, assert_no_device_error, f64, gpu, require_gpu

pytestmark = gpu

# Caches that end inside a 128-key tile, span one or many splits, and every
# query count the kernels are built for; the degenerate one-key cache.
SHAPES = [
    (1, 1, 1, 1, 128), (2, 3, 1, 100, 64), (1, 2, 2, 129, 128), (1, 2, 4, 1000, 128), (2, 2, 3, 4097, 128),
    (1, 4, 8, 700, 64), (3, 2, 5, 2500, 128), (1, 3, 8, 9000, 128), (2, 2, 6, 6, 64),
    # the tensor-core kernel (d = 128, 2..8 tokens) on a cache shorter than
    # one key tile, and on 7 tokens (padded to 8, then to the MMA's 16)
    (2, 2, 6, 6, 128), (1, 2, 7, 383, 128), (1, 1, 2, 2, 128), (3, 1, 4, 64, 64),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk,d", SHAPES)
def test_decode_matches_oracle(B, H, Nq, Nk, d, causal):
    fa = require_gpu()
    q, k, v = wl.make_decode_inputs(B, Nq, Nk, H, d, seed=Nk + 7 * Nq + d)
    o, lse = fa.attention_decode(q.cuda(), k.cuda(), v.cuda(), causal)
    torch.cuda.synchronize()
    assert_no_device_error(fa)
    O, L = oracle.forward_decode(f64(q), f64(k), f64(v), d ** -0.5, causal)
    assert np.abs(f64(o) - O).max() <= O_ATOL
    finite = np.isfinite(L)
    assert np.array_equal(np.isfinite(f64(lse)), finite)
    assert np.abs(f64(lse)[finite] - L[finite]).max() <= LSE_ATOL


def test_decode_fully_masked_query_gives_zero_and_minus_inf():
    # More new tokens than cached keys under the lower-right causal mask: the
    # first query sees no key (the definition: O = 0, LSE = -inf).
    fa = require_gpu()
    B, H, Nq, Nk, d = 1, 2, 4, 2, 128
    q, k, v = wl.make_decode_inputs(B, Nq, Nk, H, d, seed=3)
    o, lse = fa.attention_decode(q.cuda(), k.cuda(), v.cuda(), True)
    assert_no_device_error(fa)
    O, L = oracle.forward_decode(f64(q), f64(k), f64(v), d ** -0.5, True)
    assert np.abs(f64(o) - O).max() <= O_ATOL
    assert np.all(f64(lse)[:, :, :2] == -np.inf) and np.all(np.isfinite(f64(lse)[:, :, 2:]))


@pytest.mark.parametrize("name", sorted(wl.DECODE_WORKLOADS))
def test_decode_workloads_full(name):
    """The decode workloads at full size (the benchmark's launch
    configuration), every output element against the oracle."""
    fa = require_gpu()
    w = wl.DECODE_WORKLOADS[name]
    q, k, v = wl.make_decode_inputs(w.B, w.Nq, w.Nk, w.H, w.d, seed=0, amplitude=w.amplitude)
    o, lse = fa.attention_decode(q.cuda(), k.cuda(), v.cuda(), w.causal)
    assert_no_device_error(fa)
    O, L = oracle.forward_decode(f64(q), f64(k), f64(v), w.scale, w.causal)
    assert np.abs(f64(o) - O).max() <= O_ATOL
    assert np.abs(f64(lse) - L).max() <= LSE_ATOL


def test_decode_repeatable_with_reused_workspace():
    fa = require_gpu()
    B, H, Nq, Nk, d = 2, 4, 2, 3000, 128
    q, k, v = (t.cuda() for t in wl.make_decode_inputs(B, Nq, Nk, H, d, seed=11))
    ws = torch.full((fa.fa_decode_workspace_bytes(B, H, Nq, Nk, d),), 0x7F, device="cuda", dtype=torch.uint8)
    o1, l1 = fa.attention_decode(q, k, v, True, workspace=ws)
    o2, l2 = fa.attention_decode(q, k, v, True, workspace=ws)
    assert_no_device_error(fa)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
