"""Forward parity: CUDA path vs the fp64 oracle, element by element, on the
same seeded bf16 inputs."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_attention_flash_gb300 import workloads as wl
from tests.gpu_util import LSE_ATOL, O_ATOL, assert_no_device_error, f64, gpu, require_gpu

pytestmark = gpu

# Sizes the oracle finishes in seconds that still span several tiles and a
# ragged tail (N not a multiple of 128 / 256), plus the degenerate N=1.
SHAPES = [
    (1, 1, 1, 64), (1, 1, 1, 128), (1, 2, 127, 64), (2, 3, 129, 128), (1, 2, 256, 64), (2, 2, 300, 128),
    (1, 3, 513, 64), (1, 2, 1000, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", SHAPES)
def test_forward_matches_oracle(B, H, N, d, causal):
    fa = require_gpu()
    q, k, v, _ = wl.make_inputs(B, N, H, d, seed=N + d)
    scale = d ** -0.5
    o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal)
    torch.cuda.synchronize()
    assert_no_device_error(fa)
    O, L = oracle.forward(f64(q), f64(k), f64(v), scale, causal)
    assert np.abs(f64(o) - O).max() <= O_ATOL
    assert np.abs(f64(lse) - L).max() <= LSE_ATOL


@pytest.mark.parametrize("name", ["tiny", "small", "small_noncausal"])
def test_forward_small_workloads_full(name):
    fa = require_gpu()
    w = wl.WORKLOADS[name]
    q, k, v, _ = wl.workload_inputs(w, seed=0)
    o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), w.causal)
    assert_no_device_error(fa)
    O, L = oracle.forward(f64(q), f64(k), f64(v), w.scale, w.causal)
    assert np.abs(f64(o) - O).max() <= O_ATOL
    assert np.abs(f64(lse) - L).max() <= LSE_ATOL


@pytest.mark.parametrize("name", ["mid_n4096_d128", "long_n32768"])
def test_forward_full_size_sampled(name):
    """Full-size workload in the benchmark's launch configuration; sampled
    rows checked against the oracle row by row."""
    fa = require_gpu()
    w = wl.WORKLOADS[name]
    q, k, v, _ = wl.workload_inputs(w, seed=0)
    o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), w.causal)
    assert_no_device_error(fa)
    o, lse = f64(o), f64(lse)
    qd, kd, vd = f64(q), f64(k), f64(v)
    rng = np.random.default_rng(5)
    for b, h in [(0, 0), (w.B - 1, w.H - 1), (int(rng.integers(w.B)), int(rng.integers(w.H)))]:
        rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1], rng.integers(0, w.N, 40)]))
        O, L = oracle.forward_rows(qd, kd, vd, w.scale, w.causal, b, h, rows)
        assert np.abs(o[b, rows, h] - O).max() <= O_ATOL
        assert np.abs(lse[b, h, rows] - L).max() <= LSE_ATOL
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_constant_v_gives_constant_o():
    fa = require_gpu()
    B, N, H, d = 1, 700, 2, 128
    q, k, _, _ = wl.make_inputs(B, N, H, d, seed=3)
    c = torch.randn(d, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    v = c.expand(B, N, H, d).contiguous()
    for causal in (False, True):
        o, _ = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal)
        # P sums to one, so O = c up to the bf16 rounding of O
        assert np.abs(f64(o) - f64(c)[None, None, None, :]).max() <= 2 ** -7 * np.abs(f64(c)).max()


def test_large_scores_rescale_path():
    """Scores spread over a wide range force the running max to move by more
    than the skip threshold, exercising the O rescale in TMEM."""
    fa = require_gpu()
    B, N, H, d = 1, 1024, 2, 64
    q, k, v, _ = wl.make_inputs(B, N, H, d, seed=11)
    ramp = torch.linspace(0.1, 6.0, N).view(1, N, 1, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    q = (q.float() * 3).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal)
        assert_no_device_error(fa)
        O, L = oracle.forward(f64(q), f64(k), f64(v), d ** -0.5, causal)
        # Peaked attention makes |O| reach ~3, where one bf16 ulp of the
        # output is 2^-6: the bound scales with |O| (a broken rescale gives
        # errors of order |O|, far above it).
        assert np.abs(f64(o) - O).max() <= O_ATOL * max(1.0, np.abs(O).max())
        assert np.abs(f64(lse) - L).max() <= LSE_ATOL


def test_nondefault_stream_and_scale():
    fa = require_gpu()
    B, N, H, d = 2, 200, 2, 64
    q, k, v, _ = wl.make_inputs(B, N, H, d, seed=21)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), True, scale=0.3)
    s.synchronize()
    O, L = oracle.forward(f64(q), f64(k), f64(v), 0.3, True)
    assert np.abs(f64(o) - O).max() <= O_ATOL
    assert np.abs(f64(lse) - L).max() <= LSE_ATOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_forward_scores_growing_along_the_keys(d, causal):
    """Scores that grow by far more than 2^40 (in base-2 exponent terms)
    across the key tiles: the first tile's row max is a poor reference, so
    the kernel must move it (rescaling O and l) on later tiles.  Also a
    single late key far above everything before it."""
    fa = require_gpu()
    B, N, H = 1, 700, 2
    g = torch.Generator().manual_seed(17)
    ramp = torch.arange(N, dtype=torch.float32) / N
    q = torch.full((B, N, H, d), 1.0)
    k = (ramp[None, :, None, None] * 6.0).expand(B, N, H, d).clone()
    k[:, 450, 1] = 9.0   # head 1: one key far above its neighbours
    v = torch.randn(B, N, H, d, generator=g)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), causal)
    torch.cuda.synchronize()
    assert_no_device_error(fa)
    O, L = oracle.forward(f64(q), f64(k), f64(v), d ** -0.5, causal)
    assert np.abs(f64(o) - O).max() <= O_ATOL
    assert np.abs(f64(lse) - L).max() <= LSE_ATOL
