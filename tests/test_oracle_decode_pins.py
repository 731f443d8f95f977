"""Pins for the oracle's decode forward (a few new query tokens against a long
key/value cache, "LLM Systems 22: Flash Attention" section 5.1).

The mask reading (new tokens are the last Nq positions, so query i sees keys
j <= Nk - Nq + i under causal masking) is checked against PyTorch's own
lower-right causal bias, a library definition the oracle does not call; the
rest against closed forms, brute force and the prefill oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

RNG = np.random.default_rng(4321)


def _rand(*shape):
    return RNG.standard_normal(shape)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 37), (3, 40), (4, 4), (8, 65)])
def test_decode_matches_torch_sdpa_lower_right(causal, Nq, Nk):
    from torch.nn.attention.bias import causal_lower_right

    B, H, d = 2, 3, 8
    q, k, v = _rand(B, Nq, H, d), _rand(B, Nk, H, d), _rand(B, Nk, H, d)
    scale = 0.37
    O, L = oracle.forward_decode(q, k, v, scale, causal)
    tq, tk, tv = (torch.tensor(x).permute(0, 2, 1, 3) for x in (q, k, v))
    mask = causal_lower_right(Nq, Nk) if causal else None
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    assert np.allclose(O, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12)
    s = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
    if causal:
        s = s.masked_fill(~causal_lower_right(Nq, Nk)._materialize(device="cpu"), float("-inf"))
    assert np.allclose(L, torch.logsumexp(s, -1).numpy(), atol=1e-12)


def test_decode_with_full_query_block_is_prefill():
    # Nq = Nk: the decode mask is the prefill causal mask.
    B, N, H, d = 1, 19, 2, 4
    q, k, v = _rand(B, N, H, d), _rand(B, N, H, d), _rand(B, N, H, d)
    for causal in (False, True):
        O1, L1 = oracle.forward_decode(q, k, v, 0.5, causal)
        O2, L2 = oracle.forward(q, k, v, 0.5, causal)
        assert np.allclose(O1, O2, atol=1e-13) and np.allclose(L1, L2, atol=1e-13)


def test_single_token_sees_the_whole_cache():
    B, Nk, H, d = 2, 30, 2, 4
    q, k, v = _rand(B, 1, H, d), _rand(B, Nk, H, d), _rand(B, Nk, H, d)
    Oc, Lc = oracle.forward_decode(q, k, v, 0.7, True)
    On, Ln = oracle.forward_decode(q, k, v, 0.7, False)
    assert np.array_equal(Oc, On) and np.array_equal(Lc, Ln)


@pytest.mark.parametrize("causal", [False, True])
def test_decode_zero_q_is_mean_of_visible_values(causal):
    # Q = 0: uniform weights over the visible keys, LSE = ln(count).
    B, Nq, Nk, H, d = 1, 4, 23, 2, 3
    q = np.zeros((B, Nq, H, d))
    k, v = _rand(B, Nk, H, d), _rand(B, Nk, H, d)
    O, L = oracle.forward_decode(q, k, v, 0.4, causal)
    for h in range(H):
        for i in range(Nq):
            n_vis = Nk - Nq + i + 1 if causal else Nk
            assert np.allclose(O[0, i, h], v[0, :n_vis, h].mean(0), atol=1e-14)
            assert abs(L[0, h, i] - math.log(n_vis)) < 1e-14


def test_decode_brute_force_tiny():
    B, Nq, Nk, H, d = 1, 2, 5, 1, 3
    q, k, v = _rand(B, Nq, H, d), _rand(B, Nk, H, d), _rand(B, Nk, H, d)
    O, L = oracle.forward_decode(q, k, v, 0.9, True)
    for i in range(Nq):
        keys = [j for j in range(Nk) if j - (Nk - Nq) <= i]
        s = [0.9 * sum(q[0, i, 0, t] * k[0, j, 0, t] for t in range(d)) for j in keys]
        mx = max(s)
        den = sum(math.exp(x - mx) for x in s)
        assert abs(L[0, 0, i] - (mx + math.log(den))) < 1e-13
        for t in range(d):
            ref = sum(math.exp(x - mx) / den * v[0, j, 0, t] for x, j in zip(s, keys))
            assert abs(O[0, i, 0, t] - ref) < 1e-13


def _mutant_top_left(n_q, n_k, causal):
    if not causal:
        return np.ones((n_q, n_k), dtype=bool)
    return np.arange(n_k)[None, :] <= np.arange(n_q)[:, None]   # upper-left alignment


def test_planted_top_left_alignment_is_caught(monkeypatch):
    monkeypatch.setattr(oa, "decode_mask", _mutant_top_left)
    with pytest.raises(AssertionError):
        test_decode_matches_torch_sdpa_lower_right(True, 3, 40)
