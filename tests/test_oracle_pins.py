"""Pins for the fp64 oracle: checks against things the pages and mathematics fix.

None of these re-types the oracle's own formula.  They check it against
  * closed forms (constant V, zero Q),
  * a brute-force scalar triple loop on tiny inputs,
  * the pages' online-softmax recurrences (tile by tile, both forms printed),
  * central finite differences of L = sum(O * dO) (pins the backward to the
    forward),
  * gradient invariants that follow from rows of P summing to one,
  * PyTorch's float64 scaled_dot_product_attention + autograd (a library
    routine the oracle does not call),
and planted mistakes (mutants of the oracle, on the CPU) must fail them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa

RNG = np.random.default_rng(1234)


def _rand(*shape, rng=RNG):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------
# softmax rows
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one(causal):
    S = _rand(37, 37) * 5
    P, lse = oracle.softmax_rows(S, oracle.visible_mask(np.arange(37), 37, causal))
    assert np.allclose(P.sum(1), 1.0, atol=1e-14, rtol=0)
    assert (P >= 0).all()
    if causal:
        assert np.all(np.triu(P, 1) == 0)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_o(causal):
    B, N, H, d = 2, 45, 3, 8
    q, k = _rand(B, N, H, d), _rand(B, N, H, d)
    c = _rand(d)
    v = np.broadcast_to(c, (B, N, H, d)).copy()
    O, _ = oracle.forward(q, k, v, 0.37, causal)
    assert np.allclose(O, np.broadcast_to(c, O.shape), atol=1e-14, rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_q_gives_uniform_attention(causal):
    # Q = 0 makes every score 0: P is uniform over the visible keys, so O is
    # the mean of the visible V rows (a prefix mean when causal) and LSE is
    # ln(number of visible keys).
    B, N, H, d = 1, 33, 2, 4
    q = np.zeros((B, N, H, d))
    k, v = _rand(B, N, H, d), _rand(B, N, H, d)
    O, L = oracle.forward(q, k, v, 0.5, causal)
    for h in range(H):
        for i in range(N):
            n_vis = i + 1 if causal else N
            assert np.allclose(O[0, i, h], v[0, :n_vis, h].mean(0), atol=1e-14)
            assert abs(L[0, h, i] - math.log(n_vis)) < 1e-14


# ---------------------------------------------------------------------------
# brute force on tiny inputs
# ---------------------------------------------------------------------------
def _brute_force(q, k, v, scale, causal):
    B, N, H, d = q.shape
    O = np.zeros_like(q)
    L = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                keys = range(i + 1) if causal else range(N)
                s = {}
                for j in keys:
                    acc = 0.0
                    for t in range(d):
                        acc += q[b, i, h, t] * k[b, j, h, t]
                    s[j] = acc * scale
                mx = max(s.values())
                den = sum(math.exp(x - mx) for x in s.values())
                L[b, h, i] = mx + math.log(den)
                for t in range(d):
                    O[b, i, h, t] = sum(math.exp(s[j] - mx) / den * v[b, j, h, t] for j in keys)
    return O, L


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(1, 1), (5, 3), (8, 4)])
def test_brute_force_tiny(causal, N, d):
    B, H = 2, 2
    q, k, v = _rand(B, N, H, d), _rand(B, N, H, d), _rand(B, N, H, d)
    O, L = oracle.forward(q, k, v, 0.7, causal)
    O2, L2 = _brute_force(q, k, v, 0.7, causal)
    assert np.allclose(O, O2, atol=1e-13, rtol=0)
    assert np.allclose(L, L2, atol=1e-13, rtol=0)


# ---------------------------------------------------------------------------
# the pages' tiled recurrences equal the one-shot oracle
# ---------------------------------------------------------------------------
def _online_unnormalised(qh, kh, vh, scale, causal, cuts):
    """Recurrence of "08 · FlashAttention" section 二: per query row keep the
    running max m, exp-sum l (relative to m) and unnormalised output O; for a
    new key block with max m' and exp-sum l': m_new = max(m, m'),
    l_new = e^(m-m_new) l + e^(m'-m_new) l', O_new = e^(m-m_new) O +
    e^(m'-m_new) P~' V'; divide by l once at the end."""
    N, d = qh.shape
    O = np.zeros((N, vh.shape[1]))
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    bounds = [0] + list(cuts) + [kh.shape[0]]
    for a, b in zip(bounds[:-1], bounds[1:]):
        if a == b:
            continue
        S = scale * qh @ kh[a:b].T
        if causal:
            S = np.where(np.arange(a, b)[None, :] <= np.arange(N)[:, None], S, -np.inf)
        mp = S.max(1)
        Pt = np.exp(S - np.where(np.isfinite(mp), mp, 0)[:, None])
        lp = Pt.sum(1)
        m_new = np.maximum(m, mp)
        f_old = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
        f_new = np.where(np.isfinite(mp), np.exp(mp - m_new), 0.0)
        l = f_old * l + f_new * lp
        O = f_old[:, None] * O + f_new[:, None] * (Pt @ vh[a:b])
        m = m_new
    return O / l[:, None], m + np.log(l)


def _online_normalised(qh, kh, vh, scale, cuts):
    """Form of "LLM Systems 22" section 3.1 (with max subtraction): keep a
    normalised output; on a new block rescale it by
    alpha = d_old e^(m_old - m_new) / d_new and add the block's own terms
    divided by d_new (non-causal)."""
    N = qh.shape[0]
    O = np.zeros((N, vh.shape[1]))
    m = np.full(N, -np.inf)
    dsum = np.zeros(N)
    bounds = [0] + list(cuts) + [kh.shape[0]]
    for a, b in zip(bounds[:-1], bounds[1:]):
        if a == b:
            continue
        S = scale * qh @ kh[a:b].T
        m_new = np.maximum(m, S.max(1))
        E = np.exp(S - m_new[:, None])
        scale_old = np.where(np.isfinite(m), np.exp(m - m_new), 0.0)
        d_new = dsum * scale_old + E.sum(1)
        alpha = dsum * scale_old / d_new
        O = O * alpha[:, None] + (E @ vh[a:b]) / d_new[:, None]
        m, dsum = m_new, d_new
    return O, m + np.log(dsum)


@pytest.mark.parametrize("causal", [False, True])
def test_two_tile_identity_every_split(causal):
    N, d = 24, 6
    q, k, v = _rand(1, N, 1, d) * 2, _rand(1, N, 1, d) * 2, _rand(1, N, 1, d)
    O, L = oracle.forward(q, k, v, 0.8, causal)
    for cut in range(0, N + 1):
        O2, L2 = _online_unnormalised(q[0, :, 0], k[0, :, 0], v[0, :, 0], 0.8, causal, [cut])
        assert np.allclose(O[0, :, 0], O2, atol=1e-12, rtol=0)
        assert np.allclose(L[0, 0], L2, atol=1e-12, rtol=0)
        if not causal:
            O3, L3 = _online_normalised(q[0, :, 0], k[0, :, 0], v[0, :, 0], 0.8, [cut])
            assert np.allclose(O[0, :, 0], O3, atol=1e-12, rtol=0)
            assert np.allclose(L[0, 0], L3, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_k_tile_identity(causal):
    N, d = 300, 16
    q, k, v = _rand(1, N, 1, d) * 3, _rand(1, N, 1, d) * 3, _rand(1, N, 1, d)
    O, L = oracle.forward(q, k, v, 0.25, causal)
    for tile in (1, 7, 64, 128):
        cuts = list(range(tile, N, tile))
        O2, L2 = _online_unnormalised(q[0, :, 0], k[0, :, 0], v[0, :, 0], 0.25, causal, cuts)
        assert np.allclose(O[0, :, 0], O2, atol=1e-12, rtol=0)
        assert np.allclose(L[0, 0], L2, atol=1e-12, rtol=0)


def test_blockwise_without_rescaling_is_wrong():
    # "LLM Systems 22" section 3.1, first attempt: each block normalised by its
    # own local denominator and the blocks simply added.  It must not match.
    N, d = 32, 8
    q, k, v = _rand(1, N, 1, d), _rand(1, N, 1, d), _rand(1, N, 1, d)
    O, _ = oracle.forward(q, k, v, 0.5, False)
    qh, kh, vh = q[0, :, 0], k[0, :, 0], v[0, :, 0]
    naive = np.zeros((N, d))
    for a in (0, 16):
        S = 0.5 * qh @ kh[a:a + 16].T
        E = np.exp(S - S.max(1, keepdims=True))
        naive += (E / E.sum(1, keepdims=True)) @ vh[a:a + 16]
    assert np.abs(naive - O[0, :, 0]).max() > 1e-2


# ---------------------------------------------------------------------------
# backward: finite differences and invariants
# ---------------------------------------------------------------------------
def _loss(q, k, v, do, scale, causal):
    O, _ = oracle.forward(q, k, v, scale, causal)
    return float((O * do).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(5, 3), (16, 8)])
def test_backward_finite_differences(causal, N, d):
    B, H = 1, 2
    rng = np.random.default_rng(7 + N)
    q, k, v, do = (rng.standard_normal((B, N, H, d)) for _ in range(4))
    scale = 0.6
    dQ, dK, dV = oracle.backward(q, k, v, do, scale, causal)
    h = 1e-6
    for X, G in ((q, dQ), (k, dK), (v, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + h
            lp = _loss(q, k, v, do, scale, causal)
            X[idx] = old - h
            lm = _loss(q, k, v, do, scale, causal)
            X[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.linalg.norm(num - G) / max(np.linalg.norm(G), 1e-30)
        assert err < 1e-6, err


@pytest.mark.parametrize("causal", [False, True])
def test_gradient_invariants(causal):
    B, N, H, d = 2, 70, 2, 8
    q, k, v, do = (_rand(B, N, H, d) for _ in range(4))
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.4, causal)
    # rows of P sum to one  =>  sum_j dV_j = sum_i dO_i
    assert np.allclose(dV.sum(1), do.sum(1), atol=1e-12)
    # rows of dS sum to zero  =>  sum_j dK_j = 0
    assert np.abs(dK.sum(1)).max() < 1e-12 * max(1.0, np.abs(dK).max())


# ---------------------------------------------------------------------------
# a library routine: PyTorch float64 SDPA with autograd
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N,panel", [(50, None), (1100, None), (200, 48)])
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(causal, N, panel, monkeypatch):
    """N = 1100 spans three of the oracle's 512-row panels, and a 48-row panel
    at N = 200 five: the panel-by-panel accumulation of dK and dV (summed over
    query rows) is checked against a library that never splits the rows."""
    if panel is not None:
        monkeypatch.setattr(oa, "PANEL_ROWS", panel)
    B, H, d = (2, 3, 16) if N <= 200 else (1, 2, 16)
    q, k, v, do = (_rand(B, N, H, d) for _ in range(4))
    scale = 1.0 / math.sqrt(d)
    O, L = oracle.forward(q, k, v, scale, causal)
    dQ, dK, dV = oracle.backward(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.tensor(x).permute(0, 2, 1, 3).requires_grad_() for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    out.backward(torch.tensor(do).permute(0, 2, 1, 3))
    assert np.allclose(O, out.detach().permute(0, 2, 1, 3).numpy(), atol=1e-12)
    for mine, t in ((dQ, tq), (dK, tk), (dV, tv)):
        assert np.allclose(mine, t.grad.permute(0, 2, 1, 3).numpy(), atol=1e-11)
    s = torch.einsum("bhid,bhjd->bhij", tq.detach(), tk.detach()) * scale
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    assert np.allclose(L, torch.logsumexp(s, -1).numpy(), atol=1e-12)


# ---------------------------------------------------------------------------
# samplers and varlen agree with the full oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("causal", [False, True])
def test_row_samplers_agree_with_full(causal, monkeypatch):
    monkeypatch.setattr(oa, "PANEL_ROWS", 16)  # several panels at this size
    B, N, H, d = 2, 53, 2, 8
    q, k, v, do = (_rand(B, N, H, d) for _ in range(4))
    O, L = oracle.forward(q, k, v, 0.3, causal)
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.3, causal)
    rows = [0, 5, 17, 52]
    o, lse = oracle.forward_rows(q, k, v, 0.3, causal, 1, 1, rows)
    assert np.allclose(o, O[1, rows, 1], atol=1e-13) and np.allclose(lse, L[1, 1, rows], atol=1e-13)
    keys = [3, 40, 51, 52]
    dq, dk, dv = oracle.backward_rows(q, k, v, do, 0.3, causal, 0, 1, rows, keys)
    assert np.allclose(dq, dQ[0, rows, 1], atol=1e-13)
    assert np.allclose(dk, dK[0, keys, 1], atol=1e-13)
    assert np.allclose(dv, dV[0, keys, 1], atol=1e-13)


def test_varlen_sequences_are_independent():
    lens = [5, 19, 1, 12]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T, H, d = int(cu[-1]), 2, 4
    q, k, v, do = (_rand(T, H, d) for _ in range(4))
    O, L = oracle.forward_varlen(q, k, v, cu, 0.5, True)
    dQ, dK, dV = oracle.backward_varlen(q, k, v, do, cu, 0.5, True)
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        o, lse = oracle.forward(q[None, a:b], k[None, a:b], v[None, a:b], 0.5, True)
        assert np.allclose(O[a:b], o[0]) and np.allclose(L[s, :, : b - a], lse[0])
        assert np.all(np.isnan(L[s, :, b - a:]))
    # perturbing one sequence leaves the others unchanged
    k2 = k.copy()
    k2[cu[1]:cu[2]] += 1.0
    O2, _ = oracle.forward_varlen(q, k2, v, cu, 0.5, True)
    assert np.array_equal(O2[: cu[1]], O[: cu[1]]) and np.array_equal(O2[cu[2]:], O[cu[2]:])


# ---------------------------------------------------------------------------
# planted mistakes must fail a pin
# ---------------------------------------------------------------------------
def _mutant_softmax_no_max(S, mask):
    P, lse = _orig_softmax(S, mask)
    return P, lse - np.where(mask, S, -np.inf).max(axis=1)  # LSE loses its max term


_orig_softmax = oa.softmax_rows
_orig_mask = oa.visible_mask
_orig_head_bwd = oa._head_backward_panel


def _mutant_mask_strict(rows, n_k, causal):
    m = _orig_mask(rows, n_k, causal)
    if causal:
        m = m & (np.arange(n_k)[None, :] < np.asarray(rows)[:, None])
        m[:, 0] = True
    return m


def _mutant_bwd_d_from_dp(qh, kh, vh, doh, scale, causal, rows):
    S = scale * (qh[rows] @ kh.T)
    P, _ = _orig_softmax(S, _orig_mask(rows, kh.shape[0], causal))
    dP = doh[rows] @ vh.T
    D = dP.sum(axis=1)                       # dropped the P weighting
    dS = P * (dP - D[:, None])
    return scale * (dS @ kh), scale * (dS.T @ qh[rows]), P.T @ doh[rows]


def _mutant_bwd_no_scale(qh, kh, vh, doh, scale, causal, rows):
    dq, dk, dv = _orig_head_bwd(qh, kh, vh, doh, scale, causal, rows)
    return dq / scale, dk, dv                 # dQ missing its scale factor


def _run_forward_pins():
    test_zero_q_gives_uniform_attention(True)
    test_brute_force_tiny(True, 5, 3)


def _run_backward_pins():
    test_backward_finite_differences(True, 5, 3)


@pytest.mark.parametrize("name,target,mutant,pins", [
    ("lse without max", "softmax_rows", _mutant_softmax_no_max, _run_forward_pins),
    ("causal mask off by one", "visible_mask", _mutant_mask_strict, _run_forward_pins),
    ("D without P weighting", "_head_backward_panel", _mutant_bwd_d_from_dp, _run_backward_pins),
    ("dQ without scale", "_head_backward_panel", _mutant_bwd_no_scale, _run_backward_pins),
])
def test_planted_mistakes_are_caught(name, target, mutant, pins, monkeypatch):
    monkeypatch.setattr(oa, target, mutant)
    with pytest.raises(AssertionError):
        pins()
