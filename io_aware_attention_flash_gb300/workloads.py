"""Seeded synthetic inputs and the workload table.

This module holds no attention arithmetic.  It is the one place both the CUDA
path's tests/bench and the CPU oracle draw their inputs from, so that both
sides see the same bf16 values.

Recipe (every workload): one CPU ``torch.Generator`` seeded with ``seed``;
``torch.randn`` in fp32, multiplied by ``amplitude``, rounded to bf16 with
round-to-nearest-even; drawn in the order Q, K, V, dO, each a full
[B, N, H, d] tensor (packed varlen: [T, H, d]).  The varlen workload first
draws its sequence lengths with ``torch.randint(lo, hi + 1, (nseq,))`` from the
same generator.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "make_varlen_inputs", "flops_fwd", "flops_bwd",
           "min_hbm_bytes_fwd", "min_hbm_bytes_bwd", "cu_seqlens_from_lengths", "DecodeWorkload",
           "DECODE_WORKLOADS", "make_decode_inputs", "min_hbm_bytes_decode"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    amplitude: float = 1.0
    varlen: bool = False
    nseq: int = 0
    len_lo: int = 0
    len_hi: int = 0
    note: str = field(default="", compare=False)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads: a tiny non-causal head, a small batch (run causal and
# non-causal), the N=4096 d=128 causal headline, a long-context causal head set
# and a packed variable-length causal batch.
WORKLOADS = {
    "tiny": Workload("tiny", B=1, H=1, N=128, d=64, causal=False),
    "small": Workload("small", B=4, H=16, N=1024, d=64, causal=True),
    "small_noncausal": Workload("small_noncausal", B=4, H=16, N=1024, d=64, causal=False),
    "mid_n4096_d128": Workload("mid_n4096_d128", B=2, H=16, N=4096, d=128, causal=True),
    "long_n32768": Workload("long_n32768", B=1, H=8, N=32768, d=128, causal=True, amplitude=0.5),
    "varlen16": Workload("varlen16", B=1, H=32, N=0, d=128, causal=True, varlen=True,
                         nseq=16, len_lo=64, len_hi=4096),
}


@dataclass(frozen=True)
class DecodeWorkload:
    """Nq new tokens per (sequence, head) against a cache of Nk keys/values."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    amplitude: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# Decode ("LLM Systems 22", section 5.1: one to a few new tokens against a long
# cache): 4 sequences x 32 heads, a 32768-token cache (2 GiB of K and V, far
# beyond L2), one new token, and four (a short speculative / multi-token step).
DECODE_WORKLOADS = {
    "decode_n32768": DecodeWorkload("decode_n32768", B=4, H=32, Nq=1, Nk=32768, d=128, causal=True),
    "decode4_n32768": DecodeWorkload("decode4_n32768", B=4, H=32, Nq=4, Nk=32768, d=128, causal=True),
}


def _draw(gen: torch.Generator, shape, amplitude: float) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if amplitude != 1.0:
        x = x * amplitude
    return x.to(torch.bfloat16)


def make_inputs(B: int, N: int, H: int, d: int, seed: int = 0, amplitude: float = 1.0):
    """Q, K, V, dO as CPU bf16 tensors of shape [B, N, H, d]."""
    gen = torch.Generator().manual_seed(seed)
    return tuple(_draw(gen, (B, N, H, d), amplitude) for _ in range(4))


def make_decode_inputs(B: int, Nq: int, Nk: int, H: int, d: int, seed: int = 0, amplitude: float = 1.0):
    """Q [B, Nq, H, d] and K, V [B, Nk, H, d] as CPU bf16 tensors, drawn in
    that order from one generator seeded with ``seed``."""
    gen = torch.Generator().manual_seed(seed)
    q = _draw(gen, (B, Nq, H, d), amplitude)
    k = _draw(gen, (B, Nk, H, d), amplitude)
    v = _draw(gen, (B, Nk, H, d), amplitude)
    return q, k, v


def cu_seqlens_from_lengths(lengths) -> torch.Tensor:
    lengths = torch.as_tensor(lengths, dtype=torch.int64)
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(lengths, 0)
    return cu.to(torch.int32)


def make_varlen_inputs(nseq: int, len_lo: int, len_hi: int, H: int, d: int, seed: int = 0,
                       amplitude: float = 1.0, lengths=None):
    """Packed inputs: (cu_seqlens int32 [nseq+1], Q, K, V, dO each [T, H, d] bf16).

    Lengths are uniform in [len_lo, len_hi] (inclusive), drawn first from the
    seeded generator unless ``lengths`` is given explicitly.
    """
    gen = torch.Generator().manual_seed(seed)
    if lengths is None:
        lengths = torch.randint(len_lo, len_hi + 1, (nseq,), generator=gen)
    cu = cu_seqlens_from_lengths(lengths)
    T = int(cu[-1])
    return (cu,) + tuple(_draw(gen, (T, H, d), amplitude) for _ in range(4))


def workload_inputs(w: Workload, seed: int = 0):
    if w.varlen:
        return make_varlen_inputs(w.nseq, w.len_lo, w.len_hi, w.H, w.d, seed, w.amplitude)
    return make_inputs(w.B, w.N, w.H, w.d, seed, w.amplitude)


# ---------------------------------------------------------------------------
# Work and byte counts (measurement conventions, not the method).
# Forward FLOPs: 4·N²·d per head (two GEMMs of 2·N²·d), backward 2.5x that,
# both halved under a causal mask.  Varlen sums over sequences.
# ---------------------------------------------------------------------------
def _pairs(lengths, causal: bool) -> float:
    return sum(float(n) * float(n) * (0.5 if causal else 1.0) for n in lengths)


def flops_fwd(H: int, d: int, lengths, causal: bool) -> float:
    return 4.0 * H * d * _pairs(lengths, causal)


def flops_bwd(H: int, d: int, lengths, causal: bool) -> float:
    return 2.5 * flops_fwd(H, d, lengths, causal)


def min_hbm_bytes_fwd(H: int, d: int, total_rows: int) -> float:
    """Q, K, V read once and O written once (bf16), plus the fp32 LSE."""
    return 4.0 * 2.0 * H * d * total_rows + 4.0 * H * total_rows


def min_hbm_bytes_bwd(H: int, d: int, total_rows: int) -> float:
    """Q, K, V, O, dO read and dQ, dK, dV written (bf16), plus LSE in and D."""
    return 8.0 * 2.0 * H * d * total_rows + 2.0 * 4.0 * H * total_rows


def min_hbm_bytes_decode(B: int, H: int, Nq: int, Nk: int, d: int) -> float:
    """K and V read once, Q read and O written (bf16), plus the fp32 LSE."""
    return 2.0 * 2.0 * B * Nk * H * d + 2.0 * 2.0 * B * Nq * H * d + 4.0 * B * H * Nq
