"""Exact IO-aware softmax attention for GB300 (sm_103a).

O = softmax(scale · Q Kᵀ) V computed tile by tile with an online softmax
("LLM Systems 22: Flash Attention", section 3.1; "08 · FlashAttention",
section 二); the backward recomputes P from the saved log-sum-exp
("LLM Systems 22", section 3.2).  Tensors are bf16 [B, N, H, d] (packed
variable-length batches: [T, H, d] with cu_seqlens); d is 64 or 128.

The compute runs in the hand-written kernels of libfa_gb300.so behind the C
ABI in include/fa.h; PyTorch only provides device memory and streams.  This
module allocates outputs and workspace and calls the binding.
"""
from __future__ import annotations

import torch

from . import _binding
from ._binding import (  # noqa: F401  (C-ABI names)
    FaError,
    fa_decode_workspace_bytes,
    fa_fwd_decode,
    fa_bwd,
    fa_bwd_varlen,
    fa_bwd_varlen_workspace_bytes,
    fa_bwd_workspace_bytes,
    fa_cta_order,
    fa_fwd,
    fa_fwd_varlen,
    fa_get_device_error,
    fa_selftest_wait_timeout,
    fa_set_kernel_events,
)

__all__ = [
    "attention_forward", "attention_backward", "attention_forward_varlen", "attention_backward_varlen",
    "flash_attention", "FaError", "fa_fwd", "fa_bwd", "fa_fwd_varlen", "fa_bwd_varlen",
    "fa_bwd_workspace_bytes", "fa_bwd_varlen_workspace_bytes", "fa_get_device_error", "load_library",
    "attention_decode", "fa_fwd_decode", "fa_decode_workspace_bytes",
]


def load_library():
    """Load libfa_gb300.so; raises RuntimeError if it has not been built."""
    return _binding.lib()


def attention_forward(q, k, v, causal: bool = False, scale=None, stream=None):
    """Returns (o [B,N,H,d] bf16, lse [B,H,N] fp32)."""
    B, N, H, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    fa_fwd(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def attention_decode(q, k, v, causal: bool = False, scale=None, stream=None, workspace=None):
    """Decode: q [B,Nq,H,d] (Nq <= 8 newest tokens) against the cache k, v
    [B,Nk,H,d].  Returns (o [B,Nq,H,d] bf16, lse [B,H,Nq] fp32).  causal: the
    new tokens are the cache's last Nq positions (query i sees keys
    j <= Nk - Nq + i)."""
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    if workspace is None:
        workspace = torch.empty(max(fa_decode_workspace_bytes(B, H, Nq, Nk, d), 16), device=q.device,
                                dtype=torch.uint8)
    fa_fwd_decode(q, k, v, o, lse, workspace, causal, scale, stream)
    return o, lse


def attention_backward(q, k, v, o, dout, lse, causal: bool = False, scale=None, stream=None, workspace=None):
    """Returns (dq, dk, dv), each [B,N,H,d] bf16."""
    B, N, H, d = q.shape
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_bytes(B, H, N, d), device=q.device, dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, causal, scale, stream)
    return dq, dk, dv


def attention_forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False, scale=None, stream=None):
    """Packed batch: q/k/v [T,H,d]; returns (o [T,H,d], lse [nseq,H,max_seqlen])."""
    T, H, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((cu_seqlens.numel() - 1, H, max_seqlen), device=q.device, dtype=torch.float32)
    fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen, causal, scale, stream)
    return o, lse


def attention_backward_varlen(q, k, v, o, dout, lse, cu_seqlens, max_seqlen: int, causal: bool = False,
                              scale=None, stream=None, workspace=None):
    T, H, d = q.shape
    nseq = cu_seqlens.numel() - 1
    if workspace is None:
        workspace = torch.empty(fa_bwd_varlen_workspace_bytes(T, nseq, max_seqlen, H, d), device=q.device,
                                dtype=torch.uint8)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, workspace, cu_seqlens, max_seqlen, causal, scale, stream)
    return dq, dk, dv


class _FlashAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale):
        o, lse = attention_forward(q, k, v, causal, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = causal, scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = attention_backward(q, k, v, o, do.contiguous(), lse, ctx.causal, ctx.scale)
        return dq, dk, dv, None, None


def flash_attention(q, k, v, causal: bool = False, scale=None):
    """Autograd-aware attention over bf16 [B,N,H,d] CUDA tensors."""
    return _FlashAttention.apply(q, k, v, causal, scale)
