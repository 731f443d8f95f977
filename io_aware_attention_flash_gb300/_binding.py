"""ctypes binding of libfa_gb300 (argument marshalling only).

Every function here checks tensor dtypes/devices/shapes, takes raw device
pointers and the current CUDA stream from PyTorch, and calls the C entry
point of the same name.  All compute happens in the CUDA kernels behind the
C ABI; there is no other path.  If the library is not built, loading fails
with an error instead of falling back to anything.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libfa_gb300.so")

FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_ALIGN", 3: "FA_ERR_HEAD_DIM", 4: "FA_ERR_SHAPE",
    5: "FA_ERR_ARCH", 6: "FA_ERR_CUDA", 7: "FA_ERR_TIMEOUT", 8: "FA_ERR_WORKSPACE", 9: "FA_ERR_SCALE",
    10: "FA_ERR_NOT_DEVICE", 11: "FA_ERR_SCRATCH_LIMIT",
}

# Exported symbols and their C signatures (include/fa.h).
_P, _I, _F, _Z, _U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
SIGNATURES = {
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_workspace_bytes": (_Z, [_I, _I, _I, _I]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _I, _I, _I, _I, _F, _I, _P]),
    "fa_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_bwd_varlen_workspace_bytes": (_Z, [_I, _I, _I, _I, _I]),
    "fa_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "fa_get_device_error": (_I, [_P]),
    "fa_selftest_wait_timeout": (_I, [_U64, _P]),
    "fa_set_kernel_events": (_I, [_P, _P]),
    "fa_cta_order": (_I, [_I, _I, _I, ctypes.POINTER(_I), _P, _P, ctypes.c_longlong]),
    "fa_last_error_detail": (ctypes.c_char_p, []),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _P]),
    "fa_microbench": (_I, [_I, _I, ctypes.POINTER(ctypes.c_double), _P]),
    "fa_decode_workspace_bytes": (_Z, [_I, _I, _I, _I, _I]),
    "fa_fwd_decode": (_I, [_P, _P, _P, _P, _P, _P, _Z, _I, _I, _I, _I, _I, _F, _I, _P]),
}

# fa_microbench selectors: rate per SM per SM-clock of each unit (the
# MUFU-vs-tensor measurements), and the accuracy of the polynomial exp2.
MICROBENCH = {"ex2_per_sm_clk": 0, "cvt_bf16x2_per_sm_clk": 1, "ffma_per_sm_clk": 2,
              "mma_bf16_flop_per_sm_clk_n256": 3, "mma_bf16_flop_per_sm_clk_n128": 4,
              "mma_bf16_flop_per_sm_clk_n128_tmem_a": 5, "mma_bf16_flop_per_sm_clk_n256_random": 6,
              "mma_bf16_flop_per_sm_clk_n128_tmem_a_random": 7,
              "fwd_mma_stream_flop_per_sm_clk_d128": 8, "fwd_mma_stream_flop_per_sm_clk_pv64": 9,
              "fwd_mma_stream_flop_per_sm_clk_pv64_separate_p": 10,
              "fwd_mma_stream_flop_per_sm_clk_d128_pv_first": 11,
              "softmax_ex2_cvt_per_sm_clk": 38, "softmax_step_per_sm_clk": 40,
              "ex2_poly_max_rel_err": 42, "softmax_step_quarter_poly_per_sm_clk": 43}

# Size of the static scratch array behind fa_bwd_noalloc (FA_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 32 << 20

_lib = None
_lock = threading.Lock()


class FaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = f"{fn} failed: {STATUS_NAMES.get(status, status)} ({lib().fa_status_string(status).decode()})"
        if status == 6:
            msg += f": {lib().fa_last_error_detail().decode()}"
        super().__init__(msg)


def lib() -> ctypes.CDLL:
    """Load libfa_gb300.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with `python -m io_aware_attention_flash_gb300.build`")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def _check(fn: str, status: int) -> None:
    if status != FA_OK:
        raise FaError(fn, status)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _bf16(name: str, t: torch.Tensor, shape) -> None:
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16 (got {t.dtype}); fp32 and other types are not supported")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _f32(name: str, t: torch.Tensor, shape) -> None:
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be a contiguous CUDA float32 tensor of shape {tuple(shape)}")


def _scale(scale, d):
    return float(d) ** -0.5 if scale is None else float(scale)


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI)
# ---------------------------------------------------------------------------
def fa_fwd(q, k, v, o, lse, causal: bool, scale=None, stream=None) -> None:
    B, N, H, d = q.shape
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _bf16(n, t, (B, N, H, d))
    _f32("lse", lse, (B, H, N))
    _check("fa_fwd", lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d,
                                  _scale(scale, d), int(bool(causal)), _stream(stream)))


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, N, d))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, causal: bool, scale=None, stream=None) -> None:
    B, N, H, d = q.shape
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        _bf16(n, t, (B, N, H, d))
    _f32("lse", lse, (B, H, N))
    _check("fa_bwd", lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                                  _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  B, H, N, d, _scale(scale, d), int(bool(causal)), _stream(stream)))


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, causal: bool, scale=None, stream=None) -> None:
    """fa_bwd for callers that cannot provide device memory: the library's
    static scratch array stands in for the workspace (problems up to
    NOALLOC_SCRATCH_BYTES of workspace; calls must not overlap on the GPU)."""
    B, N, H, d = q.shape
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        _bf16(n, t, (B, N, H, d))
    _f32("lse", lse, (B, H, N))
    _check("fa_bwd_noalloc", lib().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                                  _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, _scale(scale, d),
                                                  int(bool(causal)), _stream(stream)))


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen: int, causal: bool, scale=None, stream=None) -> None:
    T, H, d = q.shape
    nseq = cu_seqlens.numel() - 1
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o)):
        _bf16(n, t, (T, H, d))
    _f32("lse", lse, (nseq, H, max_seqlen))
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be a CUDA int32 tensor")
    _check("fa_fwd_varlen", lib().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens),
                                                nseq, max_seqlen, T, H, d, _scale(scale, d), int(bool(causal)),
                                                _stream(stream)))


def fa_bwd_varlen_workspace_bytes(total: int, nseq: int, max_seqlen: int, H: int, d: int) -> int:
    return int(lib().fa_bwd_varlen_workspace_bytes(total, nseq, max_seqlen, H, d))


def fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, workspace, cu_seqlens, max_seqlen: int, causal: bool,
                  scale=None, stream=None) -> None:
    T, H, d = q.shape
    nseq = cu_seqlens.numel() - 1
    for n, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        _bf16(n, t, (T, H, d))
    _f32("lse", lse, (nseq, H, max_seqlen))
    _check("fa_bwd_varlen", lib().fa_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(cu_seqlens), nseq, max_seqlen, T, H, d,
        _scale(scale, d), int(bool(causal)), _stream(stream)))


def fa_decode_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(lib().fa_decode_workspace_bytes(B, H, Nq, Nk, d))


def fa_fwd_decode(q, k, v, o, lse, workspace, causal: bool, scale=None, stream=None) -> None:
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    _bf16("q", q, (B, Nq, H, d))
    _bf16("o", o, (B, Nq, H, d))
    for n, t in (("k", k), ("v", v)):
        _bf16(n, t, (B, Nk, H, d))
    _f32("lse", lse, (B, H, Nq))
    _check("fa_fwd_decode", lib().fa_fwd_decode(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), B, H, Nq, Nk, d, _scale(scale, d), int(bool(causal)),
        _stream(stream)))


def fa_get_device_error(stream=None) -> int:
    return int(lib().fa_get_device_error(_stream(stream)))


def fa_cta_order(npairs: int, ntiles: int, slots: int):
    """Launch order of the attention kernels' CTAs (host only): returns
    (group, pair, tile) with pair[b], tile[b] the work item of launch index b."""
    import numpy as np

    group = ctypes.c_int(0)
    _check("fa_cta_order", lib().fa_cta_order(npairs, ntiles, slots, ctypes.byref(group), None, None, 0))
    n = -(-npairs // group.value) * group.value * ntiles
    pair, tile = np.zeros(n, dtype=np.int32), np.zeros(n, dtype=np.int32)
    _check("fa_cta_order", lib().fa_cta_order(npairs, ntiles, slots, None, pair.ctypes.data_as(_P),
                                              tile.ctypes.data_as(_P), n))
    return group.value, pair, tile


def fa_set_kernel_events(start_event, end_event) -> None:
    """Time the main kernel of the next backward call on this thread with two
    torch.cuda.Event objects (created with enable_timing=True)."""
    for ev in (start_event, end_event):
        # torch creates the underlying cudaEvent_t lazily, on the first
        # record; record once so there is a handle (and torch regards the
        # event as recorded).  The library records it again around the kernel.
        if ev is not None and ev.cuda_event == 0:
            ev.record()
    s = None if start_event is None else ctypes.c_void_p(start_event.cuda_event)
    e = None if end_event is None else ctypes.c_void_p(end_event.cuda_event)
    _check("fa_set_kernel_events", lib().fa_set_kernel_events(s, e))


def fa_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return int(lib().fa_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def fa_microbench(name: str, iters: int, stream=None) -> float:
    """Rate per SM per clock of one unit (see MICROBENCH for the names)."""
    out = ctypes.c_double(0.0)
    _check("fa_microbench", lib().fa_microbench(MICROBENCH[name], int(iters), ctypes.byref(out), _stream(stream)))
    return out.value
