"""Shared helpers of the GPU parity tests (oracle side in fp64, CUDA side via
the C ABI).  Tolerances are the ones the method is held to: O max-abs 1e-2,
LSE max-abs 1e-3, dQ/dK/dV relative Frobenius 2e-2."""
import numpy as np
import pytest
import torch

O_ATOL = 1e-2
LSE_ATOL = 1e-3
GRAD_RTOL = 2e-2

gpu = pytest.mark.gpu


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import io_aware_attention_flash_gb300 as fa
    from io_aware_attention_flash_gb300 import build
    build.build()
    fa.load_library()  # fail loudly if the library cannot load
    return fa


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def rel_fro(a: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), 1e-30))


def assert_no_device_error(fa):
    assert fa.fa_get_device_error() == 0, "a kernel reported a device-side error"
