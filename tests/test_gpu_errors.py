"""Failure paths on the GPU, none of which faults or hangs it: argument errors
are rejected on the host before any launch, and the bounded-wait path is
exercised by a kernel waiting on an mbarrier nothing arrives on (short
limit), after which the error word reports the timeout and the context keeps
working."""
import numpy as np
import pytest
import torch

import oracle
from io_aware_attention_flash_gb300 import workloads as wl
from tests.gpu_util import O_ATOL, f64, gpu, require_gpu

pytestmark = gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    fa = require_gpu()
    assert fa.fa_get_device_error() == 0
    assert fa.fa_selftest_wait_timeout(20_000_000) == 0  # 20 ms
    assert fa.fa_get_device_error() == 7                  # FA_ERR_TIMEOUT
    assert fa.fa_get_device_error() == 0                  # cleared on read
    q, k, v, _ = wl.make_inputs(1, 200, 2, 64, seed=1)
    o, lse = fa.attention_forward(q.cuda(), k.cuda(), v.cuda(), True)
    O, _ = oracle.forward(f64(q), f64(k), f64(v), 0.125, True)
    assert np.abs(f64(o) - O).max() <= O_ATOL
    assert fa.fa_get_device_error() == 0


def test_argument_errors_raise():
    fa = require_gpu()
    q = torch.zeros(1, 128, 2, 96, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(fa.FaError, match="HEAD_DIM"):
        fa.attention_forward(q, q, q)
    x = torch.zeros(1, 128, 2, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        fa.attention_forward(x.float(), x.float(), x.float())
    # misaligned base pointer: a view starting 2 bytes into a buffer
    buf = torch.zeros(1 * 128 * 2 * 64 + 1, device="cuda", dtype=torch.bfloat16)
    mis = buf[1:].view(1, 128, 2, 64)
    with pytest.raises(fa.FaError, match="ALIGN"):
        fa.attention_forward(mis, x, x)
    host = torch.zeros(1 * 128 * 2 * 64 + 64, dtype=torch.bfloat16)
    hp = (host.data_ptr() + 15) // 16 * 16
    lse0 = torch.empty(1, 2, 128, device="cuda")
    st = fa.load_library().fa_fwd(hp, x.data_ptr(), x.data_ptr(), x.data_ptr(), lse0.data_ptr(),
                                  1, 2, 128, 64, 0.125, 0, None)
    assert st == 10  # FA_ERR_NOT_DEVICE
    o, lse = torch.empty_like(x), torch.empty(1, 2, 128, device="cuda")
    ws = torch.empty(16, device="cuda", dtype=torch.uint8)
    with pytest.raises(fa.FaError, match="WORKSPACE"):
        fa.fa_bwd(x, x, x, o, x, lse, x.clone(), x.clone(), x.clone(), ws, True)
    assert fa.fa_get_device_error() == 0
