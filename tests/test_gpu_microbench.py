"""Unit-rate microbenchmarks behind the MUFU-vs-tensor argument ("LLM Systems
22: Flash Attention", sections 4.1.2 and 4.2): they run, and their results
are in physically plausible ranges for one SM per clock."""
import pytest

from tests.gpu_util import gpu, require_gpu

pytestmark = gpu


@pytest.mark.parametrize("name,lo,hi", [
    ("ex2_per_sm_clk", 4, 256),
    ("cvt_bf16x2_per_sm_clk", 4, 256),
    ("ffma_per_sm_clk", 32, 256),
    ("softmax_ex2_cvt_per_sm_clk", 4, 256),
    ("softmax_step_per_sm_clk", 4, 256),
    ("softmax_step_quarter_poly_per_sm_clk", 4, 256),
    ("ex2_poly_max_rel_err", 0, 1e-4),
    ("mma_bf16_flop_per_sm_clk_n256", 1024, 32768),
    ("mma_bf16_flop_per_sm_clk_n128", 1024, 32768),
    ("mma_bf16_flop_per_sm_clk_n128_tmem_a", 1024, 32768),
    ("mma_bf16_flop_per_sm_clk_n256_random", 1024, 32768),
    ("mma_bf16_flop_per_sm_clk_n128_tmem_a_random", 1024, 32768),
    ("fwd_mma_stream_flop_per_sm_clk_d128", 1024, 32768),
    ("fwd_mma_stream_flop_per_sm_clk_pv64", 1024, 32768),
    ("fwd_mma_stream_flop_per_sm_clk_pv64_separate_p", 1024, 32768),
    ("fwd_mma_stream_flop_per_sm_clk_d128_pv_first", 1024, 32768),
])
def test_microbench_rates_plausible(name, lo, hi):
    fa = require_gpu()
    iters = 512 if name.startswith("fwd") else 2048 if name.startswith("mma") else 4096
    rate = fa._binding.fa_microbench(name, iters)
    print(f"{name} = {rate:.2f}")
    assert lo <= rate <= hi
    assert fa.fa_get_device_error() == 0
