"""The measurement formulas reproduce the worked numbers the pages print."""
import json
import os

import pytest

from io_aware_attention_flash_gb300 import workloads as wl

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_arithmetic.json")))


def test_attention_io_example():
    g = GOLD["attention_io_n4096_d128_bf16"]
    n, d, e = g["n"], g["d"], g["bytes_per_elem"]
    s_bytes = n * n * e
    assert s_bytes / 1e6 == pytest.approx(g["score_matrix_MB"], abs=0.1)  # the page truncates 33.55
    assert round(4 * s_bytes / 1e6) == g["score_round_trip_MB"]
    qkvo = wl.min_hbm_bytes_fwd(H=1, d=d, total_rows=n) - 4 * n  # bf16 part: Q,K,V read + O written
    assert round(qkvo / 1e6) == g["qkvo_MB"]
    flops = wl.flops_fwd(H=1, d=d, lengths=[n], causal=False)
    assert round(flops / 1e9, 1) == g["flops_G"]
    assert round(flops / (g["moved_MB"] * 1e6)) == g["flop_per_byte"]


def test_score_matrix_128k():
    g = GOLD["score_matrix_128k"]
    assert g["n"] * g["n"] * g["bytes_per_elem"] / 2**30 == g["score_matrix_GiB"]


def test_mufu_vs_gemm_ratio():
    g = GOLD["mufu_vs_gemm_h100"]
    b, hd = g["block"], g["head_dim"]
    gemm = wl.flops_fwd(H=1, d=hd, lengths=[b], causal=False)  # the two 128x128x128 GEMMs of one tile
    assert round(gemm / 1e6, 1) == g["gemm_MFLOP"]
    assert gemm / g["tensor_flop_per_clk"] == g["gemm_cycles"]
    assert b * b == g["exp_ops"]
    assert g["exp_ops"] / g["sfu_ops_per_clk"] == g["exp_cycles"]
    assert g["exp_cycles"] / g["gemm_cycles"] == g["exp_over_gemm"]
    # The same ratio with the Blackwell tensor rate doubles to 1.0.
    r = GOLD["blackwell_rates"]
    b200 = (g["exp_ops"] / r["sfu_ops_per_sm_clk"]) / (gemm / r["b200_tensor_ops_per_sm_clk"])
    assert b200 == pytest.approx(1.0)


def test_causal_and_backward_conventions():
    f = wl.flops_fwd(H=16, d=128, lengths=[4096, 4096], causal=True)
    assert f == pytest.approx(4 * 2 * 16 * 4096**2 * 128 / 2)
    assert wl.flops_bwd(H=16, d=128, lengths=[4096, 4096], causal=True) == pytest.approx(2.5 * f)
