"""One forward and one backward per sequence length, for measuring how DRAM
traffic grows with N (run it under a profiler that reads the DRAM byte
counters; it times nothing itself).

IO-aware attention keeps the N x N score matrix on chip, so its HBM traffic
is O(N·d) per head: Q, K, V, O (and dO, dQ, dK, dV) once each, plus whatever
K/V re-reads miss L2 ("LLM Systems 22: Flash Attention", section 3.3; "08 ·
FlashAttention", section 三).  A standard implementation moves O(N²).  This
driver runs causal d = 128 attention at N = 1k .. 32k with B·H fixed and prints
the algorithmic minimum bytes per call, against which the measured counters
are compared.

    python -m io_aware_attention_flash_gb300.dram_sweep [--bh 8] [--n 1024 2048 ...]
"""
from __future__ import annotations

import argparse

import torch

from . import attention_backward, attention_forward
from . import workloads as wl


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--bh", type=int, default=8, help="B*H, held fixed (B = 1)")
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--n", type=int, nargs="+", default=[1024, 2048, 4096, 8192, 16384, 32768])
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("dram_sweep needs a CUDA device")
    H, d = args.bh, args.d
    print("N,fwd_min_bytes,bwd_min_bytes", flush=True)
    for N in args.n:
        q, k, v, do = (t.cuda() for t in wl.make_inputs(1, N, H, d, seed=args.seed))
        o, lse = attention_forward(q, k, v, causal=True)
        attention_backward(q, k, v, o, do, lse, causal=True)
        torch.cuda.synchronize()
        print(f"{N},{wl.min_hbm_bytes_fwd(H, d, N):.0f},{wl.min_hbm_bytes_bwd(H, d, N):.0f}", flush=True)
        del q, k, v, do, o, lse
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
