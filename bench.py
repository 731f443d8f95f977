"""Benchmark: forward + backward exact attention on one batch per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mid_n4096_d128] [--no-cpu-baseline] [--no-e2e]
    python bench.py --dram-sweep [N ...]     (DRAM-traffic-vs-N driver for ncu)

A step is one pass of the whole hot path over one batch: fa_fwd (one kernel)
then fa_bwd (pre, main, post kernels).  Inputs are seeded synthetic bf16
tensors already resident in device memory; L2 is flushed (a 256 MiB write)
between timed steps, outside the per-step CUDA events.  FLOPs follow the
usual convention: forward 4·B·H·N²·d, backward 2.5x, both halved when causal.
The roofline's kernel (the backward main kernel) is timed in a second loop of
K backward calls with CUDA events recorded right around it.

Under torchrun (N > 1) every rank runs the same workload on its own GPU with
no collective on the data path (weak scaling); timing uses a barrier and the
maximum over ranks, and rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle (the reference definition) on the
host cores, on a bounded sample of the same workload (whole (batch, head)
problems), with the same metric and unit.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from io_aware_attention_flash_gb300 import workloads as wl  # noqa: E402

METRIC = "fwd/bwd attention TFLOP/s and % of GB300 BF16 tensor peak, N=4096 d=128"
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p.get("hbm_gbs", 0.0)), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, 6800.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _workload_desc(w: wl.Workload) -> str:
    return f"{w.name}: B={w.B} H={w.H} N={w.N} d={w.d} {'causal' if w.causal else 'non-causal'}"


def _host_cores():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"), default=0)
        if n:
            return int(n)
    except Exception:
        pass
    return os.cpu_count() or 1


# Arm CPU part numbers (/proc/cpuinfo "CPU part", implementer 0x41) of the
# server cores a GPU machine may have.
_ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
              "0xd49": "Arm Neoverse N2", "0xd84": "Arm Neoverse V3"}


def _cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                v = line.split(":", 1)[1].strip()
                return f"{_ARM_PARTS[v]} (CPU part {v})" if v in _ARM_PARTS else v
    except Exception:
        pass
    return "unknown"


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def time_oracle_sample(w: wl.Workload, budget_s: float, seed: int = 0):
    """Run the fp64 oracle forward + backward on whole (batch, head) problems
    of the workload, cycling through them, until `budget_s` has elapsed (at
    least one).  Returns (TFLOP/s by the workload's FLOP convention, seconds,
    problems done)."""
    import numpy as np

    import oracle

    q, k, v, do = wl.workload_inputs(w, seed)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    done, t0 = 0, time.perf_counter()
    while True:
        b, h = heads[done % len(heads)]
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1), slice(None))
        qd, kd, vd, dod = (t[sl].float().double().numpy() for t in (q, k, v, do))
        oracle.forward(qd, kd, vd, w.scale, w.causal)
        oracle.backward(qd, kd, vd, dod, w.scale, w.causal)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    flops = (wl.flops_fwd(1, w.d, [w.N], w.causal) + wl.flops_bwd(1, w.d, [w.N], w.causal)) * done
    del np
    return flops / dt / 1e12, dt, done


# Bounded oracle samples of the three smallest dense configurations, for the
# cpu_baseline record: (workload, seconds of work on all cores, on one core).
CPU_CONFIG_SAMPLES = (("tiny", 1.0, 1.0), ("small", 2.5, 2.5), ("mid_n4096_d128", 0.0, 3.0))


def _cpu_sample_records(names_budgets, cores):
    out = []
    for name, budget in names_budgets:
        w = wl.WORKLOADS[name]
        v, dt, n = time_oracle_sample(w, budget)
        out.append({"workload": name, "cores": cores, "value": v, "unit": "TFLOP/s", "seconds": dt,
                    "sample": f"{n} (batch, head) problem(s) of {w.B * w.H}, fwd+bwd"})
    return out


def cpu_baseline_configs(all_cores: int):
    """The oracle on the tiny, small and mid configurations, on all host cores
    (this process; BLAS threads = all cores, numpy's elementwise steps on one)
    and on one core (a child interpreter pinned to one CPU with one BLAS
    thread)."""
    recs = _cpu_sample_records([(n, b) for n, b, _ in CPU_CONFIG_SAMPLES if b > 0], all_cores)
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    spec = ",".join(f"{n}:{b1}" for n, _, b1 in CPU_CONFIG_SAMPLES)
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-one-core", spec], env=env,
                           capture_output=True, text=True, timeout=300)
        recs += json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # the all-cores records stand on their own
        recs.append({"one_core": f"not measured: {type(e).__name__}"})
    return recs


def run_cpu_one_core(spec: str):
    """Child side of cpu_baseline_configs: pin this process to one CPU and
    time the named samples; prints one JSON list."""
    try:
        os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    except (AttributeError, OSError):
        pass
    pairs = [(x.split(":")[0], float(x.split(":")[1])) for x in spec.split(",")]
    print(json.dumps(_cpu_sample_records(pairs, 1)), flush=True)
    return 0


def run_reference(args, w):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        time_oracle_sample(w, 0.0)
    vals, secs = [], []
    for _ in range(args.steps):
        v, dt, _ = time_oracle_sample(w, 0.0)
        vals.append(v)
        secs.append(dt)
    value = statistics.mean(vals)
    cores = _host_cores()
    sample = f"one (batch, head) problem of {w.name} per step (fwd+bwd, fp64 numpy oracle), {_cpu_model()}"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_desc(w), "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.rows = []
        if self.proc is None:
            return False
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)
        return False

    def summary(self):
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": reasons, "samples": len(rows)}


def run_gpu(args, w):
    import io_aware_attention_flash_gb300 as fa
    from io_aware_attention_flash_gb300 import build as fabuild

    ws_n, rank, local = _dist()
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or ws_n == 1:
        fabuild.build()
    if ws_n > 1:
        dist.barrier()
    fa.load_library()

    def barrier():
        if ws_n > 1:
            dist.barrier()

    # Inputs for this rank: every rank draws its own batch (seed + rank).
    q_h, k_h, v_h, do_h = wl.workload_inputs(w, seed=args.seed + rank)
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    wsp = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), device=dev, dtype=torch.uint8)
    flush = torch.empty(L2_FLUSH_BYTES, device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    f_fwd = wl.flops_fwd(w.H, w.d, [w.N] * w.B, w.causal)
    f_bwd = wl.flops_bwd(w.H, w.d, [w.N] * w.B, w.causal)

    def step():
        fa.fa_fwd(q, k, v, o, lse, w.causal)
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, wsp, w.causal)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    ev_main = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize(dev)
        # The K steps: nothing recorded between the backward's kernels, so each
        # starts while its predecessor finishes (programmatic dependent launch).
        for i in range(K):
            flush.zero_()
            e = ev[i]
            e[0].record(stream)
            fa.fa_fwd(q, k, v, o, lse, w.causal)
            e[1].record(stream)
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, wsp, w.causal)
            e[2].record(stream)
        # The backward main kernel alone (roofline): K more backward calls with
        # events recorded right before and after it, which also keeps it apart
        # from its neighbours.
        for i in range(K):
            flush.zero_()
            fa.fa_set_kernel_events(ev_main[i][0], ev_main[i][1])
            fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, wsp, w.causal)
        torch.cuda.synchronize(dev)
        barrier()
        e2e = None
        if not args.no_e2e:
            e2e = run_e2e(fa, w, dev, stream, (q_h, k_h, v_h, do_h), K, flush, nbuf=args.e2e_buffers)
    if fa.fa_get_device_error() != 0:
        raise RuntimeError("device error during the timed region")

    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_ms = [e[1].elapsed_time(e[2]) for e in ev]
    main_ms = [e[0].elapsed_time(e[1]) for e in ev_main]
    t_step = statistics.mean(step_ms)
    t_step, t_fwd, t_bwd, t_main = max_over_ranks(
        [t_step, statistics.mean(fwd_ms), statistics.mean(bwd_ms), statistics.mean(main_ms)], dev)
    if e2e is not None:
        e2e["ms"] = max_over_ranks([e2e["ms"]], dev)[0]

    peak, hbm_peak, peak_kind = _peaks()
    value = whole_job_tflops(ws_n, f_fwd + f_bwd, t_step)
    fwd_tflops = f_fwd / (t_fwd * 1e-3) / 1e12
    bwd_tflops = f_bwd / (t_bwd * 1e-3) / 1e12
    # Dominant kernel: the backward main kernel carries all backward FLOPs.
    main_tflops = f_bwd / (t_main * 1e-3) / 1e12
    traffic = _committed_traffic(w.name, "fa_bwd_main_kernel")
    result = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws_n, "steps": K, "warmup": args.warmup,
        "ms_per_step": t_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": _workload_desc(w), "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
                   "seed": args.seed, "l2": "flushed: 256 MiB write between steps, outside the step events",
                   "parallelism": f"weak x{ws_n} (independent batch per GPU)"},
        "fwd": {"ms": t_fwd, "tflops": fwd_tflops, "frac_of_peak": fwd_tflops / peak},
        "bwd": {"ms": t_bwd, "tflops": bwd_tflops, "frac_of_peak": bwd_tflops / peak, "main_kernel_ms": t_main},
        "roofline": {"kernel": "fa_bwd_main_kernel", "bound": "tensor", "achieved": main_tflops, "peak": peak,
                     "unit": "TFLOP/s", "frac": main_tflops / peak, "traffic": traffic,
                     "peak_source": f"{peak_kind} bf16 burst (MEASURED_PEAKS.json)" if peak_kind == "measured"
                     else "fallback 1.9 PFLOP/s bf16"},
        # 4 kernels per step (fwd; bwd pre, main, post), 3 per backward call
        # of the main-kernel timing loop.
        "gpu_launches": 7 * K,
        "clocks": clocks.summary(),
    }
    # A second reference: the tensor pipe's own issue rate at the measured
    # clock (8192 bf16 FLOP per clock per SM for 128x128x16 tcgen05 MMAs, the
    # rate the MMA-stream microbenchmark sustains), which the cuBLAS-measured
    # peak above (taken at a lower clock) understates.
    sm_mhz = result["clocks"].get("sm_mhz")
    if sm_mhz:
        mma = 8192 * torch.cuda.get_device_properties(dev).multi_processor_count * sm_mhz * 1e6 / 1e12
        result["mma_rate"] = {"tflops": mma, "basis": "8192 FLOP/clk/SM x SMs x median SM clock",
                              "fwd_frac": fwd_tflops / mma, "bwd_frac": bwd_tflops / mma,
                              "bwd_main_kernel_frac": main_tflops / mma}
    if not args.no_decode:
        result["decode"] = run_decode(fa, dev, flush, 20, args.warmup, args.seed + rank, hbm_peak)
    if e2e is not None:
        result["e2e"] = {"value": whole_job_tflops(ws_n, f_fwd + f_bwd, e2e["ms"]), "unit": "TFLOP/s",
                         "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"], "ms_per_step": e2e["ms"],
                         "note": e2e["note"]}
    if rank == 0 and not args.no_cpu_baseline and ws_n == 1:
        v_cpu, dt, heads = time_oracle_sample(w, args.cpu_budget)
        cores = _host_cores()
        result["cpu_baseline"] = {
            "value": v_cpu, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{heads} of {w.B * w.H} (batch, head) problems of {w.name}, fwd+bwd, fp64 numpy oracle, "
                      f"{dt:.1f} s on {_cpu_model()}",
            "nproc": os.cpu_count(), "cpu_model": _cpu_model(),
            "threads_note": "cores = BLAS threads of the matmuls; numpy's elementwise steps (exp, masks) run on one",
            "configs": cpu_baseline_configs(cores)}
        if w.name == "mid_n4096_d128":  # the headline sample above is this workload's all-cores record
            result["cpu_baseline"]["configs"].append({
                "workload": w.name, "cores": cores, "value": v_cpu, "unit": "TFLOP/s", "seconds": dt,
                "sample": f"{heads} (batch, head) problem(s) of {w.B * w.H}, fwd+bwd (the headline sample)"})
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws_n > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_decode(fa, dev, flush, steps: int, warmup: int, seed: int, hbm_peak: float):
    """Split-KV decode ("LLM Systems 22", section 5.2) on the decode workloads:
    K and V read once is the whole cost, so the roofline is HBM bandwidth.
    Each call (split + merge kernels) is timed with CUDA events on the
    launching stream, L2 flushed between calls (the 2 GiB cache exceeds L2
    anyway)."""
    out = []
    stream = torch.cuda.current_stream(dev)
    for name in sorted(wl.DECODE_WORKLOADS):
        w = wl.DECODE_WORKLOADS[name]
        q, k, v = (t.to(dev) for t in wl.make_decode_inputs(w.B, w.Nq, w.Nk, w.H, w.d, seed, w.amplitude))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.Nq), device=dev, dtype=torch.float32)
        ws = torch.empty(fa.fa_decode_workspace_bytes(w.B, w.H, w.Nq, w.Nk, w.d), device=dev, dtype=torch.uint8)
        for _ in range(max(3, warmup)):
            fa.fa_fwd_decode(q, k, v, o, lse, ws, w.causal)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            fa.fa_fwd_decode(q, k, v, o, lse, ws, w.causal)
            e1.record(stream)
        torch.cuda.synchronize(dev)
        if fa.fa_get_device_error() != 0:
            raise RuntimeError("device error during the decode timing")
        ms = max_over_ranks([statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)], dev)[0]
        nbytes = wl.min_hbm_bytes_decode(w.B, w.H, w.Nq, w.Nk, w.d)
        gbs = nbytes / (ms * 1e-3) / 1e9
        out.append({"workload": f"{name}: B={w.B} H={w.H} Nq={w.Nq} Nk={w.Nk} d={w.d} "
                                f"{'causal (lower-right)' if w.causal else 'non-causal'}",
                    "ms": ms, "gpu_launches": 2 * steps,
                    "roofline": {"kernels": "fa_decode_split_kernel + fa_decode_merge_kernel", "bound": "hbm",
                                 "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                                 "algorithmic_bytes": nbytes,
                                 "peak_source": "measured copy (MEASURED_PEAKS.json)"}})
        del q, k, v, o, lse, ws
        torch.cuda.empty_cache()
    return out


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over all ranks (identity without a
    process group): the slowest rank sets every timing."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_tflops(world_size: int, flops_per_rank: float, ms_max: float) -> float:
    """Weak scaling: every rank processed `flops_per_rank`; the job took the
    slowest rank's time."""
    return world_size * flops_per_rank / (ms_max * 1e-3) / 1e12


def run_e2e(fa, w, dev, stream, host_inputs, K, flush, nbuf=2):
    """The same step through the public API with pinned host buffers, as a
    user streaming batches would run it: every step's inputs go host->device
    and its O, LSE, dQ, dK, dV come back, all inside the timed region.  Steps
    are pipelined over three streams with `nbuf` sets of device tensors, so
    step i+1's upload and step i-1's download overlap step i's kernels.
    Within a step the forward starts once Q, K, V are up (dO uploads under
    it) and O, LSE go down while the backward runs, so neither direction of
    the host link waits for a whole step (the L2 flush stays in front of each
    step's kernels).  Returns the time per step of K steps."""
    hq, hk, hv, hdo = (t.pin_memory() for t in host_inputs)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo))
    s_in, s_out, s_cmp = torch.cuda.Stream(dev), torch.cuda.Stream(dev), stream
    dev_in = [tuple(torch.empty_like(t, device=dev) for t in host_inputs) for _ in range(nbuf)]
    dev_out = [None] * nbuf
    host_out = [([torch.empty_like(hq).pin_memory() for _ in range(4)],
                 torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()) for _ in range(nbuf)]
    d2h = sum(t.numel() * t.element_size() for t in host_out[0][0]) + host_out[0][1].numel() * 4
    wsp = torch.empty(fa.fa_bwd_workspace_bytes(w.B, w.H, w.N, w.d), device=dev, dtype=torch.uint8)
    n = K + nbuf
    ev_qkv, ev_in, ev_fwd, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(n)] for _ in range(5))

    def one_step(i):
        b = i % nbuf
        q, k, v, do = dev_in[b]
        if i >= nbuf:
            s_in.wait_event(ev_cmp[i - nbuf])       # the step that last read these inputs has finished
        with torch.cuda.stream(s_in):
            for dst, src in ((q, hq), (k, hk), (v, hv)):
                dst.copy_(src, non_blocking=True)
            ev_qkv[i].record(s_in)
            do.copy_(hdo, non_blocking=True)
        ev_in[i].record(s_in)
        s_cmp.wait_event(ev_qkv[i])
        if i >= nbuf:
            s_cmp.wait_event(ev_out[i - nbuf])      # its output buffers have been read back
        with torch.cuda.stream(s_cmp):
            flush.zero_()
            o, lse = fa.attention_forward(q, k, v, w.causal, stream=s_cmp)
            ev_fwd[i].record(s_cmp)
            s_cmp.wait_event(ev_in[i])
            dq, dk, dv = fa.attention_backward(q, k, v, o, do, lse, w.causal, stream=s_cmp, workspace=wsp)
        dev_out[b] = (o, lse, dq, dk, dv)
        ev_cmp[i].record(s_cmp)
        hosts, lse_h = host_out[b]
        s_out.wait_event(ev_fwd[i])
        with torch.cuda.stream(s_out):
            hosts[0].copy_(o, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
        s_out.wait_event(ev_cmp[i])
        with torch.cuda.stream(s_out):
            for dst, src in zip(hosts[1:], (dq, dk, dv)):
                dst.copy_(src, non_blocking=True)
            for t in dev_out[b]:
                t.record_stream(s_out)
        ev_out[i].record(s_out)

    for i in range(nbuf):                           # warm-up steps
        one_step(i)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(nbuf, n):
        one_step(i)
    s_in.wait_event(ev_out[n - 1])
    t1.record(s_in)
    torch.cuda.synchronize(dev)
    return {"ms": t0.elapsed_time(t1) / K, "h2d": h2d, "d2h": d2h,
            "note": f"steps pipelined over 3 streams (upload / kernels / download), {nbuf} buffer sets; "
                    "forward after Q, K, V are up, O and LSE down during the backward"}


KERNEL_SOURCES = {
    "fa_bwd_main_kernel": ["fa_bwd.cu", "ptx.cuh", "fa_kernels.cuh"],
    "fa_fwd_kernel": ["fa_fwd.cu", "ptx.cuh", "fa_kernels.cuh"],
}


def _committed_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/<kernel>__<workload>.json), or None when there is none or the
    kernel's sources changed since the counters were taken (the summary
    records a SHA-256 of those sources)."""
    import hashlib

    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.json")
    try:
        with open(path) as f:
            summary = json.load(f)
        h = hashlib.sha256()
        for name in KERNEL_SOURCES[kernel]:
            with open(os.path.join(ROOT, "io_aware_attention_flash_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        if summary.get("source_sha256") != h.hexdigest():
            return None
        return summary.get("dram_bytes_per_launch")
    except Exception:
        return None


def run_dram_sweep(args):
    """One forward and one backward per sequence length, with B·H fixed, for
    measuring how DRAM traffic grows with N under a profiler that reads the
    DRAM byte counters (this mode times nothing itself).  IO-aware attention
    keeps the N x N score matrix on chip, so its HBM traffic is O(N·d) per
    head ("LLM Systems 22: Flash Attention", section 3.3; "08 ·
    FlashAttention", section 三).  Prints the algorithmic minimum bytes per
    call for each N, against which the measured counters are compared."""
    import io_aware_attention_flash_gb300 as fa
    from io_aware_attention_flash_gb300 import build as fabuild

    if not torch.cuda.is_available():
        raise SystemExit("--dram-sweep needs a CUDA device")
    fabuild.build()
    fa.load_library()
    H, d = args.sweep_bh, 128
    print("N,fwd_min_bytes,bwd_min_bytes", flush=True)
    for N in args.dram_sweep:
        q, k, v, do = (t.cuda() for t in wl.make_inputs(1, N, H, d, seed=args.seed))
        o, lse = fa.attention_forward(q, k, v, causal=True)
        fa.attention_backward(q, k, v, o, do, lse, causal=True)
        torch.cuda.synchronize()
        if fa.fa_get_device_error() != 0:
            raise RuntimeError("device error in the DRAM sweep")
        print(f"{N},{wl.min_hbm_bytes_fwd(H, d, N):.0f},{wl.min_hbm_bytes_bwd(H, d, N):.0f}", flush=True)
        del q, k, v, do, o, lse
        torch.cuda.empty_cache()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mid_n4096_d128", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-buffers", type=int, default=2,
                    help="device buffer sets the end-to-end pipeline rotates through")
    ap.add_argument("--no-decode", action="store_true", help="skip the split-KV decode measurement")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--dram-sweep", type=int, nargs="*", default=None, metavar="N",
                    help="instead of the benchmark: one causal d=128 forward + backward per N (B=1, H=--sweep-bh), "
                         "for a DRAM-counter capture; no N given: 1024 .. 32768")
    ap.add_argument("--sweep-bh", type=int, default=8)
    ap.add_argument("--cpu-one-core", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.cpu_one_core:
        return run_cpu_one_core(args.cpu_one_core)
    if args.dram_sweep is not None:
        if not args.dram_sweep:
            args.dram_sweep = [1024, 2048, 4096, 8192, 16384, 32768]
        return run_dram_sweep(args)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = wl.WORKLOADS[args.workload]
    if w.varlen:
        ap.error("the benchmark times dense workloads; varlen is covered by the tests")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_gpu(args, w)


if __name__ == "__main__":
    raise SystemExit(main())
