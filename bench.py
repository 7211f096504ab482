"""Benchmark: one fp8 MLA decode layer-step at T = 262144 on GB300.

A step is the whole decode hot path for one layer and one new token, on one stream:
  kv8_quant_rows (the fresh f32 row -> cache row T-1)  ->  split-T partial kernel  ->  LSE merge.
Workload: H = 128 query heads, kv_lora 512 + qk_rope 64, T = 262144 e4m3 rows (152 MB incl. scales),
bf16 queries, seeded synthetic data (synth.WORKLOADS["dec262k"]).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torchrun; every rank runs an independent replica (the decode of one layer
does not need a second GPU), and the timed region is bracketed by a barrier + synchronize.

Printed (rank 0, one JSON line): metric / value (us per layer-step, whole job) / unit, timing
details, `e2e` (host-resident inputs copied in and the context copied out every step, through the
C ABI), `roofline` for the dominant kernel (CUDA-event time on its stream), `cpu_baseline` (the oracle
on this host's cores, on a bounded sample), `clocks` sampled with nvidia-smi during the timed region.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "fp8 MLA decode µs/layer-step and HBM GB/s (% of peak) at T=262144"
UNIT = "us/layer-step"
KEY = "dec262k"
ROW_BYTES = 580                 # 576 e4m3 bytes + one f32 scale per cache row
FLOP_PER_ROW_HEAD = 2 * 1088    # 576-wide score dot + 512-wide context accumulate
L2_FLUSH_BYTES = 256 << 20      # 2x the 129 MB L2
DECODE_KERNEL_SOURCES = ["fp8_latent_kv_gb300/csrc/attn_tc.cu", "fp8_latent_kv_gb300/csrc/sm100.cuh"]
DECODE_KERNEL = "attn_tc_kernel"
DECODE_BOUND = "tensor"         # e4m3 x e4m3 tensor-core contraction; 479 flop/B is above the HBM ridge
MMA_PIECES = 2                  # hi + lo e4m3 pieces of the queries and of the weights: 2 MMAs per product
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode262k_traffic.json")


# --------------------------------------------------------------------------------------------------
# distributed helpers (also exercised by a 2-rank gloo test on CPU)
# --------------------------------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def reduce_max(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def whole_job_us_per_step(max_ms_per_step: float, n_gpus: int) -> float:
    """N replicas each run one layer-step per step: the job's time per layer-step."""
    return max_ms_per_step * 1000.0 / n_gpus


# --------------------------------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                    power.append(float(p[3]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------------------------------
def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def sources_digest(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_per_launch():
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    if d.get("sources_digest") != sources_digest(DECODE_KERNEL_SOURCES):
        return None
    return d.get("dram_bytes_per_launch")


def alu_peak_tflops(sm_max_mhz: float | None) -> float:
    # f32 FMA: 152 SMs x 128 lanes x 2 flop per clock at the maximum SM clock
    mhz = sm_max_mhz or 2070.0
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def build_decode_inputs(kv, torch, dev, w):
    import synth
    rows = synth.rows_for(w)
    x = torch.from_numpy(rows).to(dev)
    kv8 = torch.empty((w.T, 576), dtype=torch.uint8, device=dev)
    sc = torch.empty(w.T, dtype=torch.float32, device=dev)
    kv.kv8_quant_rows(x[:-1], kv8, sc)            # the resident cache: rows 0..T-2
    fresh = x[-1:].clone()                        # this step's new row
    del x
    ql, qr = synth.queries_for(w, 1)
    q_lat = torch.from_numpy(ql[0]).to(dev).to(torch.bfloat16)
    q_rope = torch.from_numpy(qr[0]).to(dev).to(torch.bfloat16)
    return rows, kv8, sc, fresh, q_lat, q_rope


# --------------------------------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample of the workload
# --------------------------------------------------------------------------------------------------
def oracle_decode_sample(rows, w, n_heads: int):
    import oracle
    import synth
    q_o, s_o = oracle.quant_rows(rows)            # cache bytes from the oracle's own quantizer
    ql, qr = synth.queries_for(w, 1)
    heads = np.linspace(0, w.H - 1, n_heads).astype(int)
    ql_s, qr_s = np.ascontiguousarray(ql[0][heads]), np.ascontiguousarray(qr[0][heads])
    return q_o, s_o, ql_s, qr_s


def time_oracle_step(q_o, s_o, ql_s, qr_s, fresh_row, w) -> float:
    import oracle
    import synth
    t0 = time.perf_counter()
    oracle.quant_rows(fresh_row)                  # the step's fresh row
    oracle.attn_decode(ql_s, qr_s, q_o, s_o, synth.SM_SCALE)
    return time.perf_counter() - t0


def cpu_baseline(rows, w, n_heads: int = 32, repeats: int = 1) -> dict:
    import oracle
    q_o, s_o, ql_s, qr_s = oracle_decode_sample(rows, w, n_heads)
    ts = [time_oracle_step(q_o, s_o, ql_s, qr_s, rows[-1:], w) for _ in range(repeats)]
    t = min(ts)
    us = t * 1e6 * w.H / n_heads
    return {"value": us, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n_heads} of {w.H} heads over all T={w.T} rows (+ the fresh-row quantization), "
                      f"timed {t:.2f} s wall, scaled x{w.H // n_heads} to one layer-step"}


# --------------------------------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------------------------------
def run_reference(args, rank, world):
    """The reference arm: the oracle (plain CPU C, double accumulation) on this host's cores."""
    import synth
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = synth.WORKLOADS[KEY]
    rows = synth.rows_for(w)
    n_heads = 8
    q_o, s_o, ql_s, qr_s = oracle_decode_sample(rows, w, n_heads)
    for _ in range(args.warmup):
        time_oracle_step(q_o, s_o, ql_s, qr_s, rows[-1:], w)
    t0 = time.perf_counter()
    ts = [time_oracle_step(q_o, s_o, ql_s, qr_s, rows[-1:], w) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    us = statistics.mean(ts) * 1e6 * w.H / n_heads
    sample = f"{n_heads} of {w.H} heads over all T={w.T} rows per step, scaled x{w.H // n_heads}"
    line = {"impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1000.0, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": synth.DESCRIPTIONS[KEY], "H": w.H, "T": w.T, "sample": sample},
            "wall_s": wall,
            "cpu_baseline": {"value": us, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch

    import fp8_latent_kv_gb300 as kv
    import synth
    from fp8_latent_kv_gb300 import build as kvbuild

    if rank == 0 or not os.path.exists(kvbuild.LIB):
        kvbuild.build()
    barrier()
    kv.load()
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[KEY]
    H, T = w.H, w.T
    rows, kv8, sc, fresh, q_lat, q_rope = build_decode_inputs(kv, torch, dev, w)
    P = kv.mla_decode8_partitions(H, T)
    ws = torch.empty(kv.mla_decode8_workspace_bytes(H, T) // 4, dtype=torch.float32, device=dev)
    out = torch.empty((H, 512), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sm_scale = synth.SM_SCALE
    launches_per_step = 3  # quant + partial + merge

    def step(ev=None):
        kv.kv8_quant_rows(fresh, kv8[T - 1:], sc[T - 1:], stream=stream)
        if ev is not None:
            ev[0].record(stream)
        kv.mla_decode8_partial(q_lat, q_rope, kv8, sc, T, sm_scale, ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        kv.mla_lse_merge8(ws, 1, P, H, out, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            flush.zero_()
            step()
    torch.cuda.synchronize(dev)

    # ---- device-timed steps (inputs resident), L2 flushed before each step outside the events
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    step_ev = [(E(), E()) for _ in range(args.steps)]
    part_ev = [(E(), E()) for _ in range(args.steps)]
    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            flush.zero_()
            step_ev[k][0].record(stream)
            step(part_ev[k])
            step_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    wall_s = time.perf_counter() - t_wall
    clk = clocks.stop() if rank == 0 else {}
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    part_ms = [a.elapsed_time(b) for a, b in part_ev]
    ms_per_step = reduce_max(statistics.mean(step_ms), dev)
    part_ms_mean = reduce_max(statistics.mean(part_ms), dev)

    # ---- end to end through the C ABI with host buffers: q and the fresh row in, context out
    h_q_lat = q_lat.cpu().pin_memory()
    h_q_rope = q_rope.cpu().pin_memory()
    h_fresh = fresh.cpu().pin_memory()
    h_out = torch.empty((H, 512), dtype=torch.float32).pin_memory()
    d_fresh = torch.empty_like(fresh)
    h2d = h_q_lat.numel() * 2 + h_q_rope.numel() * 2 + h_fresh.numel() * 4
    d2h = h_out.numel() * 4

    def e2e_step():
        q_lat.copy_(h_q_lat, non_blocking=True)
        q_rope.copy_(h_q_rope, non_blocking=True)
        d_fresh.copy_(h_fresh, non_blocking=True)
        kv.kv8_quant_rows(d_fresh, kv8[T - 1:], sc[T - 1:], stream=stream)
        kv.mla_absorb_decode8(q_lat, q_rope, kv8, sc, T, sm_scale, ws, out, stream=stream)
        h_out.copy_(out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            flush.zero_()
            e2e_step()
    torch.cuda.synchronize(dev)
    e2e_ev = [(E(), E()) for _ in range(args.steps)]
    barrier()
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            flush.zero_()
            e2e_ev[k][0].record(stream)
            e2e_step()
            e2e_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(statistics.mean([a.elapsed_time(b) for a, b in e2e_ev]), dev)
    barrier()

    if rank != 0:
        return
    peaks = measured_peaks()
    alg_bytes_partial = T * ROW_BYTES + q_lat.numel() * 2 + q_rope.numel() * 2
    alg_bytes_step = T * ROW_BYTES + h2d + d2h
    flops = float(FLOP_PER_ROW_HEAD) * H * T
    part_s = part_ms_mean / 1e3
    hbm_gbs = alg_bytes_partial / part_s / 1e9
    if DECODE_BOUND == "alu":
        peak = alu_peak_tflops(clk.get("sm_max_mhz"))
        roof = {"bound": "alu", "achieved": flops / part_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                "peak_source": "derived: 152 SMs x 128 f32 FMA lanes x 2 flop x max SM clock"}
    elif DECODE_BOUND == "tensor":
        # the contraction is e4m3 x e4m3: its peak is the measured bf16 burst peak x 2 (nominal fp8/bf16 ratio)
        peak = peaks["bf16_tflops"] * 2.0
        roof = {"bound": "tensor", "achieved": flops / part_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                "peak_source": f"fp8 = 2 x bf16 burst ({peaks['source']})",
                "mma_tflops_issued": MMA_PIECES * flops / part_s / 1e12,
                "mma_frac": MMA_PIECES * flops / part_s / 1e12 / peak,
                "bf16_equiv_frac": flops / part_s / 1e12 / peaks["bf16_tflops"]}
    else:
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": hbm_gbs, "peak": peak, "unit": "GB/s",
                "peak_source": f"HBM copy, {peaks['source']}"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = traffic_per_launch()
    roof["kernel"] = DECODE_KERNEL
    roof["algorithmic_bytes"] = alg_bytes_partial
    roof["algorithmic_flops"] = flops
    roof["kernel_us"] = part_ms_mean * 1e3
    roof["hbm_gbs"] = hbm_gbs
    roof["hbm_frac"] = hbm_gbs / peaks["hbm_gbs"]

    base = cpu_baseline(rows, w) if (world == 1 and not args.no_cpu_baseline) else None
    value = whole_job_us_per_step(ms_per_step, world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3*e4m3->f32" if DECODE_BOUND == "tensor" else "f32", "data": "synthetic",
        "config": {"workload": synth.DESCRIPTIONS[KEY], "H": H, "T": T, "P": P,
                   "step": "kv8_quant_rows(1 fresh row) + split-T partial + log-sum-exp merge",
                   "l2": f"flushed ({L2_FLUSH_BYTES >> 20} MiB write) before every timed step, outside the events",
                   "parallelism": f"replicas x{world}"},
        "step_hbm_gbs": alg_bytes_step / (ms_per_step / 1e3) / 1e9,
        "step_hbm_frac": alg_bytes_step / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"],
        "e2e": {"value": whole_job_us_per_step(e2e_ms, world), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roof,
        "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "wall_s_timed_region": wall_s,
    }
    if base is not None:
        line["cpu_baseline"] = base
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    args = ap.parse_args(argv)
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return 0
            run_reference(args, 0, world)
            return 0
        import torch
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
