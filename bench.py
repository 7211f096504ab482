"""Benchmark of the fp8 MLA hot path on GB300.

Default workload (the headline): one decode layer-step at T = 262144.  A step is the whole decode
hot path for one layer and one new token, on one stream:
  kv8_quant_rows (the fresh f32 row -> cache row T-1)  ->  query prep + split-T partial kernel  ->  LSE merge.
H = 128 query heads, kv_lora 512 + qk_rope 64, T = 262144 e4m3 rows (152 MB incl. scales), bf16
queries, seeded synthetic data (synth.WORKLOADS["dec262k"]).

Other workloads (--workload), each one step of its own hot path:
  dec16k   the same decode step at T = 16384
  dsa      selected-row decode: 8 sequences x 2048 listed rows of a 131072-row cache each
  prefill  kv8_quant_rows of the chunk's 1024 fresh rows + causal prefill of 1024 queries over T = 65536
  proj_dec / proj_prefill   the absorb projections through an fmt=8 kv_b (q_nope -> q_lat, context ->
           head output) for 1 query / a 1024-query chunk of 128 heads
  indexer  the DSA lightning indexer: 8 queries x 64 index heads over 131072 e4m3 index keys each, top-2048
  batch_dec  one decode step for 8 sequences with their own caches (up to 32768 rows each, ragged)
  mixed_dec  one decode step over the mixed-precision cache (448 e4m3 + 64 bf16 per row), T = 65536

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload KEY]
For N > 1 launch with torchrun; every rank runs an independent replica (one layer's attention does
not need a second GPU), and the timed region is bracketed by a barrier + synchronize.

Printed (rank 0, one JSON line): metric / value (us per step, whole job) / unit, timing details,
`e2e` (host-resident inputs copied in and the output copied out every step, through the C ABI),
`roofline` for the dominant kernel (CUDA-event time on its stream), `cpu_baseline` (the oracle on
this host's cores, on a bounded sample), `clocks` sampled with nvidia-smi during the timed region.
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

HEADLINE_METRIC = "fp8 MLA decode µs/layer-step and HBM GB/s (% of peak) at T=262144"
ROW_BYTES = 580                 # 576 e4m3 bytes + one f32 scale per cache row
FLOP_PER_ROW_HEAD = 2 * 1088    # 576-wide score dot + 512-wide context accumulate
L2_FLUSH_BYTES = 256 << 20      # 2x the 129 MB L2
TC_KERNEL_SOURCES = ["fp8_latent_kv_gb300/csrc/attn_tc.cu", "fp8_latent_kv_gb300/csrc/sm100.cuh"]
TC_KERNEL = "attn_tc_kernel"
# the sources each committed traffic summary is tied to (a kernel's .cu and the headers its device code uses)
IDX_SOURCES = ["fp8_latent_kv_gb300/csrc/indexer.cu", "fp8_latent_kv_gb300/csrc/sm100.cuh",
               "fp8_latent_kv_gb300/csrc/quant_row.cuh"]
MIXED_SOURCES = ["fp8_latent_kv_gb300/csrc/attn_mixed.cu", "fp8_latent_kv_gb300/csrc/sm100.cuh",
                 "fp8_latent_kv_gb300/csrc/quant_row.cuh"]
PROJ_TC_SOURCES = ["fp8_latent_kv_gb300/csrc/proj8_tc.cu", "fp8_latent_kv_gb300/csrc/sm100.cuh"]
PROJ_SMALL_SOURCES = ["fp8_latent_kv_gb300/csrc/proj8.cu"]
MMA_PIECES = 2                  # hi + lo e4m3 pieces of the queries and of the weights: 2 MMAs per product


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
    """Digest of the code in the given sources: comments and whitespace are left out, so a traffic summary
    stays tied to the code it measured and not to its commentary."""
    import re
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(re.sub(r"\s+", "", text).encode())
    return h.hexdigest()[:16]


def traffic_file(key: str, kernel: str = TC_KERNEL) -> str:
    return os.path.join(ROOT, "profiles", f"{kernel}_{key}_traffic.json")


def traffic_per_launch(key: str, kernel: str = TC_KERNEL, sources=None):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, or None when there
    is none for this workload or the kernel's sources changed since the counters were taken."""
    path = traffic_file(key, kernel)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("sources_digest") != sources_digest(sources or TC_KERNEL_SOURCES):
        return None
    return d.get("dram_bytes_per_launch")


class Packed:
    """A step's host inputs packed into one pinned buffer, copied by one kv8_copy (a kernel reading the
    page-locked host memory) into one device buffer whose typed views are what the library calls
    receive (each view 256-byte aligned)."""

    def __init__(self, torch, dev, tensors):
        offs, o = [], 0
        for t in tensors:
            offs.append(o)
            o += (t.numel() * t.element_size() + 255) // 256 * 256
        self.host = torch.empty(o, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(o, dtype=torch.uint8, device=dev)
        self.views = []
        for t, off in zip(tensors, offs):
            n = t.numel() * t.element_size()
            self.host[off:off + n].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
            self.views.append(self.dev[off:off + n].view(t.dtype).view(t.shape))
        self.nbytes = sum(t.numel() * t.element_size() for t in tensors)

    def upload(self, kv, stream):
        kv.kv8_copy(self.dev, self.host, stream=stream)


def _bf16(torch, dev, a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(torch.bfloat16)


class Case:
    """One workload's step.  Subclasses build the resident inputs and define:
    step(stream, ev)   enqueue one step; ev = (start, end) events around the dominant kernel call
    e2e_step(stream)   the same step from pinned host buffers, output copied back
    and the figures of the JSON line."""
    key = ""
    unit = "us/layer-step"
    launches_per_step = 0
    kernel_calls = ""       # what the events around the dominant call bracket
    step_desc = ""
    dtype = "e4m3*e4m3->f32"

    def config(self) -> dict:
        raise NotImplementedError

    def roofline(self, kern_s: float, peaks: dict, key: str) -> dict:
        """The attention kernel's roofline: a tensor-core contraction of e4m3 operands."""
        hbm_gbs = self.alg_bytes / kern_s / 1e9
        # the contraction is e4m3 x e4m3: its peak is the measured bf16 burst peak x 2 (nominal fp8/bf16 ratio)
        peak = peaks["bf16_tflops"] * 2.0
        achieved = self.flops / kern_s / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"fp8 = 2 x bf16 burst ({peaks['source']})",
                "traffic": traffic_per_launch(key), "kernel": TC_KERNEL, "events_bracket": self.kernel_calls,
                "mma_tflops_issued": MMA_PIECES * achieved, "mma_frac": MMA_PIECES * achieved / peak,
                "bf16_equiv_frac": achieved / peaks["bf16_tflops"],
                "algorithmic_bytes": self.alg_bytes, "algorithmic_flops": self.flops, "kernel_us": kern_s * 1e6,
                "hbm_gbs": hbm_gbs, "hbm_frac": hbm_gbs / peaks["hbm_gbs"], "hbm_peak_gbs": peaks["hbm_gbs"]}


class DecodeCase(Case):
    launches_per_step = 4  # quant + query prep + partial + merge
    kernel_calls = "mla_decode8_partial: query prep + attn_tc_kernel (programmatic dependent launch)"
    step_desc = "kv8_quant_rows(1 fresh row) + query prep + split-T partial + log-sum-exp merge"

    def __init__(self, kv, torch, dev, w):
        import synth
        self.kv, self.torch, self.w = kv, torch, w
        H, T = w.H, w.T
        self.rows = synth.rows_for(w)
        x = torch.from_numpy(self.rows).to(dev)
        self.kv8 = torch.empty((T, 576), dtype=torch.uint8, device=dev)
        self.sc = torch.empty(T, dtype=torch.float32, device=dev)
        kv.kv8_quant_rows(x[:-1], self.kv8, self.sc)      # the resident cache: rows 0..T-2
        self.fresh = x[-1:].clone()                       # this step's new row
        del x
        ql, qr = synth.queries_for(w, 1)
        self.q_lat, self.q_rope = _bf16(torch, dev, ql[0]), _bf16(torch, dev, qr[0])
        self.P = kv.mla_decode8_partitions(H, T)
        self.ws = torch.empty(kv.mla_decode8_workspace_bytes(H, T) // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((H, 512), dtype=torch.float32, device=dev)
        # e2e: the step's inputs (queries, fresh row) in one pinned buffer, one copy per step
        self.pack = Packed(torch, dev, [self.q_lat, self.q_rope, self.fresh])
        self.h_out = torch.empty((H, 512), dtype=torch.float32).pin_memory()
        self.h2d = self.pack.nbytes
        self.d2h = self.h_out.numel() * 4
        self.alg_bytes = T * ROW_BYTES + self.q_lat.numel() * 2 + self.q_rope.numel() * 2
        self.alg_bytes_step = T * ROW_BYTES + self.h2d + self.d2h
        self.flops = float(FLOP_PER_ROW_HEAD) * H * T

    def step(self, stream, ev=None):
        kv, w = self.kv, self.w
        kv.kv8_quant_rows(self.fresh, self.kv8[w.T - 1:], self.sc[w.T - 1:], stream=stream)
        if ev is not None:
            ev[0].record(stream)
        kv.mla_decode8_partial(self.q_lat, self.q_rope, self.kv8, self.sc, w.T, SM_SCALE(), self.ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        kv.mla_lse_merge8(self.ws, 1, self.P, w.H, self.out, stream=stream)

    def kernel_call(self, stream):
        w = self.w
        self.kv.mla_decode8_partial(self.q_lat, self.q_rope, self.kv8, self.sc, w.T, SM_SCALE(), self.ws, stream=stream)

    def e2e_step(self, stream):
        kv, w = self.kv, self.w
        self.pack.upload(kv, stream)
        q_lat, q_rope, fresh = self.pack.views
        kv.kv8_quant_rows(fresh, self.kv8[w.T - 1:], self.sc[w.T - 1:], stream=stream)
        kv.mla_absorb_decode8(q_lat, q_rope, self.kv8, self.sc, w.T, SM_SCALE(), self.ws, self.out, stream=stream)
        kv.kv8_copy(self.h_out, self.out, stream=stream)

    def config(self):
        return {"H": self.w.H, "T": self.w.T, "P": getattr(self, "P", None)}

    # ---- the oracle on a bounded sample: n_heads of the H heads over all T rows
    def oracle_setup(self, n_heads):
        import oracle
        import synth
        w = self.w
        q_o, s_o = oracle.quant_rows(self.rows)       # cache bytes from the oracle's own quantizer
        ql, qr = synth.queries_for(w, 1)
        heads = np.linspace(0, w.H - 1, n_heads).astype(int)
        self._o = (q_o, s_o, np.ascontiguousarray(ql[0][heads]), np.ascontiguousarray(qr[0][heads]))
        self._scale = w.H / n_heads
        return (f"{n_heads} of {w.H} heads over all T={w.T} rows (+ the fresh-row quantization), "
                f"scaled x{w.H // n_heads} to one layer-step")

    def oracle_step(self) -> float:
        import oracle
        q_o, s_o, ql, qr = self._o
        t0 = time.perf_counter()
        oracle.quant_rows(self.rows[-1:])
        oracle.attn_decode(ql, qr, q_o, s_o, SM_SCALE())
        return (time.perf_counter() - t0) * self._scale


class SelectCase(Case):
    launches_per_step = 3  # query prep + partial + merge
    kernel_calls = "mla_absorb_sel8: query prep + attn_tc_kernel (row gather) + log-sum-exp merge"
    step_desc = "mla_absorb_sel8 over B=8 sequences: query prep + gathered-row partial + log-sum-exp merge"

    def __init__(self, kv, torch, dev, w):
        import synth
        self.kv, self.torch, self.w = kv, torch, w
        B, H, T, NS = w.B, w.H, w.T, w.NS
        self.kv8 = torch.empty((B * T, 576), dtype=torch.uint8, device=dev)
        self.sc = torch.empty(B * T, dtype=torch.float32, device=dev)
        chunk = 65536
        for b in range(B):
            for start in range(0, T, chunk):
                x = torch.from_numpy(synth.rows_for(w, b, start, chunk)).to(dev)
                r0 = b * T + start
                kv.kv8_quant_rows(x, self.kv8[r0:r0 + chunk], self.sc[r0:r0 + chunk])
        torch.cuda.synchronize(dev)
        self.idx_np = synth.selection_for(w)
        self.idx = torch.from_numpy(self.idx_np).to(dev)
        ql, qr = synth.queries_for(w)
        self.q_lat, self.q_rope = _bf16(torch, dev, ql), _bf16(torch, dev, qr)
        self.ws = torch.empty(kv.mla_sel8_workspace_bytes(B, H, NS) // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((B, H, 512), dtype=torch.float32, device=dev)
        self.pack = Packed(torch, dev, [self.q_lat, self.q_rope, self.idx])
        self.h_out = torch.empty((B, H, 512), dtype=torch.float32).pin_memory()
        self.h2d = self.pack.nbytes
        self.d2h = self.h_out.numel() * 4
        # listed rows (576 bytes + scale each), the index lists, the queries and the output
        self.alg_bytes = B * NS * (ROW_BYTES + 4) + self.q_lat.numel() * 2 + self.q_rope.numel() * 2 + \
            self.out.numel() * 4
        self.alg_bytes_step = self.alg_bytes
        self.flops = float(FLOP_PER_ROW_HEAD) * H * B * NS

    def _sel(self, stream):
        w = self.w
        self.kv.mla_absorb_sel8(self.q_lat, self.q_rope, self.kv8, self.sc, w.T, w.T, self.idx, SM_SCALE(), self.ws,
                                self.out, stream=stream)

    def step(self, stream, ev=None):
        if ev is not None:
            ev[0].record(stream)
        self._sel(stream)
        if ev is not None:
            ev[1].record(stream)

    def kernel_call(self, stream):
        self._sel(stream)

    def e2e_step(self, stream):
        kv, w = self.kv, self.w
        self.pack.upload(kv, stream)
        q_lat, q_rope, idx = self.pack.views
        kv.mla_absorb_sel8(q_lat, q_rope, self.kv8, self.sc, w.T, w.T, idx, SM_SCALE(), self.ws, self.out,
                           stream=stream)
        kv.kv8_copy(self.h_out, self.out, stream=stream)

    def config(self):
        w = self.w
        return {"B": w.B, "H": w.H, "T": w.T, "NS": w.NS}

    def oracle_setup(self, n_heads):
        import oracle
        import synth
        w = self.w
        rows = np.concatenate([synth.rows_for(w, b, 0, w.T)[self.idx_np[b]] for b in range(w.B)])
        q_o, s_o = oracle.quant_rows(rows)            # only the listed rows: index i of sequence b -> b*NS + i
        ql, qr = synth.queries_for(w)
        heads = np.linspace(0, w.H - 1, n_heads).astype(int)
        idx_local = np.tile(np.arange(w.NS, dtype=np.int32), (w.B, 1))
        self._o = (q_o, s_o, np.ascontiguousarray(ql[:, heads]), np.ascontiguousarray(qr[:, heads]), idx_local)
        self._scale = w.H / n_heads
        return (f"{n_heads} of {w.H} heads of all B={w.B} sequences over their NS={w.NS} listed rows, "
                f"scaled x{w.H // n_heads} to one step")

    def oracle_step(self) -> float:
        import oracle
        q_o, s_o, ql, qr, idx_local = self._o
        t0 = time.perf_counter()
        oracle.attn_select(ql, qr, q_o, s_o, self.w.NS, self.w.NS, idx_local, SM_SCALE())
        return (time.perf_counter() - t0) * self._scale


class PrefillCase(Case):
    unit = "us/chunk"
    launches_per_step = 2  # quant of the chunk's rows + prefill
    kernel_calls = "mla_absorb_prefill8: attn_tc_kernel"
    step_desc = "kv8_quant_rows(1024 fresh rows) + causal prefill of 1024 queries"

    def __init__(self, kv, torch, dev, w):
        import synth
        self.kv, self.torch, self.w = kv, torch, w
        H, T, S, pos0 = w.H, w.T, w.S, w.pos0
        self.kv8 = torch.empty((T, 576), dtype=torch.uint8, device=dev)
        self.sc = torch.empty(T, dtype=torch.float32, device=dev)
        x = torch.from_numpy(synth.rows_for(w)).to(dev)
        kv.kv8_quant_rows(x[:pos0], self.kv8[:pos0], self.sc[:pos0])   # the resident prefix
        self.fresh = x[pos0:].clone()                                   # the chunk's rows
        del x
        ql, qr = synth.queries_for(w)
        self.q_lat, self.q_rope = _bf16(torch, dev, ql), _bf16(torch, dev, qr)
        self.out = torch.empty((S, H, 512), dtype=torch.float32, device=dev)
        self.pack = Packed(torch, dev, [self.q_lat, self.q_rope, self.fresh])
        self.h_out = torch.empty((S, H, 512), dtype=torch.float32).pin_memory()
        self.h2d = self.pack.nbytes
        self.d2h = self.h_out.numel() * 4
        self.alg_bytes = T * ROW_BYTES + self.q_lat.numel() * 2 + self.q_rope.numel() * 2 + self.out.numel() * 4
        self.alg_bytes_step = self.alg_bytes + self.fresh.numel() * 4 + S * ROW_BYTES
        n_pairs = S * pos0 + S * (S + 1) // 2           # (query, row) pairs under the causal mask
        self.flops = float(FLOP_PER_ROW_HEAD) * H * n_pairs

    def step(self, stream, ev=None):
        kv, w = self.kv, self.w
        kv.kv8_quant_rows(self.fresh, self.kv8[w.pos0:], self.sc[w.pos0:], stream=stream)
        if ev is not None:
            ev[0].record(stream)
        kv.mla_absorb_prefill8(self.q_lat, self.q_rope, w.pos0, self.kv8, self.sc, w.T, SM_SCALE(), self.out,
                               stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def kernel_call(self, stream):
        w = self.w
        self.kv.mla_absorb_prefill8(self.q_lat, self.q_rope, w.pos0, self.kv8, self.sc, w.T, SM_SCALE(), self.out,
                                    stream=stream)

    def e2e_step(self, stream):
        kv, w = self.kv, self.w
        self.pack.upload(kv, stream)
        q_lat, q_rope, fresh = self.pack.views
        kv.kv8_quant_rows(fresh, self.kv8[w.pos0:], self.sc[w.pos0:], stream=stream)
        kv.mla_absorb_prefill8(q_lat, q_rope, w.pos0, self.kv8, self.sc, w.T, SM_SCALE(), self.out, stream=stream)
        kv.kv8_copy(self.h_out, self.out, stream=stream)

    def config(self):
        w = self.w
        return {"S": w.S, "H": w.H, "T": w.T, "pos0": w.pos0}

    def oracle_setup(self, n_heads):
        import oracle
        import synth
        w = self.w
        rows = synth.rows_for(w)
        q_o, s_o = oracle.quant_rows(rows)
        ql, qr = synth.queries_for(w)
        nq = 2
        qsel = np.array([0, w.S - 1])[:nq]                # the first and last query of the chunk
        heads = np.linspace(0, w.H - 1, n_heads).astype(int)
        self._o = (q_o, s_o, [np.ascontiguousarray(ql[i][heads]) for i in qsel],
                   [np.ascontiguousarray(qr[i][heads]) for i in qsel], [w.pos0 + int(i) + 1 for i in qsel])
        n_pairs = w.S * w.pos0 + w.S * (w.S + 1) // 2
        self._scale = (w.H / n_heads) * n_pairs / sum(self._o[4])
        return (f"{n_heads} of {w.H} heads of the chunk's first and last query ({sum(self._o[4])} causal rows), "
                f"scaled by (query, row, head) triples to the whole chunk")

    def oracle_step(self) -> float:
        import oracle
        q_o, s_o, qls, qrs, lens = self._o
        t0 = time.perf_counter()
        for ql, qr, n in zip(qls, qrs, lens):
            oracle.attn_decode(ql, qr, q_o[:n], s_o[:n], SM_SCALE())
        return (time.perf_counter() - t0) * self._scale


class ProjCase(Case):
    """The absorb projections through an fmt=8 kv_b: q_nope -> q_lat (bf16, the attention's query) and a
    context -> the head outputs, both on one stream.  A decode step (S = 1) reads every weight byte once
    on the CUDA cores; a prefill chunk (S = 1024) runs on the tensor cores; both are HBM-bound."""
    launches_per_step = 2
    kernel_calls = "mla_q_absorb8 + mla_out_project8"

    @property
    def unit(self):
        return "us/chunk" if self.w.S > 1 else "us/layer-step"

    step_desc = "q_nope -> q_lat (bf16) through the kv_b key rows + context -> head output through the value rows"
    dtype = "e4m3*f32->f32"

    def __init__(self, kv, torch, dev, w):
        import synth
        self.kv, self.torch, self.w = kv, torch, w
        S, H = w.S, w.H
        self.w8_np, self.sc_np = synth.kvb_fmt8(H)
        self.w8 = torch.from_numpy(self.w8_np).to(dev)
        self.wsc = torch.from_numpy(self.sc_np).to(dev)
        self.q_nope = _bf16(torch, dev, synth.q_nope_for(w))
        self.ctx = torch.from_numpy(synth.context_for(w)).to(dev)
        self.q_lat = torch.empty((S, H, 512), dtype=torch.bfloat16, device=dev)
        self.out = torch.empty((S, H, 128), dtype=torch.float32, device=dev)
        self.pack = Packed(torch, dev, [self.q_nope, self.ctx])
        self.h_q_lat = torch.empty((S, H, 512), dtype=torch.bfloat16).pin_memory()
        self.h_out = torch.empty((S, H, 128), dtype=torch.float32).pin_memory()
        self.h2d = self.pack.nbytes
        self.d2h = self.h_q_lat.numel() * 2 + self.h_out.numel() * 4
        act = self.q_nope.numel() * 2 + self.q_lat.numel() * 2 + self.ctx.numel() * 4 + self.out.numel() * 4
        self.alg_bytes = self.w8_np.nbytes + self.sc_np.nbytes + act
        self.alg_bytes_step = self.alg_bytes
        self.flops = 2.0 * S * H * 128 * 512 * 2  # two products of 128 x 512 per (row, head)

    def step(self, stream, ev=None):
        if ev is not None:
            ev[0].record(stream)
        self.kernel_call(stream)
        if ev is not None:
            ev[1].record(stream)

    def kernel_call(self, stream):
        self.kv.mla_q_absorb8(self.q_nope, self.w8, self.wsc, self.q_lat, stream=stream)
        self.kv.mla_out_project8(self.ctx, self.w8, self.wsc, self.out, stream=stream)

    def e2e_step(self, stream):
        kv = self.kv
        self.pack.upload(kv, stream)
        q_nope, ctx = self.pack.views
        kv.mla_q_absorb8(q_nope, self.w8, self.wsc, self.q_lat, stream=stream)
        kv.mla_out_project8(ctx, self.w8, self.wsc, self.out, stream=stream)
        kv.kv8_copy(self.h_q_lat, self.q_lat, stream=stream)
        kv.kv8_copy(self.h_out, self.out, stream=stream)

    def config(self):
        return {"S": self.w.S, "H": self.w.H, "kv_b": "fmt=8: 128x256 rows x 512 e4m3 bytes, 128x128-block f32 scales"}

    def roofline(self, kern_s, peaks, key):
        # both shapes sit below the ridge (S = 1: 2 flop per weight byte; S = 1024: ~68 flop per byte of
        # activations in and out), so the bound is HBM; the tensor-core rate is reported beside it
        hbm_gbs = self.alg_bytes / kern_s / 1e9
        tflops = self.flops / kern_s / 1e12
        kern = "q_absorb_small + out_project_small (proj8.cu, CUDA cores)" if self.w.S <= 8 else \
            "q_absorb_tc_kernel + out_project_tc_kernel (proj8_tc.cu, tcgen05 kind::f16)"
        return {"bound": "hbm", "achieved": hbm_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": hbm_gbs / peaks["hbm_gbs"], "peak_source": f"copy bandwidth ({peaks['source']})",
                "kernel": kern, "events_bracket": self.kernel_calls,
                # DRAM bytes of one launch of each of the two kernels (one step)
                "traffic": traffic_per_launch(key, "proj8_small_kernels", PROJ_SMALL_SOURCES) if self.w.S <= 8
                else traffic_per_launch(key, "proj8_tc_kernels", PROJ_TC_SOURCES),
                "algorithmic_bytes": self.alg_bytes, "algorithmic_flops": self.flops,
                "kernel_us": kern_s * 1e6, "hbm_gbs": hbm_gbs, "hbm_frac": hbm_gbs / peaks["hbm_gbs"],
                "hbm_peak_gbs": peaks["hbm_gbs"], "tflops": tflops,
                "tensor_frac_of_bf16_peak": tflops / peaks["bf16_tflops"] if self.w.S > 8 else None}

    def oracle_setup(self, n_rows):
        import synth
        w = self.w
        if not hasattr(self, "w8_np"):
            self.w8_np, self.sc_np = synth.kvb_fmt8(w.H)
        rows = np.unique(np.linspace(0, w.S - 1, min(n_rows, w.S)).astype(int))
        self._o = (np.ascontiguousarray(synth.q_nope_for(w)[rows]), np.ascontiguousarray(synth.context_for(w)[rows]))
        self._scale = w.S / len(rows)
        return f"{len(rows)} of {w.S} query rows, all {w.H} heads, both projections, scaled by rows to the whole step"

    def oracle_step(self) -> float:
        import oracle
        q, x = self._o
        t0 = time.perf_counter()
        oracle.q_absorb(q, self.w8_np, self.sc_np)
        oracle.out_project(x, self.w8_np, self.sc_np)
        return (time.perf_counter() - t0) * self._scale


class IndexerCase(Case):
    """The DSA lightning indexer for B queries: e4m3 index keys streamed from HBM through the tensor cores
    (scores), then the top-NS positions of each query."""
    launches_per_step = 2  # score kernel + top-k kernel (plus a memset of the top-k's counters)
    kernel_calls = "dsa_index_topk8: index_score_kernel + topk_kernel"
    step_desc = "index scores (e4m3 query x e4m3 keys, ReLU-weighted head sum) + top-2048 per query"
    dtype = "e4m3*e4m3->f32"

    def __init__(self, kv, torch, dev, w):
        import synth
        self.kv, self.torch, self.w = kv, torch, w
        B, T, HI = w.B, w.T, w.H
        self.k8 = torch.empty((B * T, 128), dtype=torch.uint8, device=dev)
        self.ks = torch.empty(B * T, dtype=torch.float32, device=dev)
        for b in range(B):
            rows = torch.from_numpy(synth.index_keys_for(w, b)).to(dev)
            kv.kv8_quant_rows_w(rows, self.k8[b * T:(b + 1) * T], self.ks[b * T:(b + 1) * T])
            del rows
        self.q = _bf16(torch, dev, synth.index_queries_for(w))
        self.wts = torch.from_numpy(synth.index_weights_for(w)).to(dev)
        self.scores = torch.empty((B, T), dtype=torch.float32, device=dev)
        self.idx = torch.empty((B, w.NS), dtype=torch.int32, device=dev)
        self.ws = torch.empty(kv.dsa_index_workspace_bytes(B) // 4, dtype=torch.int32, device=dev)
        self.pack = Packed(torch, dev, [self.q, self.wts])
        self.h_idx = torch.empty((B, w.NS), dtype=torch.int32).pin_memory()
        self.h2d = self.pack.nbytes
        self.d2h = self.h_idx.numel() * 4
        self.alg_bytes = (B * T * (128 + 4) + self.q.numel() * 2 + self.wts.numel() * 4 + B * T * 4
                          + self.idx.numel() * 4)
        self.alg_bytes_step = self.alg_bytes
        self.flops = 2.0 * B * T * HI * 128

    def _call(self, q, wts, stream):
        w = self.w
        self.kv.dsa_index_topk8(q, wts, self.k8, self.ks, w.T, w.T, w.NS, self.ws, self.scores, self.idx,
                                stream=stream)

    def step(self, stream, ev=None):
        if ev is not None:
            ev[0].record(stream)
        self._call(self.q, self.wts, stream)
        if ev is not None:
            ev[1].record(stream)

    def kernel_call(self, stream):
        self._call(self.q, self.wts, stream)

    def e2e_step(self, stream):
        kv = self.kv
        self.pack.upload(kv, stream)
        q, wts = self.pack.views
        self._call(q, wts, stream)
        kv.kv8_copy(self.h_idx, self.idx, stream=stream)

    def config(self):
        w = self.w
        return {"B": w.B, "T": w.T, "index_heads": w.H, "index_dim": 128, "NS": w.NS}

    def roofline(self, kern_s, peaks, key):
        hbm_gbs = self.alg_bytes / kern_s / 1e9
        tflops = self.flops / kern_s / 1e12
        return {"bound": "hbm", "achieved": hbm_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": hbm_gbs / peaks["hbm_gbs"], "peak_source": f"copy bandwidth ({peaks['source']})",
                "kernel": "index_score_kernel + topk_kernel (indexer.cu)", "events_bracket": self.kernel_calls,
                "traffic": traffic_per_launch(key, "index_score_kernel", IDX_SOURCES),
                "algorithmic_bytes": self.alg_bytes, "algorithmic_flops": self.flops, "kernel_us": kern_s * 1e6,
                "hbm_gbs": hbm_gbs, "hbm_frac": hbm_gbs / peaks["hbm_gbs"], "hbm_peak_gbs": peaks["hbm_gbs"],
                "tflops": tflops, "tensor_frac_of_fp8_peak": tflops / (2.0 * peaks["bf16_tflops"])}

    def oracle_setup(self, n_seq):
        import oracle
        import synth
        w = self.w
        n_seq = max(1, min(n_seq, w.B))
        q8, qs = oracle.quant_rows_w(synth.index_queries_for(w).reshape(w.B * w.H, 128), 128)
        q8, qs = q8.reshape(w.B, w.H, 128), qs.reshape(w.B, w.H)
        wts = synth.index_weights_for(w)
        keys = [oracle.quant_rows_w(synth.index_keys_for(w, b), 128) for b in range(n_seq)]
        self._o = (q8[:n_seq], qs[:n_seq], wts[:n_seq], keys)
        self._scale = w.B / n_seq
        return (f"{n_seq} of {w.B} queries over all T={w.T} index keys (the index query quantized first), "
                f"scaled by queries to the whole step")

    def oracle_step(self) -> float:
        import oracle
        q8, qs, wts, keys = self._o
        t0 = time.perf_counter()
        for b, (k8, ks) in enumerate(keys):
            sc = oracle.index_scores(q8[b:b + 1], qs[b:b + 1], wts[b:b + 1], k8, ks, self.w.T, 0)
            oracle.topk(sc[0], self.w.NS)
        return (time.perf_counter() - t0) * self._scale


class BatchDecodeCase(Case):
    """One decode step for B sequences at once: the fresh row of each sequence appended to its own cache
    (one scatter call), then the batched split-T partials and the merge."""
    launches_per_step = 5  # scatter quant + prep + partial + merge (+ the partial's dependent launch)
    kernel_calls = "mla_absorb_batch_decode8: query prep + attn_tc_kernel + lse_merge_kernel"
    step_desc = "kv8_quant_rows_scatter(B fresh rows) + batched split-T decode + log-sum-exp merge"

    def __init__(self, kv, torch, dev, w):
        import synth
        self.kv, self.torch, self.w = kv, torch, w
        B, T, H = w.B, w.T, w.H
        self.lens_list = synth.batch_lengths(w)
        self.kv8 = torch.zeros((B * T, 576), dtype=torch.uint8, device=dev)
        self.sc = torch.zeros(B * T, dtype=torch.float32, device=dev)
        fresh, dst = [], []
        for b in range(B):
            n = self.lens_list[b]
            x = torch.from_numpy(synth.rows_for(w, b, 0, n)).to(dev)
            kv.kv8_quant_rows(x[:-1], self.kv8[b * T:b * T + n - 1], self.sc[b * T:b * T + n - 1])
            fresh.append(x[-1:].clone())
            dst.append(b * T + n - 1)
            del x
        self.fresh = torch.cat(fresh)
        self.dst = torch.tensor(dst, dtype=torch.int64, device=dev)
        self.lens = torch.tensor(self.lens_list, dtype=torch.int32, device=dev)
        ql, qr = synth.queries_for(w, B)
        self.q_lat, self.q_rope = _bf16(torch, dev, ql), _bf16(torch, dev, qr)
        self.ws = torch.empty(kv.mla_batch_decode8_workspace_bytes(B, H, T) // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((B, H, 512), dtype=torch.float32, device=dev)
        self.pack = Packed(torch, dev, [self.q_lat, self.q_rope, self.fresh])
        self.h_out = torch.empty((B, H, 512), dtype=torch.float32).pin_memory()
        self.h2d = self.pack.nbytes
        self.d2h = self.h_out.numel() * 4
        rows = sum(self.lens_list)
        self.alg_bytes = rows * ROW_BYTES + self.q_lat.numel() * 2 + self.q_rope.numel() * 2
        self.alg_bytes_step = rows * ROW_BYTES + self.h2d + self.d2h
        self.flops = float(FLOP_PER_ROW_HEAD) * H * rows

    def _decode(self, q_lat, q_rope, stream):
        w = self.w
        self.kv.mla_absorb_batch_decode8(q_lat, q_rope, self.kv8, self.sc, w.T, w.T, self.lens, SM_SCALE(), self.ws,
                                         self.out, stream=stream)

    def step(self, stream, ev=None):
        self.kv.kv8_quant_rows_scatter(self.fresh, self.dst, self.kv8, self.sc, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        self._decode(self.q_lat, self.q_rope, stream)
        if ev is not None:
            ev[1].record(stream)

    def kernel_call(self, stream):
        self._decode(self.q_lat, self.q_rope, stream)

    def e2e_step(self, stream):
        kv = self.kv
        self.pack.upload(kv, stream)
        q_lat, q_rope, fresh = self.pack.views
        kv.kv8_quant_rows_scatter(fresh, self.dst, self.kv8, self.sc, stream=stream)
        self._decode(q_lat, q_rope, stream)
        kv.kv8_copy(self.h_out, self.out, stream=stream)

    def config(self):
        w = self.w
        return {"B": w.B, "H": w.H, "T_max": w.T, "lengths": getattr(self, "lens_list", None)}

    def oracle_setup(self, n_heads):
        import oracle
        import synth
        w = self.w
        self.lens_list = synth.batch_lengths(w)
        ql, qr = synth.queries_for(w, w.B)
        heads = np.linspace(0, w.H - 1, n_heads).astype(int)
        self._o = []
        for b in range(w.B):
            q_o, s_o = oracle.quant_rows(synth.rows_for(w, b, 0, self.lens_list[b]))
            self._o.append((np.ascontiguousarray(ql[b][heads]), np.ascontiguousarray(qr[b][heads]), q_o, s_o))
        self._scale = w.H / n_heads
        return f"{n_heads} of {w.H} heads of every sequence over its whole length, scaled by heads to the step"

    def oracle_step(self) -> float:
        import oracle
        t0 = time.perf_counter()
        for ql, qr, q_o, s_o in self._o:
            oracle.attn_decode(ql, qr, q_o, s_o, SM_SCALE())
        return (time.perf_counter() - t0) * self._scale


class MixedDecodeCase(Case):
    """One decode step over the mixed-precision cache: the fresh row's no-position part quantized into the
    cache and its bf16 RoPE part stored, then the decode (tensor cores) and the merge."""
    launches_per_step = 5  # quant (448) + RoPE copy + query prep + partial + merge
    kernel_calls = "mla_absorb_mixed_decode8: mixed_prep_kernel + attn_mixed_tc_kernel + lse_merge_kernel"
    step_desc = "kv8_quant_rows_w(fresh row, width 448) + RoPE copy + mixed-cache split-T decode + merge"
    dtype = "e4m3*e4m3 + bf16*bf16 -> f32"

    def __init__(self, kv, torch, dev, w):
        import synth
        self.kv, self.torch, self.w = kv, torch, w
        H, T = w.H, w.T
        nope, rope = synth.mixed_rows_for(w)
        self.k8 = torch.empty((T, 448), dtype=torch.uint8, device=dev)
        self.ks = torch.empty(T, dtype=torch.float32, device=dev)
        xn = torch.from_numpy(nope).to(dev)
        kv.kv8_quant_rows_w(xn[:-1], self.k8[:-1], self.ks[:-1])
        self.fresh_nope = xn[-1:].clone()
        del xn
        self.k_rope = torch.from_numpy(rope).to(dev).to(torch.bfloat16)
        self.fresh_rope = self.k_rope[-1:].clone()
        qn, qr = synth.mixed_queries_for(w)
        self.qn, self.qr = _bf16(torch, dev, qn), _bf16(torch, dev, qr)
        self.ws = torch.empty(kv.mla_mixed_decode8_workspace_bytes(H, T) // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((H, 512), dtype=torch.float32, device=dev)
        self.pack = Packed(torch, dev, [self.qn, self.qr, self.fresh_nope, self.fresh_rope])
        self.h_out = torch.empty((H, 512), dtype=torch.float32).pin_memory()
        self.h2d = self.pack.nbytes
        self.d2h = self.h_out.numel() * 4
        self.alg_bytes = T * (448 + 4 + 128) + self.qn.numel() * 2 + self.qr.numel() * 2
        self.alg_bytes_step = self.alg_bytes + self.d2h
        self.flops = 2.0 * H * T * (448 + 64 + 512)

    def _decode(self, qn, qr, stream):
        self.kv.mla_absorb_mixed_decode8(qn, qr, self.k8, self.ks, self.k_rope, SM_SCALE(), self.ws, self.out,
                                         stream=stream)

    def _append(self, fresh_nope, fresh_rope, stream):
        T = self.w.T
        self.kv.kv8_quant_rows_w(fresh_nope, self.k8[T - 1:], self.ks[T - 1:], stream=stream)
        self.kv.kv8_copy(self.k_rope[T - 1:], fresh_rope, stream=stream)

    def step(self, stream, ev=None):
        self._append(self.fresh_nope, self.fresh_rope, stream)
        if ev is not None:
            ev[0].record(stream)
        self._decode(self.qn, self.qr, stream)
        if ev is not None:
            ev[1].record(stream)

    def kernel_call(self, stream):
        self._decode(self.qn, self.qr, stream)

    def e2e_step(self, stream):
        kv = self.kv
        self.pack.upload(kv, stream)
        qn, qr, fn, fr = self.pack.views
        self._append(fn, fr, stream)
        self._decode(qn, qr, stream)
        kv.kv8_copy(self.h_out, self.out, stream=stream)

    def config(self):
        w = self.w
        return {"H": w.H, "T": w.T, "row": "448 e4m3 + f32 scale + 64 bf16"}

    def roofline(self, kern_s, peaks, key):
        # the score and the context are e4m3 contractions but for the RoPE parts (bf16): the fp8 peak
        # (measured bf16 burst x 2) is the ceiling of the whole
        hbm_gbs = self.alg_bytes / kern_s / 1e9
        tflops = self.flops / kern_s / 1e12
        peak = peaks["bf16_tflops"] * 2.0
        return {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                "peak_source": f"fp8 = 2 x bf16 burst ({peaks['source']})",
                "kernel": "attn_mixed_tc_kernel (attn_mixed.cu) + lse_merge_kernel", "events_bracket": self.kernel_calls,
                "traffic": traffic_per_launch(key, "attn_mixed_tc_kernel", MIXED_SOURCES),
                "algorithmic_bytes": self.alg_bytes, "algorithmic_flops": self.flops, "kernel_us": kern_s * 1e6,
                "hbm_gbs": hbm_gbs, "hbm_frac": hbm_gbs / peaks["hbm_gbs"], "hbm_peak_gbs": peaks["hbm_gbs"],
                "tflops": tflops}

    def oracle_setup(self, n_heads):
        import oracle
        import synth
        w = self.w
        nope, rope = synth.mixed_rows_for(w)
        k8, ks = oracle.quant_rows_w(nope, 448)
        qn, qr = synth.mixed_queries_for(w)
        heads = np.linspace(0, w.H - 1, n_heads).astype(int)
        self._o = (np.ascontiguousarray(qn[heads]), np.ascontiguousarray(qr[heads]), k8, ks, rope)
        self._scale = w.H / n_heads
        return f"{n_heads} of {w.H} heads over all T={w.T} rows, scaled by heads to the step"

    def oracle_step(self) -> float:
        import oracle
        qn, qr, k8, ks, rope = self._o
        t0 = time.perf_counter()
        oracle.attn_mixed_decode(qn, qr, k8, ks, rope, SM_SCALE())
        return (time.perf_counter() - t0) * self._scale


CASES = {"dec262k": DecodeCase, "dec16k": DecodeCase, "dsa": SelectCase, "prefill": PrefillCase,
         "proj_dec": ProjCase, "proj_prefill": ProjCase, "indexer": IndexerCase, "batch_dec": BatchDecodeCase,
         "mixed_dec": MixedDecodeCase}
# the oracle's sample: heads for the attention workloads, query rows for the projections
ORACLE_HEADS = {"dec262k": 32, "dec16k": 128, "dsa": 128, "prefill": 8, "proj_dec": 1, "proj_prefill": 64,
                "indexer": 1, "batch_dec": 16, "mixed_dec": 32}
REFERENCE_HEADS = {"dec262k": 8, "dec16k": 32, "dsa": 32, "prefill": 4, "proj_dec": 1, "proj_prefill": 16,
                   "indexer": 1, "batch_dec": 4, "mixed_dec": 8}
# workloads whose oracle sample is a set of heads (the oracle runs one thread per head, or per (query,
# head)): the reference arm samples at least as many heads as the oracle has threads, so its per-head
# rate is that of a full host
HEAD_SAMPLED = {"dec262k", "dec16k", "dsa", "prefill", "batch_dec", "mixed_dec"}


def reference_sample(key: str, w, threads: int) -> int:
    n = REFERENCE_HEADS[key]
    if key in HEAD_SAMPLED:
        n = min(w.H, max(n, threads))
    return n


def SM_SCALE():
    import synth
    return synth.SM_SCALE


def metric_for(key: str) -> str:
    if key == "dec262k":
        return HEADLINE_METRIC
    import synth
    return f"fp8 MLA {key} step time ({synth.DESCRIPTIONS[key]})"


# --------------------------------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample of the workload
# --------------------------------------------------------------------------------------------------
def cpu_baseline(case: Case, n_heads: int, key: str = "") -> dict:
    import oracle
    sample = case.oracle_setup(n_heads)
    t_us = case.oracle_step() * 1e6
    out = {"value": t_us, "unit": case.unit, "cores": oracle.num_threads(), "kind": "oracle", "sample": sample}
    if key in ("dec262k", "dec16k"):
        out["single_thread"] = single_thread_decode_baselines()
    return out


# heads timed single-threaded per decode workload (scaled by heads to the whole step)
SINGLE_THREAD_HEADS = {"tiny": 16, "dec16k": 8, "dec262k": 1}


def single_thread_decode_baselines() -> dict:
    """The oracle on ONE host thread for the three decode workloads (tiny, dec16k, dec262k), each on a
    bounded sample of heads over all rows, scaled by heads to one layer-step."""
    import oracle
    import synth
    threads = oracle.num_threads()
    res = {}
    try:
        for key, nh in SINGLE_THREAD_HEADS.items():
            w = synth.WORKLOADS[key]
            rows = synth.rows_for(w)
            oracle.set_num_threads(threads)      # set-up (the cache bytes) on all threads, untimed
            q_o, s_o = oracle.quant_rows(rows)
            oracle.set_num_threads(1)
            ql, qr = synth.queries_for(w, 1)
            heads = np.linspace(0, w.H - 1, nh).astype(int)
            qls, qrs = np.ascontiguousarray(ql[0][heads]), np.ascontiguousarray(qr[0][heads])
            t0 = time.perf_counter()
            oracle.quant_rows(rows[-1:])
            oracle.attn_decode(qls, qrs, q_o, s_o, synth.SM_SCALE)
            dt = (time.perf_counter() - t0) * w.H / nh
            res[key] = {"value": dt * 1e6, "unit": "us/layer-step", "cores": 1,
                        "sample": f"{nh} of {w.H} heads over all T={w.T} rows, scaled x{w.H / nh:g}"}
    finally:
        oracle.set_num_threads(threads)
    return res


def host_case(key: str):
    import synth
    w = synth.WORKLOADS[key]
    c = CASES[key].__new__(CASES[key])
    c.w = w
    if key in ("dec262k", "dec16k"):
        c.rows = synth.rows_for(w)
    elif key == "dsa":
        c.idx_np = synth.selection_for(w)
    return c


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
    key = args.workload
    case = host_case(key)
    sample = case.oracle_setup(reference_sample(key, case.w, oracle.num_threads()))
    for _ in range(args.warmup):
        case.oracle_step()
    t0 = time.perf_counter()
    ts = [case.oracle_step() for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    us = statistics.mean(ts) * 1e6
    cfg = dict({"workload": synth.DESCRIPTIONS[key], "sample": sample}, **case.config())
    line = {"impl": "reference", "metric": metric_for(key), "value": us, "unit": case.unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1000.0, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "wall_s": wall,
            "cpu_baseline": {"value": us, "unit": case.unit, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": us, "unit": case.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
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
    key = args.workload
    w = synth.WORKLOADS[key]
    case = CASES[key](kv, torch, dev, w)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    # The L2 flush writes a buffer twice the L2's size, then reads a second one as large.  The write evicts
    # every line of the step's data; the read evicts the write's dirty lines in turn.  So a timed step
    # starts with none of its data in L2 and nothing to write back.  After the write alone, ~129 MB of
    # dirty lines would be written back during the step, sharing the DRAM with its reads.
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def l2_flush():
        flush.zero_()
        torch.sum(flush_rd, dim=0, out=flush_sink)

    stream = torch.cuda.Stream(device=dev)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            l2_flush()
            case.step(stream)
            case.e2e_step(stream)
    torch.cuda.synchronize(dev)

    # One step is captured once as a CUDA graph and replayed: the same library calls and kernels, without
    # the host's per-call launch cost (about 12 us per call from Python) between them.  The graph holds
    # no events: an event node between two calls would cut the programmatic dependent launch that lets
    # a kernel start while its predecessor drains.  The dominant call is timed from its own graph,
    # replayed after each step (L2 flushed before each).
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        case.step(stream)
    k0, k1 = E(), E()
    g_kern = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_kern, stream=stream):
        case.kernel_call(stream)
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        case.e2e_step(stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            l2_flush()
            g_step.replay()
            g_kern.replay()
            g_e2e.replay()
    torch.cuda.synchronize(dev)

    # ---- device-timed steps (inputs resident), L2 flushed before each step outside the events
    step_ms, kern_ms = [], []
    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    for k in range(args.steps):
        e0, e1 = E(), E()
        with torch.cuda.stream(stream):
            l2_flush()
            e0.record(stream)
            g_step.replay()
            e1.record(stream)
            l2_flush()
            k0.record(stream)
            g_kern.replay()
            k1.record(stream)
        k1.synchronize()
        e1.synchronize()
        step_ms.append(e0.elapsed_time(e1))
        kern_ms.append(k0.elapsed_time(k1))
    torch.cuda.synchronize(dev)
    barrier()
    wall_s = time.perf_counter() - t_wall
    clk = clocks.stop() if rank == 0 else {}
    ms_per_step = reduce_max(statistics.mean(step_ms), dev)
    kern_ms_mean = reduce_max(statistics.mean(kern_ms), dev)

    # ---- the same steps without the L2 flush (a workload whose rows fit in L2 then reads them from L2)
    warm_ms = []
    for k in range(args.steps):
        e0, e1 = E(), E()
        with torch.cuda.stream(stream):
            e0.record(stream)
            g_step.replay()
            e1.record(stream)
        e1.synchronize()
        warm_ms.append(e0.elapsed_time(e1))
    warm_ms_mean = reduce_max(statistics.mean(warm_ms), dev)

    # ---- the same steps after the write alone (the flush's dirty lines written back during the step)
    wflush_ms = []
    for k in range(args.steps):
        e0, e1 = E(), E()
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            g_step.replay()
            e1.record(stream)
        e1.synchronize()
        wflush_ms.append(e0.elapsed_time(e1))
    wflush_ms_mean = reduce_max(statistics.mean(wflush_ms), dev)

    # ---- clock soak: >= 1 s of back-to-back step replays with the clocks sampled throughout
    soak = None
    if rank == 0 and not args.no_soak:
        # replays are enqueued in batches until at least 1.1 s of GPU time has passed
        batch = max(10, int(0.1 / max(ms_per_step * 1e-3, 1e-6)) + 1)
        sampler = ClockSampler(local_rank)
        sampler.start()
        s0, s1 = E(), E()
        n_soak = 0
        with torch.cuda.stream(stream):
            s0.record(stream)
            while True:
                for _ in range(batch):
                    g_step.replay()
                n_soak += batch
                s1.record(stream)
                s1.synchronize()
                if s0.elapsed_time(s1) >= 1100.0:
                    break
        s1.synchronize()
        sclk = sampler.stop()
        soak_ms = s0.elapsed_time(s1)
        us_soak = soak_ms * 1e3 / n_soak
        soak = {"seconds": soak_ms / 1e3, "steps": n_soak, "us_per_step": us_soak,
                "sm_mhz_median": sclk.get("sm_mhz"), "sm_max_mhz": sclk.get("sm_max_mhz"),
                "reasons": sclk.get("reasons"), "samples": sclk.get("samples"),
                "power_w_max": sclk.get("power_w_max"),
                "cycles_per_step": us_soak * sclk["sm_mhz"] if sclk.get("sm_mhz") else None,
                "how": "step graph replayed back to back (no L2 flush) for >= 1 s; cycles = us x median SM MHz"}
    barrier()

    # ---- end to end through the C ABI with host buffers: inputs in, output out, every step; as a
    # replayed graph of the same calls, and as direct calls (each paying the host's launch cost)
    def timed(fn):
        ev = [(E(), E()) for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                l2_flush()
                ev[k][0].record(stream)
                fn()
                ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        return reduce_max(statistics.mean([a.elapsed_time(b) for a, b in ev]), dev)

    barrier()
    e2e_ms = timed(g_e2e.replay)
    e2e_direct_ms = timed(lambda: case.e2e_step(stream))
    barrier()

    if rank != 0:
        return
    peaks = measured_peaks()
    roof = case.roofline(kern_ms_mean / 1e3, peaks, key)

    n_heads = ORACLE_HEADS[key]
    base = cpu_baseline(case, n_heads, key) if (world == 1 and not args.no_cpu_baseline) else None
    value = whole_job_us_per_step(ms_per_step, world)
    cfg = {"workload": synth.DESCRIPTIONS[key]}
    cfg.update(case.config())
    cfg.update({"step": case.step_desc,
                "l2": (f"flushed before every timed step, outside the events: a {L2_FLUSH_BYTES >> 20} MiB write, then a "
                       f"{L2_FLUSH_BYTES >> 20} MiB read of a second buffer (none of the step's data and no dirty line left in L2)"),
                "timing": "each step is one replay of a CUDA graph of the step's library calls (captured once)",
                "parallelism": f"replicas x{world}"})
    line = {
        "metric": metric_for(key), "value": value, "unit": case.unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": case.dtype, "data": "synthetic", "config": cfg,
        "step_hbm_gbs": case.alg_bytes_step / (ms_per_step / 1e3) / 1e9,
        "step_hbm_frac": case.alg_bytes_step / (ms_per_step / 1e3) / 1e9 / peaks["hbm_gbs"],
        "e2e": {"value": whole_job_us_per_step(e2e_ms, world), "unit": case.unit, "h2d_bytes_per_step": case.h2d,
                "d2h_bytes_per_step": case.d2h, "how": "CUDA graph of the copies (kv8_copy kernels: pinned host -> device in, device -> pinned host out) and library calls, replayed",
                "direct_calls_value": whole_job_us_per_step(e2e_direct_ms, world)},
        "gpu_launches": case.launches_per_step * args.steps,
        "roofline": roof,
        "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "power_w_max")},
        "warm_l2": {"value": whole_job_us_per_step(warm_ms_mean, world), "unit": case.unit,
                    "how": "the same step replays without the L2 flush before each step"},
        "l2_write_flush": {"value": whole_job_us_per_step(wflush_ms_mean, world), "unit": case.unit,
                           "how": (f"the same step after the {L2_FLUSH_BYTES >> 20} MiB write alone: the write's "
                                   "dirty lines are written back during the step")},
        "clock_soak": soak,
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
    ap.add_argument("--no-soak", action="store_true", help="skip the 1 s clock soak (profiling runs)")
    ap.add_argument("--workload", choices=sorted(CASES), default="dec262k",
                    help="dec262k (default: the headline decode step), dec16k, dsa or prefill")
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
