"""Seeded synthetic inputs for the five workloads.

This module draws random numbers with the shapes, sizes and value distributions of the workloads
and nothing else: it holds no quantisation and no attention arithmetic.  Both the oracle tests and
the CUDA-path tests / benchmark take their inputs from here.

Generator: numpy's ``default_rng(seed)`` (PCG64), seed = 1000 + workload number.  Normal draws
are f32; "bf16 queries" are f32 N(0,1) draws rounded to bf16 by torch (round-to-nearest-even).

Workloads (one query position = one decode step of one layer):
  1 tiny      H=16,  T=256     rows N(0,1)*10^U(-3,2); row 17 all zero (element 0 = -0.0);
                               row 42 N(0,1)*1e-39 (subnormal amax); q f32 N(0,1)
  2 dec16k    H=128, T=16384   rows N(0,1)*10^U(-1,1); row T-1 is the fresh f32 row; q bf16
  3 dec262k   H=128, T=262144  as 2, plus a seeded 1% of rows times 50; q bf16
  4 dsa       B=8, H=128, T=131072 per sequence, NS=2048 sorted unique indices uniform in [0,T)
  5 prefill   S=1024, H=128, T=65536, pos0=64512; rows 64512.. are the fresh f32 rows; q bf16
  6 proj_dec      absorb projections, S=1, H=128: q_nope N(0,1) bf16, context N(0,1) f32, fmt=8 kv_b
  7 proj_prefill  the same for S=1024 query rows
  8 indexer   B=8 queries x 64 index heads x 128 (bf16 N(0,1)), head weights N(0,1)/8; per query its own
              T=131072 index-key rows N(0,1)*10^U(-0.5,0.5) of width 128; top NS=2048
  10 mixed_dec H=128, T=65536: rows of 448 no-position values N(0,1)*10^U(-1,1) (quantized in set-up) and 64
              RoPE values N(0,1) rounded to bf16; queries N(0,1) rounded to bf16 (448 + 64 per head)
  9 batch_dec B=8 sequences, sequence b of length 32768 - 997 b (its own cache of 32768 rows, rows drawn
              as for dec16k with sequence index b), H=128, bf16 queries; its last row is the fresh row
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

D, KL, KR = 576, 512, 64
SM_SCALE = float(np.float32(1.0 / np.sqrt(192.0)))


@dataclass(frozen=True)
class Workload:
    key: str
    number: int
    H: int
    T: int
    B: int = 1
    NS: int = 0
    S: int = 1
    pos0: int = 0
    mag_lo: float = 0.1
    mag_hi: float = 10.0
    heavy_frac: float = 0.0
    heavy_mult: float = 1.0
    q_f32: bool = False

    @property
    def seed(self) -> int:
        return 1000 + self.number


WORKLOADS = {
    "tiny": Workload("tiny", 1, H=16, T=256, mag_lo=1e-3, mag_hi=1e2, q_f32=True),
    "dec16k": Workload("dec16k", 2, H=128, T=16384),
    "dec262k": Workload("dec262k", 3, H=128, T=262144, heavy_frac=0.01, heavy_mult=50.0),
    "dsa": Workload("dsa", 4, H=128, T=131072, B=8, NS=2048),
    "prefill": Workload("prefill", 5, H=128, T=65536, S=1024, pos0=64512),
    # the absorb projections through an fmt=8 kv_b, at a decode step and at a prefill chunk
    "proj_dec": Workload("proj_dec", 6, H=128, T=0, S=1),
    "proj_prefill": Workload("proj_prefill", 7, H=128, T=0, S=1024),
    # the DSA lightning indexer that chooses the selection: 64 index heads of width 128 per query
    "indexer": Workload("indexer", 8, H=64, T=131072, B=8, NS=2048, mag_lo=10 ** -0.5, mag_hi=10 ** 0.5),
    # one decode step for a batch of sequences, each its own cache (ragged lengths, one fresh row each)
    "batch_dec": Workload("batch_dec", 9, H=128, T=32768, B=8),
    # decode over the mixed-precision cache: 448 e4m3 no-position values + row scale, 64 bf16 RoPE values
    "mixed_dec": Workload("mixed_dec", 10, H=128, T=65536),
}

DESCRIPTIONS = {
    "tiny": "tiny decode: 1 query, H=16, T=256, f32 queries",
    "dec16k": "single-sequence decode: H=128, T=16384, bf16 queries, 1 fresh row quantized per step",
    "dec262k": "long-context split-T decode: H=128, T=262144 (152 MB fp8 rows + scales), bf16 queries, "
               "1 fresh row quantized per step, 1% of rows x50",
    "dsa": "DSA sparse decode: B=8 sequences x T=131072 rows, NS=2048 selected rows each, H=128, bf16 queries",
    "prefill": "causal prefill chunk: S=1024 queries at 64512..65535 over T=65536 rows, H=128, bf16 queries",
    "proj_dec": "absorb projections at a decode step: 1 query x H=128 heads through an fmt=8 kv_b "
                "(128x256 rows x 512, 128x128-block scales): q_nope -> q_lat and context -> head output",
    "proj_prefill": "absorb projections for a prefill chunk: S=1024 queries x H=128 heads through an fmt=8 kv_b",
    "indexer": "DSA lightning indexer: B=8 queries, each scoring its own T=131072 e4m3 index keys (width 128) "
               "with 64 index heads, then top-2048",
    "mixed_dec": "mixed-precision cache decode: H=128 heads over T=65536 rows of 448 e4m3 no-position values "
                 "(per-row f32 scale) + 64 bf16 RoPE values; bf16 queries",
    "batch_dec": "batched decode: B=8 sequences, each its own cache of up to T=32768 rows (lengths 32768 - 997 b), "
                 "H=128, bf16 queries, one fresh row appended to each sequence per step",
}


def rng_for(w: Workload, stream: int = 0) -> np.random.Generator:
    return np.random.default_rng([w.seed, stream])


def latent_rows(rng: np.random.Generator, n: int, mag_lo: float, mag_hi: float,
                heavy_frac: float = 0.0, heavy_mult: float = 1.0) -> np.ndarray:
    """f32 [n][576]: N(0,1) per element times a per-row magnitude log-uniform in [mag_lo, mag_hi];
    a Bernoulli(heavy_frac) subset of rows is further multiplied by heavy_mult."""
    x = rng.standard_normal((n, D), dtype=np.float32)
    mag = 10.0 ** rng.uniform(np.log10(mag_lo), np.log10(mag_hi), size=n)
    if heavy_frac > 0.0:
        heavy = rng.random(n) < heavy_frac
        mag = np.where(heavy, mag * heavy_mult, mag)
    x *= mag.astype(np.float32)[:, None]
    return x


def normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round f32 -> bf16 (RNE, by torch) and return the bf16 values as f32 (exact)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float32).numpy()


def rows_for(w: Workload, seq: int = 0, start: int = 0, count: int | None = None) -> np.ndarray:
    """f32 latent rows [count][576] of sequence `seq`, rows start..start+count-1.  Rows are drawn in
    fixed blocks of 4096 so any sub-range reproduces the same values."""
    if count is None:
        count = w.T - start
    blk = 4096
    out = np.empty((count, D), dtype=np.float32)
    b0, b1 = start // blk, (start + count - 1) // blk if count > 0 else start // blk - 1
    for b in range(b0, b1 + 1):
        rng = np.random.default_rng([w.seed, 1, seq, b])
        n_b = min(blk, w.T - b * blk)
        rows = latent_rows(rng, n_b, w.mag_lo, w.mag_hi, w.heavy_frac, w.heavy_mult)
        if w.key == "tiny":
            for t in range(n_b):
                g = b * blk + t
                if g == 17:
                    rows[t, :] = 0.0
                    rows[t, 0] = -0.0
                elif g == 42:
                    rows[t, :] = (rng.standard_normal(D).astype(np.float64) * 1e-39).astype(np.float32)
        lo = max(start, b * blk)
        hi = min(start + count, b * blk + n_b)
        out[lo - start:hi - start] = rows[lo - b * blk:hi - b * blk]
    return out


def queries_for(w: Workload, n_query: int | None = None):
    """(q_lat, q_rope) as f32 arrays holding the query values ([nq][H][512], [nq][H][64]).
    For bf16 workloads the values are bf16-representable."""
    if n_query is None:
        n_query = w.S if w.key == "prefill" else w.B
    rng = rng_for(w, 2)
    q = normal_f32(rng, (n_query, w.H, D))
    if not w.q_f32:
        q = to_bf16_values(q)
    return np.ascontiguousarray(q[..., :KL]), np.ascontiguousarray(q[..., KL:])


def selection_for(w: Workload) -> np.ndarray:
    """idx [B][NS] int32: per sequence, NS unique indices drawn uniformly from [0, T), sorted."""
    rng = rng_for(w, 3)
    out = np.empty((w.B, w.NS), dtype=np.int32)
    for b in range(w.B):
        out[b] = np.sort(rng.choice(w.T, size=w.NS, replace=False)).astype(np.int32)
    return out


NOPE, VH, BLK = 128, 128, 128


def kvb_fmt8(H: int, seed: int = 2000):
    """Synthetic kv_b_proj in fmt=8 for H heads: (w8 [H*256][512] u8, w_scale [H*2][4] f32).

    The bytes are drawn directly as e4m3 codes (no encoding): random sign, exponent field uniform in
    6..11 and mantissa uniform in 0..7, so |code value| spans 0.5 .. 30 (never a NaN code, never
    zero); the 128x128 block scales are log-uniform in [1e-3, 1e-2] (weights of magnitude ~1e-3 ..
    0.3, the range of a trained up-projection)."""
    rng = np.random.default_rng([seed, H])
    n = H * (NOPE + VH) * KL
    sign = rng.integers(0, 2, n, dtype=np.uint8)
    expo = rng.integers(6, 12, n, dtype=np.uint8)
    mant = rng.integers(0, 8, n, dtype=np.uint8)
    w8 = ((sign << 7) | (expo << 3) | mant).astype(np.uint8).reshape(H * (NOPE + VH), KL)
    w_scale = (10.0 ** rng.uniform(-3.0, -2.0, (H * (NOPE + VH) // BLK, KL // BLK))).astype(np.float32)
    return w8, w_scale


def q_nope_for(w: Workload, n_query: int | None = None) -> np.ndarray:
    """The queries' no-position parts [nq][H][128] (f32 holding bf16-representable N(0,1) values unless
    the workload's queries are f32)."""
    if n_query is None:
        n_query = w.S if w.S > 1 else w.B
    rng = rng_for(w, 4)
    q = normal_f32(rng, (n_query, w.H, NOPE))
    return q if w.q_f32 else to_bf16_values(q)


def context_for(w: Workload) -> np.ndarray:
    """A normalised-context stand-in [S][H][512] f32 N(0,1) for the output projection."""
    return normal_f32(rng_for(w, 5), (max(w.S, w.B), w.H, KL))


IDX_D = 128  # index head / key width


def index_keys_for(w: Workload, seq: int = 0, start: int = 0, count: int | None = None) -> np.ndarray:
    """Index-key rows [count][128] f32 of sequence `seq`: N(0,1) times a per-row magnitude
    10^U(log10 mag_lo, log10 mag_hi), drawn in blocks of 4096 rows so any sub-range reproduces."""
    if count is None:
        count = w.T - start
    out = np.empty((count, IDX_D), dtype=np.float32)
    blk = 4096
    b0, b1 = start // blk, (start + count + blk - 1) // blk
    for bi in range(b0, b1):
        rng = np.random.default_rng([w.seed, 6, seq, bi])
        x = normal_f32(rng, (blk, IDX_D))
        mag = 10.0 ** rng.uniform(np.log10(w.mag_lo), np.log10(w.mag_hi), blk)
        x = (x * mag[:, None]).astype(np.float32)
        lo, hi = max(start, bi * blk), min(start + count, (bi + 1) * blk)
        out[lo - start:hi - start] = x[lo - bi * blk:hi - bi * blk]
    return out


def index_queries_for(w: Workload) -> np.ndarray:
    """Index queries [B][64][128]: bf16-representable N(0,1)."""
    return to_bf16_values(normal_f32(rng_for(w, 7), (w.B, w.H, IDX_D)))


def index_weights_for(w: Workload) -> np.ndarray:
    """Per-query head weights [B][64] f32: N(0,1)/8 (either sign)."""
    return (normal_f32(rng_for(w, 8), (w.B, w.H)) / np.float32(8.0)).astype(np.float32)


def batch_lengths(w: Workload) -> list[int]:
    """Ragged sequence lengths of the batched-decode workload."""
    return [w.T - 997 * b for b in range(w.B)]


MX_NOPE, MX_ROPE = 448, 64


def mixed_rows_for(w: Workload, start: int = 0, count: int | None = None):
    """(no-position values [count][448] f32, RoPE values [count][64] f32 holding bf16 values) of the
    mixed-cache workload, drawn in blocks of 4096 rows so any sub-range reproduces."""
    if count is None:
        count = w.T - start
    nope = np.empty((count, MX_NOPE), dtype=np.float32)
    rope = np.empty((count, MX_ROPE), dtype=np.float32)
    blk = 4096
    for bi in range(start // blk, (start + count + blk - 1) // blk):
        rng = np.random.default_rng([w.seed, 9, bi])
        x = normal_f32(rng, (blk, MX_NOPE))
        mag = 10.0 ** rng.uniform(np.log10(w.mag_lo), np.log10(w.mag_hi), blk)
        x = (x * mag[:, None]).astype(np.float32)
        r = to_bf16_values(normal_f32(rng, (blk, MX_ROPE)))
        lo, hi = max(start, bi * blk), min(start + count, (bi + 1) * blk)
        nope[lo - start:hi - start] = x[lo - bi * blk:hi - bi * blk]
        rope[lo - start:hi - start] = r[lo - bi * blk:hi - bi * blk]
    return nope, rope


def mixed_queries_for(w: Workload):
    """(q_nope [H][448], q_rope [H][64]): bf16-representable N(0,1)."""
    q = to_bf16_values(normal_f32(rng_for(w, 10), (w.H, MX_NOPE + MX_ROPE)))
    return np.ascontiguousarray(q[:, :MX_NOPE]), np.ascontiguousarray(q[:, MX_NOPE:])
