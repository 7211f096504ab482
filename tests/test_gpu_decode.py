"""GPU split-T decode (partial kernel + log-sum-exp merge) vs the oracle.

The cache rows come from the oracle's quantizer (never from the GPU); the step's fresh row (row
T-1) is quantized by the GPU in-step, as in the benchmark, and checked bit-exact against the
oracle's bytes first.  Full outputs for the tiny, 16k and 262k workloads (262k: every head, each on
its own scale, in the benchmark's launch configuration).  Edge cases: T = 1, ragged T, H not a
multiple of the head group, P = 1 (unsplit) vs automatic vs forced partitions, f32 and bf16 queries,
row scales spanning 1e-3 .. 1e2 inside one partition in random / ascending / descending order.
"""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_cache, parity, parity_per_head

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _qtensor(v: np.ndarray, f32: bool):
    t = torch.from_numpy(np.ascontiguousarray(v)).to(DEV)
    return t if f32 else t.to(torch.bfloat16)


def _decode(lib, q_lat, q_rope, kv8, sc, T, P_req=0, sm=synth.SM_SCALE):
    H = q_lat.shape[0]
    ws = torch.empty(lib.mla_decode8_workspace_bytes(H, T, P_req) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty((H, 512), dtype=torch.float32, device=DEV)
    lib.mla_absorb_decode8(q_lat, q_rope, kv8, sc, T, sm, ws, out, P_req=P_req)
    torch.cuda.synchronize()
    return out.cpu().numpy()


class Step:
    """A decode workload: oracle cache for rows 0..T-1, the fresh f32 row T-1 quantized on the GPU."""

    def __init__(self, lib, oracle, key):
        w = synth.WORKLOADS[key]
        self.w = w
        rows = synth.rows_for(w)
        self.q_o, self.s_o = oracle_cache(oracle, rows)
        self.kv8 = torch.from_numpy(self.q_o).to(DEV)
        self.sc = torch.from_numpy(self.s_o).to(DEV)
        self.kv8[-1].fill_(0)
        self.sc[-1:].fill_(0)
        fresh = torch.from_numpy(rows[-1:].copy()).to(DEV)
        lib.kv8_quant_rows(fresh, self.kv8[-1:], self.sc[-1:])
        torch.cuda.synchronize()
        assert np.array_equal(self.kv8[-1].cpu().numpy(), self.q_o[-1])
        assert self.sc[-1].item() == self.s_o[-1] or (np.isnan(self.s_o[-1]) and np.isnan(self.sc[-1].item()))
        ql, qr = synth.queries_for(w, 1)
        self.ql, self.qr = ql[0], qr[0]
        self.q_lat = _qtensor(self.ql, w.q_f32)
        self.q_rope = _qtensor(self.qr, w.q_f32)


_steps = {}


def step(lib, oracle, key):
    if key not in _steps:
        _steps.clear()  # hold one large workload at a time
        _steps[key] = Step(lib, oracle, key)
    return _steps[key]


@pytest.mark.parametrize("key", ["tiny", "dec16k"])
def test_decode_full_output(lib, oracle, key):
    s = step(lib, oracle, key)
    got = _decode(lib, s.q_lat, s.q_rope, s.kv8, s.sc, s.w.T)
    ref = oracle.attn_decode(s.ql, s.qr, s.q_o, s.s_o, synth.SM_SCALE)
    parity(got, ref, key)


def test_decode_262k_every_head(lib, oracle):
    """The headline workload in the launch configuration the benchmark times (automatic partitions):
    all 128 heads against the oracle, each head on its own scale."""
    s = step(lib, oracle, "dec262k")
    got = _decode(lib, s.q_lat, s.q_rope, s.kv8, s.sc, s.w.T)
    ref = oracle.attn_decode(s.ql, s.qr, s.q_o, s.s_o, synth.SM_SCALE)
    parity_per_head(got, ref, "dec262k every head")


@pytest.mark.parametrize("P_req", [1, 7, 0, 200])
def test_decode_partition_counts_agree(lib, oracle, P_req):
    s = step(lib, oracle, "dec16k")
    got = _decode(lib, s.q_lat, s.q_rope, s.kv8, s.sc, s.w.T, P_req=P_req)
    heads = list(range(0, 128, 9))
    ref = oracle.attn_decode(s.ql[heads], s.qr[heads], s.q_o, s.s_o, synth.SM_SCALE)
    parity(got[heads], ref, f"P={P_req}")


def test_partial_then_merge_equals_combined(lib, oracle):
    s = step(lib, oracle, "dec16k")
    T, H = s.w.T, 128
    P = lib.mla_decode8_partitions(H, T)
    ws = torch.empty(lib.mla_decode8_workspace_bytes(H, T) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty((H, 512), dtype=torch.float32, device=DEV)
    lib.mla_decode8_partial(s.q_lat, s.q_rope, s.kv8, s.sc, T, synth.SM_SCALE, ws)
    lib.mla_lse_merge8(ws, 1, P, H, out)
    torch.cuda.synchronize()
    combined = _decode(lib, s.q_lat, s.q_rope, s.kv8, s.sc, T)
    assert np.array_equal(out.cpu().numpy(), combined)


@pytest.mark.parametrize("P", [1, 5, 16, 17, 32, 33, 64, 65, 96, 97, 128, 129, 300])
def test_merge_alone_every_partition_class(lib, oracle, P):
    """The merge kernel fed the oracle's own split-T partials (cl, m, z in double; m in natural-log
    units, so m * log2(e) in the library's layout) for B = 3 queries: every kernel size class of P,
    and P > T, where some partitions are empty (m = -inf, z = 0)."""
    T, H, B = 257, 8, 3
    rng = np.random.default_rng(1000 + P)
    rows = synth.latent_rows(rng, T, 0.1, 10.0)
    q_o, s_o = oracle.quant_rows(rows)
    cl = np.zeros((B, P, H, 512), np.float32)
    m = np.zeros((B, P, H), np.float32)
    z = np.zeros((B, P, H), np.float32)
    ref = np.zeros((B, H, 512), np.float32)
    for b in range(B):
        q = synth.normal_f32(rng, (H, 576)) * np.float32(1 + 3 * b)
        ref[b], cl_b, m_b, z_b = oracle.attn_decode_split(q[:, :512], q[:, 512:], q_o, s_o, synth.SM_SCALE, P)
        cl[b], m[b], z[b] = cl_b, m_b * np.log2(np.e), z_b
    if P > T:
        assert np.isinf(m).any(), "some partitions are empty"
    ws = torch.from_numpy(np.concatenate([cl.ravel(), m.ravel(), z.ravel()])).to(DEV)
    out = torch.empty((B, H, 512), dtype=torch.float32, device=DEV)
    lib.mla_lse_merge8(ws, B, P, H, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    # inputs rounded to f32 (m to ~1e-5 log2 units): far inside the attention tolerance
    err = np.abs(got - ref).max() / np.abs(ref).max()
    assert err <= 1e-4, f"P={P}: max error {err:.2e} of max |out|"


def _random_case(oracle, T, H, seed, mag=(0.1, 10.0)):
    rng = np.random.default_rng(seed)
    rows = synth.latent_rows(rng, T, *mag)
    q_o, s_o = oracle.quant_rows(rows)
    q = synth.normal_f32(rng, (H, 576))
    return q_o, s_o, q


@pytest.mark.parametrize("T,H,f32", [(1, 16, True), (1, 128, False), (2, 5, True), (129, 33, False),
                                     (1000, 1, True), (4097, 128, False), (777, 96, True), (777, 96, False),
                                     (300, 65, False), (2, 1, False)])
def test_decode_ragged_shapes(lib, oracle, T, H, f32):
    q_o, s_o, q = _random_case(oracle, T, H, seed=T * 131 + H)
    if not f32:
        q = synth.to_bf16_values(q)
    kv8 = torch.from_numpy(q_o).to(DEV)
    sc = torch.from_numpy(s_o).to(DEV)
    ql, qr = np.ascontiguousarray(q[:, :512]), np.ascontiguousarray(q[:, 512:])
    got = _decode(lib, _qtensor(ql, f32), _qtensor(qr, f32), kv8, sc, T)
    ref = oracle.attn_decode(ql, qr, q_o, s_o, synth.SM_SCALE)
    parity(got, ref, f"T={T} H={H}")
    if T == 1:
        # one row: the context is that row's dequantized latent, exactly up to f32 rounding
        np.testing.assert_allclose(got, np.broadcast_to(ref[0], got.shape), rtol=1e-6, atol=0)


def test_decode_peaky_and_tiny_magnitudes(lib, oracle):
    """Rows spanning 1e-3..1e2 with a few x1000 rows: a near one-hot softmax, and a subnormal row."""
    rng = np.random.default_rng(77)
    T, H = 3000, 64
    rows = synth.latent_rows(rng, T, 1e-3, 1e2, heavy_frac=0.002, heavy_mult=1000.0)
    rows[17] = 0.0
    rows[42] = (rng.standard_normal(576) * 1e-39).astype(np.float32)
    q_o, s_o = oracle.quant_rows(rows)
    q = synth.to_bf16_values(synth.normal_f32(rng, (H, 576)))
    ql, qr = np.ascontiguousarray(q[:, :512]), np.ascontiguousarray(q[:, 512:])
    got = _decode(lib, _qtensor(ql, False), _qtensor(qr, False), torch.from_numpy(q_o).to(DEV),
                  torch.from_numpy(s_o).to(DEV), T)
    parity(got, oracle.attn_decode(ql, qr, q_o, s_o, synth.SM_SCALE), "peaky")


def test_decode_query_magnitudes(lib, oracle):
    """bf16 query heads whose magnitudes span the bf16 range (the tensor-core path scales each head by a
    power of two before splitting it into e4m3 pieces), an all-zero head and a one-element head."""
    rng = np.random.default_rng(91)
    T, H = 900, 24
    rows = synth.latent_rows(rng, T, 0.1, 10.0)
    q_o, s_o = oracle.quant_rows(rows)
    q = synth.normal_f32(rng, (H, 576)).astype(np.float64)
    # up to 2^120: larger heads would give scores beyond the f32 range (|s| > 3e38 log2 units)
    exps = np.array([-130, -126, -100, -60, -20, -5, 0, 3, 10, 20, 40, 60, 80, 100, 120, 110,
                     -128, -110, -90, -40, 30, 50, 0, 0], dtype=np.float64)
    q *= np.exp2(exps)[:, None]
    q[22] = 0.0                       # all-zero head: uniform softmax
    q[23] = 0.0
    q[23, 511] = 3.0                  # one latent element
    q = synth.to_bf16_values(q.astype(np.float32))
    assert np.all(np.isfinite(q))
    ql, qr = np.ascontiguousarray(q[:, :512]), np.ascontiguousarray(q[:, 512:])
    got = _decode(lib, _qtensor(ql, False), _qtensor(qr, False), torch.from_numpy(q_o).to(DEV),
                  torch.from_numpy(s_o).to(DEV), T)
    ref = oracle.attn_decode(ql, qr, q_o, s_o, synth.SM_SCALE)
    assert np.all(np.isfinite(got))
    for h in range(H):  # each head against its own scale
        parity(got[h], ref[h], f"head {h} (2^{int(exps[h])})")


@pytest.mark.parametrize("order", ["random", "ascending", "descending"])
@pytest.mark.parametrize("P_req", [1, 0])
def test_decode_row_scales_span_one_partition(lib, oracle, order, P_req):
    """bf16 queries over rows whose scales (amax/448) span 1e-3 .. 1e2 inside one partition: the running
    max keeps moving (ascending order rescales on most tiles), a few rows dominate, most weights are
    tiny.  Every head checked on its own scale."""
    rng = np.random.default_rng(4242)
    T, H = 3001, 128
    rows = synth.latent_rows(rng, T, 0.15, 1.5e4)
    amax = np.abs(rows).max(axis=1)
    if order != "random":
        rows = rows[np.argsort(amax if order == "ascending" else -amax, kind="stable")]
    q_o, s_o = oracle.quant_rows(rows)
    assert s_o.min() < 2e-3 and s_o.max() > 50.0  # the span the test is about
    q = synth.to_bf16_values(synth.normal_f32(rng, (H, 576)))
    ql, qr = np.ascontiguousarray(q[:, :512]), np.ascontiguousarray(q[:, 512:])
    kv8, sc = torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)
    got = _decode(lib, _qtensor(ql, False), _qtensor(qr, False), kv8, sc, T, P_req=P_req)
    ref = oracle.attn_decode(ql, qr, q_o, s_o, synth.SM_SCALE)
    parity_per_head(got, ref, f"row scales 1e-3..1e2, {order} order, P_req={P_req}")


def test_decode_repeated_calls_identical(lib, oracle):
    """The kernels are deterministic (fixed MMA and reduction orders, order-free atomics), so repeated
    calls must give bit-identical outputs: a race between the pipeline's stages shows up as a mismatch.
    Few partitions (long CTAs, many tiles per CTA) give races the most chances."""
    s = step(lib, oracle, "dec16k")
    for P_req in (1, 2, 3):
        first = _decode(lib, s.q_lat, s.q_rope, s.kv8, s.sc, s.w.T, P_req=P_req)
        for _ in range(12):
            again = _decode(lib, s.q_lat, s.q_rope, s.kv8, s.sc, s.w.T, P_req=P_req)
            assert np.array_equal(again, first), f"P={P_req}: outputs differ between identical calls"
        heads = list(range(0, 128, 9))
        parity(first[heads], oracle.attn_decode(s.ql[heads], s.qr[heads], s.q_o, s.s_o, synth.SM_SCALE), f"P={P_req}")
