"""The seeded input recipe, checked against what the workloads state (CPU only).

Every parity test and the benchmark draw their inputs from `synth`; these tests check that the draws
have the shapes, value ranges and structure the workloads call for: the tiny config's all-zero and
subnormal-amax rows, the per-row log-uniform magnitudes, the long-context config's 1 % of rows x50,
bf16-representable queries, sorted unique selections, the ragged batch lengths, the fmt=8 weight codes,
and that any sub-range of rows reproduces the same values.  Statistical bounds are several standard
deviations wide; the draws are seeded, so each check is deterministic.
"""
import numpy as np
import torch

import synth

W = synth.WORKLOADS


def _rms(rows: np.ndarray) -> np.ndarray:
    return np.sqrt(np.mean(rows.astype(np.float64) ** 2, axis=1))


def _bf16_exact(x: np.ndarray) -> bool:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return bool(torch.equal(t.to(torch.bfloat16).to(torch.float32), t))


def test_tiny_rows_and_queries():
    w = W["tiny"]
    assert (w.H, w.T, w.q_f32) == (16, 256, True)
    x = synth.rows_for(w)
    assert x.shape == (256, synth.D) and x.dtype == np.float32
    # row 17: all zero, element 0 a negative zero
    assert np.all(x[17] == 0.0) and np.signbit(x[17, 0]) and not np.any(np.signbit(x[17, 1:]))
    # row 42: a non-zero row whose largest magnitude is below the smallest normal f32
    amax = np.max(np.abs(x[42]))
    assert 0.0 < amax < np.finfo(np.float32).tiny
    # the other rows: magnitudes 10^U(-3, 2) (a row's RMS is its magnitude within a few per cent)
    keep = np.ones(256, bool)
    keep[[17, 42]] = False
    r = _rms(x[keep])
    assert r.min() > 1e-3 * 0.85 and r.max() < 1e2 * 1.15
    assert r.min() < 1e-2 and r.max() > 10.0  # the draw spans the range
    q_lat, q_rope = synth.queries_for(w)
    assert q_lat.shape == (1, 16, synth.KL) and q_rope.shape == (1, 16, synth.KR)
    assert not _bf16_exact(q_lat)  # f32 queries, not rounded


def test_log_uniform_magnitudes():
    w = W["dec16k"]
    r = _rms(synth.rows_for(w, count=8192))
    assert r.min() > 0.1 * 0.85 and r.max() < 10.0 * 1.15
    lg = np.log10(r)
    # log10 of the magnitude is U(-1, 1): mean 0, standard deviation 2/sqrt(12)
    assert abs(lg.mean()) < 0.05
    assert abs(lg.std() - 2.0 / np.sqrt(12.0)) < 0.03


def test_long_context_heavy_rows():
    w = W["dec262k"]
    assert (w.heavy_frac, w.heavy_mult) == (0.01, 50.0)
    r = _rms(synth.rows_for(w, count=16384))
    # a heavy row's magnitude is 50 x 10^U(-1, 1); rows above 10 x 1.15 are heavy rows whose base
    # exceeds 10^-0.64, i.e. 82 % of the heavy rows: 16384 x 0.01 x 0.82 = 134 +- 12 expected
    n_big = int(np.sum(r > 11.5))
    assert 95 <= n_big <= 175, n_big
    assert r.max() < 500.0 * 1.15 and r.max() > 100.0
    # the light rows keep the single-sequence range
    assert r.min() > 0.1 * 0.85


def test_row_subranges_reproduce():
    w = W["dec16k"]
    full = synth.rows_for(w, count=8192)
    assert np.array_equal(synth.rows_for(w, start=4000, count=200), full[4000:4200])  # crosses a block
    assert np.array_equal(synth.rows_for(w, start=8191, count=1), full[8191:])
    assert np.array_equal(synth.rows_for(w, count=8192), full)  # seeded: the same draw twice
    wi = W["indexer"]
    k_full = synth.index_keys_for(wi, seq=3, count=8192)
    assert np.array_equal(synth.index_keys_for(wi, seq=3, start=4090, count=12), k_full[4090:4102])
    assert not np.array_equal(synth.index_keys_for(wi, seq=2, count=16), k_full[:16])  # per sequence
    wm = W["mixed_dec"]
    n_full, r_full = synth.mixed_rows_for(wm, count=8192)
    n_sub, r_sub = synth.mixed_rows_for(wm, start=4095, count=3)
    assert np.array_equal(n_sub, n_full[4095:4098]) and np.array_equal(r_sub, r_full[4095:4098])


def test_bf16_queries_and_rope_values():
    for key in ("dec16k", "dec262k", "prefill"):
        q_lat, q_rope = synth.queries_for(W[key], n_query=2)
        assert _bf16_exact(q_lat) and _bf16_exact(q_rope), key
    q_nope, q_rope = synth.mixed_queries_for(W["mixed_dec"])
    assert q_nope.shape == (128, 448) and q_rope.shape == (128, 64)
    assert _bf16_exact(q_nope) and _bf16_exact(q_rope)
    _, rope = synth.mixed_rows_for(W["mixed_dec"], count=64)
    assert _bf16_exact(rope)
    assert _bf16_exact(synth.index_queries_for(W["indexer"]))


def test_selection_lists():
    w = W["dsa"]
    idx = synth.selection_for(w)
    assert idx.shape == (8, 2048) and idx.dtype == np.int32
    assert np.all(idx >= 0) and np.all(idx < w.T)
    assert np.all(np.diff(idx, axis=1) > 0)  # sorted and unique
    # uniform in [0, T): each list's mean is T/2 within ~5 standard errors (T / sqrt(12 NS) each)
    assert np.all(np.abs(idx.mean(axis=1) - w.T / 2) < 5 * w.T / np.sqrt(12 * w.NS))
    assert not np.array_equal(idx[0], idx[1])


def test_workload_structure():
    p = W["prefill"]
    assert (p.S, p.pos0, p.T, p.H) == (1024, 64512, 65536, 128) and p.pos0 + p.S == p.T
    b = W["batch_dec"]
    lens = synth.batch_lengths(b)
    assert lens == [32768 - 997 * i for i in range(8)] and min(lens) >= 1 and max(lens) == b.T
    assert (W["dsa"].B, W["dsa"].NS, W["dsa"].T) == (8, 2048, 131072)
    assert (W["dec262k"].T, W["dec16k"].T) == (262144, 16384)
    wi = W["indexer"]
    wts = synth.index_weights_for(wi)
    assert wts.shape == (8, 64) and np.any(wts < 0) and np.any(wts > 0)
    assert 0.1 < wts.std() < 0.15  # N(0,1)/8
    assert abs(synth.SM_SCALE - 1.0 / np.sqrt(192.0)) < 1e-7


def test_fmt8_weight_codes():
    w8, w_scale = synth.kvb_fmt8(4)
    assert w8.shape == (4 * 256, 512) and w8.dtype == np.uint8
    assert w_scale.shape == (4 * 2, 4) and w_scale.dtype == np.float32
    expo = (w8 >> 3) & 15
    assert expo.min() == 6 and expo.max() == 11  # never zero, subnormal or the NaN codes 0x7F / 0xFF
    assert np.all((w8 & 0x7F) != 0x7F)
    assert w_scale.min() >= 1e-3 and w_scale.max() <= 1e-2
    assert np.any(w8 >> 7) and np.any((w8 >> 7) == 0)  # both signs
