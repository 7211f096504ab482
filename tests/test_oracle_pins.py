"""Pins for the oracle: checks against things other than the oracle itself.

Each test fixes the oracle to a closed form, an invariant, a hand-derived value (tests/golden/,
each file citing its source), brute force, or an independent library routine (torch's
float8_e4m3fn conversion).  Chosen so that a dropped term, a wrong sign or index, or a transposed
operand in the oracle fails at least one of them.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
D, KL, KR = 576, 512, 64


def f32_from_bits(h):
    return np.array([h], dtype=np.uint32).view(np.float32)[0]


def torch_e4m3(y: np.ndarray) -> np.ndarray:
    """torch's f32 -> float8_e4m3fn conversion (round to nearest even), as bytes."""
    return torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


# ------------------------------------------------------------------------------------------------
# e4m3 decode table
# ------------------------------------------------------------------------------------------------
def test_decode_table_matches_torch_float8(oracle):
    tab = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.all(np.isnan(tab[nan]))
    assert np.array_equal(tab[~nan], ref[~nan])
    # signed zero
    assert math.copysign(1.0, tab[0x80]) == -1.0 and math.copysign(1.0, tab[0x00]) == 1.0


def test_decode_closed_form_points(oracle):
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x08) == 2.0 ** -6
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9
    assert oracle.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert oracle.e4m3_decode(0x38) == 1.0
    assert oracle.e4m3_decode(0xFE) == -448.0
    # the table is strictly increasing over 0x00..0x7E
    tab = oracle.e4m3_table()
    assert np.all(np.diff(tab[:0x7F]) > 0)


# ------------------------------------------------------------------------------------------------
# e4m3 encode
# ------------------------------------------------------------------------------------------------
def _golden_encode_cases():
    cases = []
    with open(os.path.join(GOLDEN, "e4m3_encode_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            bits, code, *_ = line.split()
            cases.append((int(bits, 16), int(code, 16), line))
    return cases


def test_encode_golden_cases(oracle):
    cases = _golden_encode_cases()
    assert len(cases) >= 25
    for bits, code, line in cases:
        y = f32_from_bits(bits)
        assert oracle.e4m3_encode(y) == code, line
        assert oracle.e4m3_encode_scan(y) == code, line


def _interesting_values(oracle, rng):
    tab = oracle.e4m3_table()[:0x7F]
    mids = (tab[:-1] + tab[1:]) / 2
    pts = np.concatenate([tab, mids, [464.0, 447.99, 0.0]]).astype(np.float32)
    bits = pts.view(np.uint32).astype(np.int64)
    near = (bits[:, None] + np.arange(-3, 4)[None, :]).reshape(-1)
    near = near[(near >= 0) & (near < 0x7F800000)].astype(np.uint32).view(np.float32)
    rand = (rng.standard_normal(200_000) * 10.0 ** rng.uniform(-6, 3, 200_000)).astype(np.float32)
    vals = np.concatenate([near, -near, rand])
    return vals[np.abs(vals) <= 464.0]


def test_encode_matches_torch_rne_in_range(oracle):
    """Inside |y| <= 464, where no saturation or NaN rule applies, the encoder is plain RNE and
    must equal torch's conversion (an independent implementation)."""
    rng = np.random.default_rng(7)
    vals = _interesting_values(oracle, rng)
    got = oracle.encode_array(vals)
    ref = torch_e4m3(vals)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:10]]


def test_encode_bisection_equals_scan(oracle):
    rng = np.random.default_rng(8)
    vals = _interesting_values(oracle, rng)[::37]
    vals = np.concatenate([vals, [np.inf, -np.inf, np.nan, 1e30, -1e30]]).astype(np.float32)
    for v in vals:
        assert oracle.e4m3_encode(v) == oracle.e4m3_encode_scan(v), v


def test_encode_saturation_and_nan(oracle):
    for v in [448.0, 449.0, 464.0, 465.0, 480.0, 1e6, 3.4e38, np.inf]:
        assert oracle.e4m3_encode(v) == 0x7E
        assert oracle.e4m3_encode(-v) == 0xFE
    for bits in [0x7FC00000, 0xFFC00000, 0x7F800001, 0xFFFFFFFF, 0x7FFFFFFF]:
        assert oracle.e4m3_encode(f32_from_bits(bits)) == 0x00


def test_encode_roundtrip_all_codes(oracle):
    """encode(decode(b)) == b for the 254 non-NaN codes (page: exhaustive e4m3 roundtrip)."""
    tab = oracle.e4m3_table()
    for b in range(256):
        if b in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(np.float32(tab[b])) == b, hex(b)


def test_encode_change_points_structure(oracle):
    """The change-point list the exhaustive GPU test compares against: 126 steps per sign, codes
    rising by exactly one at each, every step agreeing with torch at p and p-1."""
    cp = oracle.encode_change_points()
    assert len(cp) == 126 + 2 + 126 + 1
    assert np.all(np.diff(cp.astype(np.int64)) > 0)
    pos = cp[:126]
    neg = cp[128:254]
    assert list(cp[126:128]) == [0x7F800001, 0x80000000] and cp[-1] == 0xFF800001
    for group, sign in ((pos, 0), (neg, 0x80)):
        for k, p in enumerate(group):
            a = oracle.e4m3_encode(f32_from_bits(int(p)))
            b = oracle.e4m3_encode(f32_from_bits(int(p) - 1))
            assert a == sign | (k + 1) and b == sign | k
            ya = np.array([f32_from_bits(int(p)), f32_from_bits(int(p) - 1)], dtype=np.float32)
            if np.all(np.abs(ya) <= 464.0):
                assert list(torch_e4m3(ya)) == [a, b]


# ------------------------------------------------------------------------------------------------
# row quantizer
# ------------------------------------------------------------------------------------------------
def _golden_quant_cases():
    out = []
    with open(os.path.join(GOLDEN, "quant_rows_cases.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            elems, scale, codes = [p.strip() for p in line.split("|")]
            x = np.zeros(D, dtype=np.float32)
            e = [np.float32(v) for v in elems.split()]
            x[:len(e)] = e
            c = np.zeros(D, dtype=np.uint8)
            cc = [int(v, 16) for v in codes.split()]
            c[:len(cc)] = cc
            out.append((x, int(scale, 16), c, line))
    return out


def test_quant_golden_rows(oracle):
    for x, scale_bits, codes, line in _golden_quant_cases():
        q, s = oracle.quant_rows(x[None, :])
        assert s.view(np.uint32)[0] == scale_bits, line
        assert np.array_equal(q[0], codes), line


def test_quant_matches_torch_on_normal_rows(oracle):
    """scale = amax/448 and y = x*(448/amax) in f32, then RNE: torch does the same steps with its
    own f32 ops and its own fp8 conversion (|y| <= 448 here, so no saturation rule applies)."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((300, D)) * 10.0 ** rng.uniform(-20, 20, (300, 1))).astype(np.float32)
    q, s = oracle.quant_rows(x)
    xt = torch.from_numpy(x)
    amax = xt.abs().amax(dim=1)
    st = amax / 448.0
    inv = torch.tensor(448.0, dtype=torch.float32) / amax
    y = xt * inv[:, None]
    qt = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(s.view(np.uint32), st.numpy().view(np.uint32))
    assert np.array_equal(q, qt)


def test_quant_amax_element_and_zero_row(oracle):
    rng = np.random.default_rng(12)
    x = rng.standard_normal((50, D)).astype(np.float32)
    q, s = oracle.quant_rows(x)
    i = np.abs(x).argmax(axis=1)
    for r in range(50):
        assert q[r, i[r]] == (0xFE if x[r, i[r]] < 0 else 0x7E)
    z = np.zeros((1, D), dtype=np.float32)
    z[0, 5] = -0.0
    qz, sz = oracle.quant_rows(z)
    assert sz[0] == 0.0 and qz[0, 5] == 0x80 and np.count_nonzero(qz) == 1


def test_quant_scale_invariance_and_subnormal_guard(oracle):
    """Scaling a row by 2^k changes its scale by 2^k and not its bytes; a subnormal-amax row (where
    448/amax overflows) gives the bytes of the same row scaled into the normal range."""
    rng = np.random.default_rng(13)
    base = rng.standard_normal((20, D)).astype(np.float32)
    q0, s0 = oracle.quant_rows(base)
    for k in (-40, -5, 7, 60):
        qk, sk = oracle.quant_rows((base.astype(np.float64) * 2.0 ** k).astype(np.float32))
        assert np.array_equal(qk, q0)
        assert np.array_equal(sk, (s0.astype(np.float64) * 2.0 ** k).astype(np.float32))
    # subnormal amax: build rows whose values are exactly base * 2^-140 (representable only with
    # fewer bits, so compare against the same reduced-precision values scaled by 2^64).
    sub = (base.astype(np.float64) * 2.0 ** -140).astype(np.float32)
    assert np.all(np.abs(sub).max(axis=1) < 448.0 / np.finfo(np.float32).max)
    qs, ss = oracle.quant_rows(sub)
    up = (sub.astype(np.float64) * 2.0 ** 64).astype(np.float32)
    qu, su = oracle.quant_rows(up)
    assert np.array_equal(qs, qu)
    assert np.all(ss >= 0.0) and np.all(np.isfinite(ss))


def test_quant_error_bound(oracle):
    """|dequant - x| <= half an e4m3 step of y, times the scale (plus the f32 rounding of y)."""
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((200, D)) * 10.0 ** rng.uniform(-3, 3, (200, 1))).astype(np.float32)
    q, s = oracle.quant_rows(x)
    deq = oracle.dequant_rows(q, s)
    y = np.abs(x.astype(np.float64)) * (448.0 / np.abs(x).max(axis=1, keepdims=True).astype(np.float64))
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half_step = 0.5 * 2.0 ** (e - 3)
    bound = (half_step * (1 + 1e-6) + 448.0 * 2.0 ** -23) * s[:, None].astype(np.float64) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)


# ------------------------------------------------------------------------------------------------
# attention (decode / split / select / prefill)
# ------------------------------------------------------------------------------------------------
def _rand_cache(rng, T, mag=1.0):
    codes = rng.integers(0, 256, size=(T, D), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    scale = (rng.uniform(0.5, 2.0, T) * mag).astype(np.float32)
    return codes, scale


def test_attn_single_row_returns_dequantized_row(oracle):
    rng = np.random.default_rng(20)
    kv, sc = _rand_cache(rng, 1)
    ql = rng.standard_normal((3, KL)).astype(np.float32)
    qr = rng.standard_normal((3, KR)).astype(np.float32)
    out = oracle.attn_decode(ql, qr, kv, sc, 0.07)
    tab = oracle.e4m3_table()
    want = (tab[kv[0, :KL]] * np.float64(sc[0])).astype(np.float32)
    for h in range(3):
        assert np.array_equal(out[h], want)


def test_attn_zero_query_is_mean_of_rows(oracle):
    rng = np.random.default_rng(21)
    kv, sc = _rand_cache(rng, 37)
    out = oracle.attn_decode(np.zeros((2, KL)), np.zeros((2, KR)), kv, sc, 0.3)
    tab = oracle.e4m3_table()
    deq = tab[kv[:, :KL]] * sc.astype(np.float64)[:, None]
    np.testing.assert_allclose(out[0], deq.mean(axis=0), rtol=1e-6, atol=1e-30)


def _two_row_case(which):
    """Two rows that differ only in one coordinate of Lc (index 511) or Rc (index 63)."""
    kv = np.full((2, D), 0x38, dtype=np.uint8)  # every element 1.0
    kv[1, :KL] = 0x40  # row 1's latent is 2.0 everywhere
    sc = np.array([1.0, 1.0], dtype=np.float32)
    ql = np.zeros((1, KL), dtype=np.float32)
    qr = np.zeros((1, KR), dtype=np.float32)
    if which == "rope":
        kv[0, KL + 63] = 0x38   # 1.0
        kv[1, KL + 63] = 0xC0   # -2.0
        qr[0, 63] = 1.5
        s = np.array([1.5 * 1.0, 1.5 * -2.0])
    else:
        # Lc row 1 is 2.0 at index 511 as well; q_lat picks index 511 only
        ql[0, 511] = -0.75
        s = np.array([-0.75 * 1.0, -0.75 * 2.0])
    return kv, sc, ql, qr, s


@pytest.mark.parametrize("which", ["rope", "latent"])
def test_attn_two_rows_closed_form(oracle, which):
    kv, sc, ql, qr, s = _two_row_case(which)
    sm = 0.625
    out = oracle.attn_decode(ql, qr, kv, sc, sm)
    w1 = 1.0 / (1.0 + math.exp(sm * (s[0] - s[1])))
    w0 = 1.0 - w1
    want = w0 * 1.0 + w1 * 2.0
    np.testing.assert_allclose(out[0], np.full(KL, want), rtol=1e-7)


def test_attn_row_scale_enters_score_and_value(oracle):
    """Doubling a row's scale doubles its score and its value (s_t multiplies both)."""
    kv = np.full((2, D), 0x38, dtype=np.uint8)
    sc = np.array([1.0, 2.0], dtype=np.float32)
    ql = np.zeros((1, KL), dtype=np.float32)
    ql[0, 0] = 1.0
    sm = 0.5
    out = oracle.attn_decode(ql, np.zeros((1, KR)), kv, sc, sm)
    s0, s1 = sm * 1.0 * 1.0, sm * 2.0 * 1.0
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    want = (1 - w1) * 1.0 + w1 * 2.0
    np.testing.assert_allclose(out[0], np.full(KL, want), rtol=1e-7)


def test_attn_sharp_softmax_selects_argmax_row(oracle):
    rng = np.random.default_rng(22)
    kv, sc = _rand_cache(rng, 64)
    ql = rng.standard_normal((4, KL)).astype(np.float32)
    qr = rng.standard_normal((4, KR)).astype(np.float32)
    tab = oracle.e4m3_table()
    deq = tab[kv] * sc.astype(np.float64)[:, None]
    scores = ql.astype(np.float64) @ deq[:, :KL].T + qr.astype(np.float64) @ deq[:, KL:].T
    out = oracle.attn_decode(ql, qr, kv, sc, 1e4)
    for h in range(4):
        top = np.argsort(scores[h])[-2:]
        assert (scores[h, top[1]] - scores[h, top[0]]) * 1e4 > 50  # a clear winner
        np.testing.assert_allclose(out[h], deq[top[1], :KL], rtol=1e-6)


def test_attn_permutation_invariance(oracle):
    rng = np.random.default_rng(23)
    kv, sc = _rand_cache(rng, 200)
    ql = rng.standard_normal((3, KL)).astype(np.float32)
    qr = rng.standard_normal((3, KR)).astype(np.float32)
    perm = rng.permutation(200)
    a = oracle.attn_decode(ql, qr, kv, sc, 0.05)
    b = oracle.attn_decode(ql, qr, kv[perm], sc[perm], 0.05)
    np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-12)


@pytest.mark.parametrize("P", [1, 2, 7, 64, 300])
def test_split_merge_equals_unsplit(oracle, P):
    rng = np.random.default_rng(24)
    T = 300
    kv, sc = _rand_cache(rng, T)
    ql = rng.standard_normal((5, KL)).astype(np.float32)
    qr = rng.standard_normal((5, KR)).astype(np.float32)
    ref = oracle.attn_decode(ql, qr, kv, sc, 0.08)
    out, cl, m, z = oracle.attn_decode_split(ql, qr, kv, sc, 0.08, P)
    np.testing.assert_allclose(out, ref, rtol=2e-6, atol=1e-30)
    # each partial normalised on its own equals the dense result over its rows
    for p in sorted({0, P // 2, P - 1}):
        t0, t1 = T * p // P, T * (p + 1) // P
        if t1 > t0:
            np.testing.assert_allclose(cl[p] / z[p][:, None], oracle.attn_decode(ql, qr, kv[t0:t1], sc[t0:t1], 0.08),
                                       rtol=2e-6, atol=1e-30)


def test_split_with_empty_partitions(oracle):
    rng = np.random.default_rng(25)
    kv, sc = _rand_cache(rng, 3)
    ql = rng.standard_normal((2, KL)).astype(np.float32)
    qr = rng.standard_normal((2, KR)).astype(np.float32)
    out, cl, m, z = oracle.attn_decode_split(ql, qr, kv, sc, 0.1, 8)  # 5 of 8 partitions empty
    assert np.sum(np.isinf(m)) == 2 * 5 and np.all(z[np.isinf(m)] == 0)
    np.testing.assert_allclose(out, oracle.attn_decode(ql, qr, kv, sc, 0.1), rtol=2e-6)


def test_select_full_index_equals_dense_and_subset_equals_gathered(oracle):
    rng = np.random.default_rng(26)
    B, T, H = 3, 120, 2
    kv, sc = _rand_cache(rng, B * T)
    ql = rng.standard_normal((B, H, KL)).astype(np.float32)
    qr = rng.standard_normal((B, H, KR)).astype(np.float32)
    full = np.tile(np.arange(T, dtype=np.int32), (B, 1))
    out, bad = oracle.attn_select(ql, qr, kv, sc, T, T, full, 0.07)
    assert bad == 0
    for b in range(B):
        np.testing.assert_allclose(out[b], oracle.attn_decode(ql[b], qr[b], kv[b * T:(b + 1) * T],
                                                              sc[b * T:(b + 1) * T], 0.07), rtol=1e-6)
    sel = np.stack([np.sort(rng.choice(T, 17, replace=False)) for _ in range(B)]).astype(np.int32)
    out, _ = oracle.attn_select(ql, qr, kv, sc, T, T, sel, 0.07)
    for b in range(B):
        rows = b * T + sel[b]
        np.testing.assert_allclose(out[b], oracle.attn_decode(ql[b], qr[b], kv[rows], sc[rows], 0.07), rtol=1e-6)
    one = sel[:, :1].copy()
    out, _ = oracle.attn_select(ql, qr, kv, sc, T, T, one, 0.07)
    tab = oracle.e4m3_table()
    for b in range(B):
        r = b * T + one[b, 0]
        np.testing.assert_array_equal(out[b, 0], (tab[kv[r, :KL]] * np.float64(sc[r])).astype(np.float32))


def test_select_skips_out_of_range(oracle):
    rng = np.random.default_rng(27)
    T = 50
    kv, sc = _rand_cache(rng, 2 * T)
    ql = rng.standard_normal((2, 1, KL)).astype(np.float32)
    qr = rng.standard_normal((2, 1, KR)).astype(np.float32)
    idx = np.array([[3, 60, 7, -1], [0, 1, 2, 49]], dtype=np.int32)
    out, bad = oracle.attn_select(ql, qr, kv, sc, T, T, idx, 0.1)
    assert bad == 2
    np.testing.assert_allclose(out[0], oracle.attn_decode(ql[0], qr[0], kv[[3, 7]], sc[[3, 7]], 0.1), rtol=1e-6)


def test_prefill_query_equals_decode_over_prefix(oracle):
    rng = np.random.default_rng(28)
    T, pos0, S, H = 90, 80, 10, 2
    kv, sc = _rand_cache(rng, T)
    ql = rng.standard_normal((S, H, KL)).astype(np.float32)
    qr = rng.standard_normal((S, H, KR)).astype(np.float32)
    pos = pos0 + np.arange(S)
    out = oracle.attn_prefill(ql, qr, pos, kv, sc, 0.09)
    for i in range(S):
        ref = oracle.attn_decode(ql[i], qr[i], kv[:pos[i] + 1], sc[:pos[i] + 1], 0.09)
        np.testing.assert_array_equal(out[i], ref)
    # the first query cannot see the second query's row
    kv2 = kv.copy()
    kv2[pos0 + 1:] = 0x7E
    out2 = oracle.attn_prefill(ql[:1], qr[:1], pos[:1], kv2, sc, 0.09)
    np.testing.assert_array_equal(out2[0], out[0])


# ------------------------------------------------------------------------------------------------
# absorb projections through an fmt=8 kv_b (e4m3 bytes, one f32 scale per 128x128 block)
# ------------------------------------------------------------------------------------------------
def _kvb_dense(w8, w_scale):
    """Dequantized kv_b in double, decoded by torch's float8_e4m3fn (independent of the oracle's table)."""
    vals = torch.from_numpy(np.ascontiguousarray(w8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return vals * np.repeat(np.repeat(w_scale.astype(np.float64), 128, axis=0), 128, axis=1)


def test_q_absorb_identity_weights_copy_the_query(oracle):
    H = 3
    w8 = np.zeros((H * 256, KL), np.uint8)
    for h in range(H):
        w8[h * 256 + np.arange(128), np.arange(128)] = 0x38  # 1.0
    sc = np.ones((H * 2, 4), np.float32)
    q = np.random.default_rng(1).standard_normal((5, H, 128)).astype(np.float32)
    got = oracle.q_absorb(q, w8, sc)
    assert np.array_equal(got[..., :128], q) and not got[..., 128:].any()


@pytest.mark.parametrize("h,j,c", [(0, 0, 0), (1, 127, 511), (2, 5, 300), (2, 64, 129)])
def test_q_absorb_single_weight_lands_at_its_index(oracle, h, j, c):
    """One nonzero weight at kv_b row 256h+j, column c: only q_lat[:, h, c] is nonzero, equal to
    q_nope[:, h, j] * value * block scale (pins the row/column order and the head offset)."""
    H = 3
    w8 = np.zeros((H * 256, KL), np.uint8)
    w8[256 * h + j, c] = 0x4C  # 1.5 * 2^2 = 6
    sc = np.full((H * 2, 4), 0.5, np.float32)
    sc[2 * h, c // 128] = 0.125
    q = np.random.default_rng(2).standard_normal((4, H, 128)).astype(np.float32)
    got = oracle.q_absorb(q, w8, sc)
    want = np.zeros_like(got)
    want[:, h, c] = (q[:, h, j].astype(np.float64) * 6.0 * 0.125).astype(np.float32)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("h,v,c", [(0, 0, 0), (1, 127, 511), (2, 9, 200)])
def test_out_project_single_weight_lands_at_its_index(oracle, h, v, c):
    H = 3
    w8 = np.zeros((H * 256, KL), np.uint8)
    w8[256 * h + 128 + v, c] = 0xC4  # -(1.5) * 2^1 = -3
    sc = np.full((H * 2, 4), 0.5, np.float32)
    sc[2 * h + 1, c // 128] = 2.0
    x = np.random.default_rng(3).standard_normal((2, H, KL)).astype(np.float32)
    got = oracle.out_project(x, w8, sc)
    want = np.zeros_like(got)
    want[:, h, v] = (x[:, h, c].astype(np.float64) * -3.0 * 2.0).astype(np.float32)
    assert np.array_equal(got, want)


def test_projections_match_a_double_matmul(oracle):
    """Against torch-decoded weights times block scales and an einsum in double."""
    import synth
    H = 4
    w8, sc = synth.kvb_fmt8(H, seed=7)
    W = _kvb_dense(w8, sc).reshape(H, 256, KL)
    rng = np.random.default_rng(4)
    q = rng.standard_normal((3, H, 128)).astype(np.float32)
    x = rng.standard_normal((3, H, KL)).astype(np.float32)
    want_q = np.einsum("shj,hjc->shc", q.astype(np.float64), W[:, :128, :])
    want_o = np.einsum("hvc,shc->shv", W[:, 128:, :], x.astype(np.float64))
    np.testing.assert_allclose(oracle.q_absorb(q, w8, sc), want_q, rtol=2e-7, atol=1e-30 + 1e-7 * np.abs(want_q).max())
    np.testing.assert_allclose(oracle.out_project(x, w8, sc), want_o, rtol=2e-7, atol=1e-7 * np.abs(want_o).max())


def test_block_scale_enters_only_its_block(oracle):
    import synth
    H = 2
    w8, sc = synth.kvb_fmt8(H, seed=8)
    rng = np.random.default_rng(5)
    q = rng.standard_normal((2, H, 128)).astype(np.float32)
    x = rng.standard_normal((2, H, KL)).astype(np.float32)
    base_q, base_o = oracle.q_absorb(q, w8, sc), oracle.out_project(x, w8, sc)
    sc2 = sc.copy()
    sc2[2 * 1 + 0, 2] *= 2.0  # head 1, W_UK, columns 256..383
    got = oracle.q_absorb(q, w8, sc2)
    assert np.array_equal(got[:, 1, 256:384], 2 * base_q[:, 1, 256:384])
    keep = np.ones(got.shape, bool)
    keep[:, 1, 256:384] = False
    assert np.array_equal(got[keep], base_q[keep])
    # value side: the block's share of head 1's outputs doubles, i.e. is added once more
    sc3 = sc.copy()
    sc3[2 * 1 + 1, 3] *= 2.0
    only = np.zeros_like(sc)
    only[2 * 1 + 1, 3] = sc[2 * 1 + 1, 3]
    share = oracle.out_project(x, w8, only)
    got_o = oracle.out_project(x, w8, sc3)
    np.testing.assert_allclose(got_o[:, 1], base_o[:, 1] + share[:, 1], rtol=1e-6, atol=1e-6 * np.abs(base_o).max())
    assert np.array_equal(got_o[:, 0], base_o[:, 0])


def test_absorbed_score_equals_unabsorbed_score(oracle):
    """The absorption identity: q_lat . c == q_nope . (W_UK c) for a latent row c.  W_UK c is computed
    with the value-side function on a kv_b whose value rows are the key rows."""
    import synth
    H = 3
    w8, sc = synth.kvb_fmt8(H, seed=9)
    swapped8 = w8.reshape(H, 2, 128, KL)[:, ::-1].reshape(H * 256, KL).copy()
    swapped_sc = sc.reshape(H, 2, 4)[:, ::-1].reshape(H * 2, 4).copy()
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, H, 128)).astype(np.float32)
    c = rng.standard_normal((1, 1, KL)).astype(np.float32)
    q_lat = oracle.q_absorb(q, w8, sc)[0].astype(np.float64)                        # [H][512]
    k_nope = oracle.out_project(np.repeat(c, H, axis=1), swapped8, swapped_sc)[0]    # [H][128] = W_UK c
    absorbed = q_lat @ c[0, 0].astype(np.float64)
    direct = np.einsum("hj,hj->h", q[0].astype(np.float64), k_nope.astype(np.float64))
    np.testing.assert_allclose(absorbed, direct, rtol=1e-5, atol=1e-5 * np.abs(direct).max())


# ------------------------------------------------------------------------------------------------
# DSA lightning indexer: quantized index query / keys, ReLU-weighted head sum, top-k
# ------------------------------------------------------------------------------------------------
def test_quant_rows_any_width_matches_torch(oracle):
    """Width-128 rows (index keys, index query heads) through the same row quantizer = torch's f32
    amax / multiply-by-448/amax / float8_e4m3fn conversion."""
    rng = np.random.default_rng(20)
    x = (rng.standard_normal((300, 128)) * 10.0 ** rng.uniform(-3, 3, (300, 1))).astype(np.float32)
    q, s = oracle.quant_rows_w(x, 128)
    t = torch.from_numpy(x)
    amax = t.abs().amax(dim=1, keepdim=True)
    y = t * (torch.tensor(448.0, dtype=torch.float32) / amax)
    assert np.array_equal(q, torch_e4m3(y.numpy()))
    assert np.array_equal(s, (amax[:, 0] / torch.tensor(448.0, dtype=torch.float32)).numpy())
    # width 576 through the generic entry = the cache-row quantizer
    x5 = rng.standard_normal((7, 576)).astype(np.float32)
    a, b = oracle.quant_rows(x5), oracle.quant_rows_w(x5, 576)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def _index_case(seed, B=2, HI=5, T=37, stride=50):
    rng = np.random.default_rng(seed)
    qf = rng.standard_normal((B, HI, 128)).astype(np.float32)
    import oracle as o
    q8, qs = o.quant_rows_w(qf.reshape(B * HI, 128), 128)
    kf = (rng.standard_normal(((B - 1) * stride + T, 128)) * 10.0 ** rng.uniform(-1, 1, (((B - 1) * stride + T), 1))).astype(np.float32)
    k8, ks = o.quant_rows_w(kf, 128)
    w = rng.standard_normal((B, HI)).astype(np.float32)
    return q8.reshape(B, HI, 128), qs.reshape(B, HI), w, k8, ks, T, stride


def test_index_scores_match_a_double_einsum(oracle):
    q8, qs, w, k8, ks, T, stride = _index_case(21)
    B, HI, _ = q8.shape
    dq = torch.from_numpy(q8).view(torch.float8_e4m3fn).to(torch.float64).numpy() * qs[..., None].astype(np.float64)
    dk = torch.from_numpy(k8).view(torch.float8_e4m3fn).to(torch.float64).numpy() * ks[:, None].astype(np.float64)
    want = np.zeros((B, T))
    for b in range(B):
        dots = dq[b] @ dk[b * stride:b * stride + T].T          # [HI][T]
        want[b] = (w[b].astype(np.float64)[:, None] * np.maximum(dots, 0.0)).sum(axis=0)
    got = oracle.index_scores(q8, qs, w, k8, ks, T, stride)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_index_score_single_element_closed_form(oracle):
    """One head whose query is a single 1.0 at position j (q_scale 1), weight 2: I_t = 2 max(0, k_scale_t * key_t[j])."""
    T, j = 40, 77
    rng = np.random.default_rng(22)
    k8, ks = oracle.quant_rows_w(rng.standard_normal((T, 128)).astype(np.float32), 128)
    q8 = np.zeros((1, 1, 128), np.uint8)
    q8[0, 0, j] = 0x38
    got = oracle.index_scores(q8, np.ones((1, 1), np.float32), np.full((1, 1), 2.0, np.float32), k8, ks, T, 0)
    key = torch.from_numpy(k8[:, j].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(got[0], 2.0 * np.maximum(ks.astype(np.float64) * key, 0.0))


def test_index_scores_relu_and_linearity(oracle):
    q8, qs, w, k8, ks, T, stride = _index_case(23)
    base = oracle.index_scores(q8, qs, w, k8, ks, T, stride)
    # negating a head's query (sign bit of every byte) swaps which rows its ReLU passes
    neg = q8.copy()
    neg[:, 0] ^= 0x80
    only0 = np.zeros_like(w)
    only0[:, 0] = w[:, 0]
    pos_part = oracle.index_scores(q8, qs, only0, k8, ks, T, stride)
    neg_part = oracle.index_scores(neg, qs, only0, k8, ks, T, stride)
    assert np.all((pos_part == 0) | (neg_part == 0)), "a row passes the ReLU for q or for -q, not both"
    # the weights enter linearly; permuting heads together with their weights changes nothing
    np.testing.assert_allclose(oracle.index_scores(q8, qs, 2 * w, k8, ks, T, stride), 2 * base, rtol=1e-15, atol=0)
    perm = np.array([3, 1, 4, 0, 2])
    np.testing.assert_allclose(oracle.index_scores(q8[:, perm], qs[:, perm], w[:, perm], k8, ks, T, stride), base,
                               rtol=1e-12, atol=1e-12 * np.abs(base).max())


def test_topk_ties_order_and_brute_force(oracle):
    assert list(oracle.topk(np.array([3.0, 1.0, 3.0, 2.0, 3.0]), 2)) == [0, 2]   # ties: the smaller index
    assert list(oracle.topk(np.array([3.0, 1.0, 3.0, 2.0, 3.0]), 4)) == [0, 2, 3, 4]
    assert list(oracle.topk(np.array([1.0, 2.0]), 5)) == [0, 1]                  # k > n: every index
    rng = np.random.default_rng(24)
    for n, k in ((1, 1), (10, 3), (1000, 100), (5000, 2048)):
        s = np.round(rng.standard_normal(n), 1)  # many ties
        got = oracle.topk(s, k)
        order = sorted(range(n), key=lambda i: (-s[i], i))[:k]
        assert list(got) == sorted(order)
        assert np.all(np.diff(got) > 0)


# ------------------------------------------------------------------------------------------------
# mixed-precision cache (448 e4m3 no-position values + f32 row scale, 64 bf16 RoPE values per row)
# ------------------------------------------------------------------------------------------------
def _mixed_cache(oracle, T, seed, mag=(0.1, 10.0)):
    rng = np.random.default_rng(seed)
    nope = (rng.standard_normal((T, 448)) * 10.0 ** rng.uniform(np.log10(mag[0]), np.log10(mag[1]), (T, 1))).astype(np.float32)
    k8, ks = oracle.quant_rows_w(nope, 448)
    kr = torch.from_numpy(rng.standard_normal((T, 64)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    return rng, k8, ks, kr


def _torch_q8(qn):
    """Independent per-row quantization of the queries: torch's f32 amax / multiply / float8_e4m3fn."""
    t = torch.from_numpy(qn)
    amax = t.abs().amax(dim=1, keepdim=True)
    q8 = (t * (torch.tensor(448.0) / amax)).to(torch.float8_e4m3fn)
    return q8.to(torch.float64).numpy(), (amax[:, 0] / torch.tensor(448.0)).double().numpy()


def test_mixed_quant_width_448_matches_torch(oracle):
    rng = np.random.default_rng(50)
    x = (rng.standard_normal((200, 448)) * 10.0 ** rng.uniform(-3, 3, (200, 1))).astype(np.float32)
    q, s = oracle.quant_rows_w(x, 448)
    d, sc = _torch_q8(x)
    assert np.array_equal(torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy(), d)
    assert np.array_equal(s.astype(np.float64), sc)


def test_mixed_single_row_returns_the_row(oracle):
    _, k8, ks, kr = _mixed_cache(oracle, 1, 51)
    rng = np.random.default_rng(52)
    out = oracle.attn_mixed_decode(rng.standard_normal((4, 448)).astype(np.float32),
                                   rng.standard_normal((4, 64)).astype(np.float32), k8, ks, kr, 0.07)
    dk = torch.from_numpy(k8).view(torch.float8_e4m3fn).to(torch.float64).numpy()[0] * np.float64(ks[0])
    for h in range(4):
        assert np.array_equal(out[h, :448], dk.astype(np.float32)) and np.array_equal(out[h, 448:], kr[0])


def test_mixed_zero_query_is_the_mean(oracle):
    T = 37
    _, k8, ks, kr = _mixed_cache(oracle, T, 53)
    out = oracle.attn_mixed_decode(np.zeros((2, 448), np.float32), np.zeros((2, 64), np.float32), k8, ks, kr, 0.07)
    dk = torch.from_numpy(k8).view(torch.float8_e4m3fn).to(torch.float64).numpy() * ks[:, None].astype(np.float64)
    want = np.concatenate([dk.mean(axis=0), kr.astype(np.float64).mean(axis=0)]).astype(np.float32)
    np.testing.assert_allclose(out[0], want, rtol=1e-6, atol=1e-6 * np.abs(want).max())


def test_mixed_two_rows_differing_in_rope_closed_form(oracle):
    """Equal no-position parts, different RoPE parts: the weights are sigma(+-Delta) with Delta the
    sm_scale-weighted RoPE dot difference (the RoPE part enters the score unscaled)."""
    _, k8, ks, kr = _mixed_cache(oracle, 2, 54)
    k8[1], ks[1] = k8[0], ks[0]
    rng = np.random.default_rng(55)
    qn = rng.standard_normal((3, 448)).astype(np.float32)
    qr = torch.from_numpy(rng.standard_normal((3, 64)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    sm = 0.25
    out = oracle.attn_mixed_decode(qn, qr, k8, ks, kr, sm)
    delta = sm * (qr.astype(np.float64) @ (kr[0].astype(np.float64) - kr[1].astype(np.float64)))
    w0 = 1.0 / (1.0 + np.exp(-delta))
    dk = torch.from_numpy(k8[0].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy() * np.float64(ks[0])
    for h in range(3):
        want_rope = w0[h] * kr[0] + (1 - w0[h]) * kr[1]
        np.testing.assert_allclose(out[h, 448:], want_rope, rtol=1e-6, atol=1e-6)
        np.testing.assert_allclose(out[h, :448], dk, rtol=1e-6, atol=1e-6 * np.abs(dk).max())


def test_mixed_matches_a_double_softmax(oracle):
    T, H = 300, 5
    rng, k8, ks, kr = _mixed_cache(oracle, T, 56)
    qn = torch.from_numpy(rng.standard_normal((H, 448)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    qr = torch.from_numpy(rng.standard_normal((H, 64)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    sm = float(np.float32(1.0 / np.sqrt(512.0)))
    q8, qs = _torch_q8(qn)
    dk = torch.from_numpy(k8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s = sm * ((qs[:, None] * ks[None, :].astype(np.float64)) * (q8 @ dk.T) + qr.astype(np.float64) @ kr.T.astype(np.float64))
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    vals = np.concatenate([dk * ks[:, None].astype(np.float64), kr.astype(np.float64)], axis=1)
    want = p @ vals
    got = oracle.attn_mixed_decode(qn, qr, k8, ks, kr, sm)
    np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-6 * np.abs(want).max())
