"""GPU DSA lightning indexer (index-key quantizer, tensor-core scores, top-k) vs the oracle.

Index keys come from the oracle's quantizer (never from the GPU), except in the quantizer's own
bit-exact test.  Scores are compared with the oracle's double-precision scores; the selection is
integer work, so the GPU's top-k must equal the oracle's top-k applied to the same (GPU) scores
exactly, and must agree with the oracle's own selection wherever the scores are not within the
tolerance of the k-th score.  Edge cases: T not a multiple of the 128-row tile, T = 1, NS > T, rows
with zero scores (ties resolved by position), f32 and bf16 queries, HI = 16 / 64 / 128.
"""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_cache, parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")
SCORE_TOL = 1e-5  # f32 sums of exact e4m3 products vs double, relative to max |score|


def _keys(oracle, rows):
    k8, ks = oracle.quant_rows_w(rows, 128)
    return k8, ks, torch.from_numpy(k8).to(DEV), torch.from_numpy(ks).to(DEV)


def _run(lib, q, w, tk8, tks, B, T, stride, NS):
    scores = torch.empty((B, T), dtype=torch.float32, device=DEV)
    idx = torch.full((B, NS), -7, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(lib.dsa_index_workspace_bytes(B) // 4, dtype=torch.int32, device=DEV)
    lib.dsa_index_topk8(q, w, tk8, tks, T, stride, NS, ws, scores, idx, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return scores.cpu().numpy(), idx.cpu().numpy()


def _qtensor(q, bf16):
    t = torch.from_numpy(np.ascontiguousarray(q)).to(DEV)
    return t.to(torch.bfloat16) if bf16 else t


def test_quant_rows_width_128_bit_exact(lib, oracle):
    rng = np.random.default_rng(30)
    x = (rng.standard_normal((1000, 128)) * 10.0 ** rng.uniform(-4, 4, (1000, 1))).astype(np.float32)
    x[5] = 0.0
    x[6] = rng.standard_normal(128).astype(np.float32) * np.float32(1e-39)   # subnormal amax
    x[7, 3] = np.float32(-0.0)
    q = torch.empty((1000, 128), dtype=torch.uint8, device=DEV)
    s = torch.empty(1000, dtype=torch.float32, device=DEV)
    lib.kv8_quant_rows_w(torch.from_numpy(x).to(DEV), q, s)
    torch.cuda.synchronize()
    q_o, s_o = oracle.quant_rows_w(x, 128)
    assert np.array_equal(q.cpu().numpy(), q_o)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), s_o.view(np.uint32))


@pytest.mark.parametrize("B,HI,T,stride,bf16", [(1, 64, 1, 1, True), (2, 64, 129, 200, True), (3, 16, 1000, 1000, False),
                                                (2, 128, 700, 901, True), (1, 48, 5000, 5000, False)])
def test_index_scores_and_topk(lib, oracle, B, HI, T, stride, bf16):
    rng = np.random.default_rng(B * 1000 + HI + T)
    rows = (rng.standard_normal(((B - 1) * stride + T, 128)) * 10.0 ** rng.uniform(-0.5, 0.5, ((B - 1) * stride + T, 1))).astype(np.float32)
    k8, ks, tk8, tks = _keys(oracle, rows)
    q = rng.standard_normal((B, HI, 128)).astype(np.float32)
    if bf16:
        q = synth.to_bf16_values(q)
    q[0, 1] = 0.0  # a head whose query is all zero
    w = (rng.standard_normal((B, HI)) / 8).astype(np.float32)
    NS = max(1, T // 3)
    scores, idx = _run(lib, _qtensor(q, bf16), torch.from_numpy(w).to(DEV), tk8, tks, B, T, stride, NS)
    q8, qs = oracle.quant_rows_w(q.reshape(B * HI, 128), 128)
    ref = oracle.index_scores(q8.reshape(B, HI, 128), qs.reshape(B, HI), w, k8, ks, T, stride)
    err = np.abs(scores - ref).max() / max(np.abs(ref).max(), 1e-30)
    assert err <= SCORE_TOL, f"scores: max error {err:.2e} of max |score|"
    for b in range(B):
        # the selection is integer work on the GPU's scores: exact
        assert np.array_equal(idx[b], oracle.topk(scores[b].astype(np.float64), NS))
        # and it agrees with the oracle's selection away from the k-th score
        kth = np.sort(ref[b])[::-1][NS - 1]
        margin = SCORE_TOL * np.abs(ref).max()
        sel = np.zeros(T, bool)
        sel[idx[b]] = True
        assert sel[ref[b] > kth + margin].all() and not sel[ref[b] < kth - margin].any()


def test_topk_ties_and_short_lists(lib, oracle):
    """Rows with zero scale score exactly 0: many equal scores, resolved by position; NS > T takes all."""
    B, HI, T = 2, 64, 3000
    rng = np.random.default_rng(31)
    rows = rng.standard_normal((B * T, 128)).astype(np.float32)
    rows[rng.random(B * T) < 0.7] = 0.0
    k8, ks, tk8, tks = _keys(oracle, rows)
    q = synth.to_bf16_values(rng.standard_normal((B, HI, 128)).astype(np.float32))
    w = np.abs(rng.standard_normal((B, HI))).astype(np.float32)
    for NS in (1, 1500, 2999, 4096):
        scores, idx = _run(lib, _qtensor(q, True), torch.from_numpy(w).to(DEV), tk8, tks, B, T, T, NS)
        for b in range(B):
            want = oracle.topk(scores[b].astype(np.float64), NS)
            got = idx[b][:len(want)]
            assert np.array_equal(got, want), f"NS={NS} b={b}"
            if NS >= T:
                assert np.array_equal(got, np.arange(T)) and np.all(idx[b][T:] == -7)  # nothing past min(NS, T)


@pytest.mark.parametrize("B,T,zero_frac", [(2, 20000, 0.9), (76, 10000, 0.9), (8, 40000, 0.95)])
def test_topk_heavy_ties_across_ctas(lib, oracle, B, T, zero_frac):
    """Most rows score exactly 0 and the k-th score is 0, so the selection ends inside a tie thousands of
    keys long that spans every CTA of a query.  All B queries read the same key rows (stride 0) with their
    own query.  On a 152-SM GPU a query has 76 CTAs (B=2), 2 CTAs of 5000 positions, ~4500 of them tied
    (B=76), or 19 CTAs over 38,000 tied keys (B=8).  The selection must equal the oracle's top-k of the
    GPU scores: every positive score, then the tied zeros from the smallest position on."""
    HI = 16
    rng = np.random.default_rng(T + B)
    rows = rng.standard_normal((T, 128)).astype(np.float32)
    rows[rng.random(T) < zero_frac] = 0.0
    k8, ks, tk8, tks = _keys(oracle, rows)
    q = synth.to_bf16_values(rng.standard_normal((B, HI, 128)).astype(np.float32))
    w = np.abs(rng.standard_normal((B, HI))).astype(np.float32)
    NS = 3000
    scores, idx = _run(lib, _qtensor(q, True), torch.from_numpy(w).to(DEV), tk8, tks, B, T, 0, NS)
    zero = ks == 0.0
    assert np.all(scores[:, zero] == 0.0)
    for b in range(B):
        assert np.count_nonzero(scores[b] > 0) < NS  # the k-th score is 0
        assert np.array_equal(idx[b], oracle.topk(scores[b].astype(np.float64), NS)), f"query {b}"


def test_indexer_workload_sampled(lib, oracle):
    """The indexer workload (B=8 x T=131072, HI=64, NS=2048): scores of sequences 0 and 7 against the
    oracle; every sequence's selection = the oracle's top-k of the GPU scores."""
    w_ = synth.WORKLOADS["indexer"]
    B, T, HI, NS = w_.B, w_.T, w_.H, w_.NS
    k8 = torch.empty((B * T, 128), dtype=torch.uint8, device=DEV)
    ks = torch.empty(B * T, dtype=torch.float32, device=DEV)
    keys_o = {}
    for b in range(B):
        rows = synth.index_keys_for(w_, b)
        q_o, s_o = oracle.quant_rows_w(rows, 128)
        if b in (0, B - 1):
            keys_o[b] = (q_o, s_o)
        k8[b * T:(b + 1) * T] = torch.from_numpy(q_o).to(DEV)
        ks[b * T:(b + 1) * T] = torch.from_numpy(s_o).to(DEV)
    q = synth.index_queries_for(w_)
    w = synth.index_weights_for(w_)
    scores, idx = _run(lib, _qtensor(q, True), torch.from_numpy(w).to(DEV), k8, ks, B, T, T, NS)
    q8, qs = oracle.quant_rows_w(q.reshape(B * HI, 128), 128)
    q8, qs = q8.reshape(B, HI, 128), qs.reshape(B, HI)
    for b, (kq, kss) in keys_o.items():
        ref = oracle.index_scores(q8[b:b + 1], qs[b:b + 1], w[b:b + 1], kq, kss, T, 0)[0]
        err = np.abs(scores[b] - ref).max() / np.abs(ref).max()
        assert err <= SCORE_TOL, f"sequence {b}: max error {err:.2e}"
    for b in range(B):
        assert np.array_equal(idx[b], oracle.topk(scores[b].astype(np.float64), NS))


def test_indexer_then_selected_attention(lib, oracle):
    """The DSA chain: the indexer's selection feeds mla_absorb_sel8; the attention over those rows matches
    the oracle's attention over the same list."""
    B, HI, T, NS, H = 2, 64, 3000, 500, 128
    rng = np.random.default_rng(32)
    krows = rng.standard_normal((B * T, 128)).astype(np.float32)
    k8, ks, tk8, tks = _keys(oracle, krows)
    qi = synth.to_bf16_values(rng.standard_normal((B, HI, 128)).astype(np.float32))
    w = (rng.standard_normal((B, HI)) / 8).astype(np.float32)
    _, idx = _run(lib, _qtensor(qi, True), torch.from_numpy(w).to(DEV), tk8, tks, B, T, T, NS)
    lat = synth.latent_rows(rng, B * T, 0.1, 10.0)
    q_o, s_o = oracle_cache(oracle, lat)
    ql = synth.to_bf16_values(rng.standard_normal((B, H, 512)).astype(np.float32))
    qr = synth.to_bf16_values(rng.standard_normal((B, H, 64)).astype(np.float32))
    ws = torch.empty(lib.mla_sel8_workspace_bytes(B, H, NS) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty((B, H, 512), dtype=torch.float32, device=DEV)
    lib.mla_absorb_sel8(_qtensor(ql, True), _qtensor(qr, True), torch.from_numpy(q_o).to(DEV),
                        torch.from_numpy(s_o).to(DEV), T, T, torch.from_numpy(idx).to(DEV), synth.SM_SCALE, ws, out)
    torch.cuda.synchronize()
    ref, n_bad = oracle.attn_select(ql, qr, q_o, s_o, T, T, idx, synth.SM_SCALE)
    assert n_bad == 0
    parity(out.cpu().numpy(), ref, "attention over the indexer's selection")


def test_workspace_reused_and_dirty(lib, oracle):
    """The call zeroes its workspace itself (histograms, counts, barrier counters): a workspace that holds
    garbage, or the previous call's state, gives the same scores and the same selection."""
    rng = np.random.default_rng(35)
    B, HI, T, NS = 3, 64, 5000, 300
    rows = (rng.standard_normal((B * T, 128)) * 10.0 ** rng.uniform(-1, 1, (B * T, 1))).astype(np.float32)
    k8, ks, tk8, tks = _keys(oracle, rows)
    q = _qtensor(synth.to_bf16_values(rng.standard_normal((B, HI, 128)).astype(np.float32)), True)
    w = torch.from_numpy(rng.standard_normal((B, HI)).astype(np.float32)).to(DEV)
    ws = torch.full((lib.dsa_index_workspace_bytes(B) // 4,), 0x5A5A5A5A, dtype=torch.int32, device=DEV)
    outs = []
    for _ in range(3):
        scores = torch.empty((B, T), dtype=torch.float32, device=DEV)
        idx = torch.full((B, NS), -7, dtype=torch.int32, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        lib.dsa_index_topk8(q, w, tk8, tks, T, T, NS, ws, scores, idx, err_word=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        outs.append((scores.cpu().numpy(), idx.cpu().numpy()))
    for s_, i_ in outs[1:]:
        assert np.array_equal(s_, outs[0][0]) and np.array_equal(i_, outs[0][1])
    for b in range(B):
        assert np.array_equal(outs[0][1][b], oracle.topk(outs[0][0][b], NS))


def test_more_queries_than_ctas_per_wave(lib, oracle):
    """B = 160 queries: more than the GPU's SMs, so each query gets one CTA (no barrier between CTAs, not
    a cooperative launch) and the grid runs in more than one wave; short ragged key lists.  Every
    query's selection = the oracle's top-k of the GPU scores; scores of two queries against the oracle."""
    rng = np.random.default_rng(36)
    B, HI, T, NS = 160, 16, 300, 64
    rows = (rng.standard_normal((B * T, 128)) * 10.0 ** rng.uniform(-0.5, 0.5, (B * T, 1))).astype(np.float32)
    k8, ks, tk8, tks = _keys(oracle, rows)
    q = synth.to_bf16_values(rng.standard_normal((B, HI, 128)).astype(np.float32))
    w = (rng.standard_normal((B, HI)) / 8).astype(np.float32)
    scores, idx = _run(lib, _qtensor(q, True), torch.from_numpy(w).to(DEV), tk8, tks, B, T, T, NS)
    q8, qs = oracle.quant_rows_w(q.reshape(B * HI, 128), 128)
    q8, qs = q8.reshape(B, HI, 128), qs.reshape(B, HI)
    for b in (0, B - 1):
        ref = oracle.index_scores(q8[b:b + 1], qs[b:b + 1], w[b:b + 1], k8[b * T:(b + 1) * T], ks[b * T:(b + 1) * T], T, 0)[0]
        err = np.abs(scores[b] - ref).max() / np.abs(ref).max()
        assert err <= SCORE_TOL, f"query {b}: max error {err:.2e}"
    for b in range(B):
        assert np.array_equal(idx[b], oracle.topk(scores[b].astype(np.float64), NS)), f"query {b}"
