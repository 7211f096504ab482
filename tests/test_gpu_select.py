"""GPU selected-row (DSA gather) decode vs the oracle.

Full workload: B = 8 sequences, each with its own T = 131072-row cache, NS = 2048 sorted unique
indices; every head of the first and the last sequence (each head on its own scale) and sampled heads
of every sequence compared with the oracle.  Edge cases: a full index list
equals dense decode, NS = 1, duplicate indices, out-of-range indices (skipped and flagged).
"""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_cache, parity, parity_per_head

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _sel(lib, q_lat, q_rope, kv8, sc, T, stride, idx, err=None):
    B, NS = idx.shape
    H = q_lat.shape[1]
    ws = torch.empty(lib.mla_sel8_workspace_bytes(B, H, NS) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty((B, H, 512), dtype=torch.float32, device=DEV)
    lib.mla_absorb_sel8(q_lat, q_rope, kv8, sc, T, stride, idx, synth.SM_SCALE, ws, out, err_word=err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_select_full_workload_sampled_heads(lib, oracle):
    w = synth.WORKLOADS["dsa"]
    q_all = np.empty((w.B * w.T, 576), dtype=np.uint8)
    s_all = np.empty(w.B * w.T, dtype=np.float32)
    for b in range(w.B):
        for start in range(0, w.T, 65536):
            rows = synth.rows_for(w, b, start, 65536)
            q, s = oracle_cache(oracle, rows)
            q_all[b * w.T + start:b * w.T + start + 65536] = q
            s_all[b * w.T + start:b * w.T + start + 65536] = s
    idx = synth.selection_for(w)
    ql, qr = synth.queries_for(w)
    kv8 = torch.from_numpy(q_all).to(DEV)
    sc = torch.from_numpy(s_all).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _sel(lib, torch.from_numpy(ql).to(DEV).to(torch.bfloat16), torch.from_numpy(qr).to(DEV).to(torch.bfloat16),
               kv8, sc, w.T, w.T, torch.from_numpy(idx).to(DEV), err)
    assert err.item() == 0
    # every head of the first and the last sequence, each head on its own scale
    for b in (0, w.B - 1):
        ref, bad = oracle.attn_select(ql[b:b + 1], qr[b:b + 1], q_all[b * w.T:(b + 1) * w.T],
                                      s_all[b * w.T:(b + 1) * w.T], w.T, w.T, idx[b:b + 1], synth.SM_SCALE)
        assert bad == 0
        parity_per_head(got[b], ref[0], f"dsa sequence {b} every head")
    # sampled heads of all sequences
    heads = [0, 5, 64, 127]
    ref, bad = oracle.attn_select(ql[:, heads], qr[:, heads], q_all, s_all, w.T, w.T, idx, synth.SM_SCALE)
    assert bad == 0
    parity(got[:, heads], ref, "dsa sampled heads")


def _small(oracle, B, T, H, seed):
    rng = np.random.default_rng(seed)
    rows = synth.latent_rows(rng, B * T, 0.1, 10.0)
    q_o, s_o = oracle.quant_rows(rows)
    q = synth.to_bf16_values(synth.normal_f32(rng, (B, H, 576)))
    return q_o, s_o, np.ascontiguousarray(q[..., :512]), np.ascontiguousarray(q[..., 512:]), rng


def _bf(v):
    return torch.from_numpy(v).to(DEV).to(torch.bfloat16)


def test_select_full_index_equals_dense(lib, oracle):
    B, T, H = 2, 300, 40
    q_o, s_o, ql, qr, _ = _small(oracle, B, T, H, 1)
    kv8, sc = torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)
    idx = np.tile(np.arange(T, dtype=np.int32), (B, 1))
    got = _sel(lib, _bf(ql), _bf(qr), kv8, sc, T, T, torch.from_numpy(idx).to(DEV))
    for b in range(B):
        ref = oracle.attn_decode(ql[b], qr[b], q_o[b * T:(b + 1) * T], s_o[b * T:(b + 1) * T], synth.SM_SCALE)
        parity(got[b], ref, f"full index b={b}")
        ws = torch.empty(lib.mla_decode8_workspace_bytes(H, T) // 4, dtype=torch.float32, device=DEV)
        dense = torch.empty((H, 512), dtype=torch.float32, device=DEV)
        lib.mla_absorb_decode8(_bf(ql[b]), _bf(qr[b]), kv8[b * T:(b + 1) * T], sc[b * T:(b + 1) * T], T,
                               synth.SM_SCALE, ws, dense)
        torch.cuda.synchronize()
        parity(got[b], dense.cpu().numpy(), f"select vs dense b={b}")


def test_select_single_duplicate_and_out_of_range(lib, oracle):
    B, T, H = 3, 500, 16
    q_o, s_o, ql, qr, rng = _small(oracle, B, T, H, 2)
    kv8, sc = torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)
    # NS = 1
    idx1 = np.array([[7], [499], [0]], dtype=np.int32)
    got = _sel(lib, _bf(ql), _bf(qr), kv8, sc, T, T, torch.from_numpy(idx1).to(DEV))
    ref, bad = oracle.attn_select(ql, qr, q_o, s_o, T, T, idx1, synth.SM_SCALE)
    assert bad == 0
    parity(got, ref, "NS=1")
    # duplicates and unsorted order
    idx2 = np.array([[5, 5, 9, 1, 5], [2, 3, 4, 2, 2], [499, 0, 499, 10, 11]], dtype=np.int32)
    got = _sel(lib, _bf(ql), _bf(qr), kv8, sc, T, T, torch.from_numpy(idx2).to(DEV))
    parity(got, oracle.attn_select(ql, qr, q_o, s_o, T, T, idx2, synth.SM_SCALE)[0], "duplicates")
    # out of range: skipped and flagged
    idx3 = np.array([[5, -1, 9, 500, 7], [2, 3, 4, 5, 6], [1 << 30, 8, 9, 10, -7]], dtype=np.int32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _sel(lib, _bf(ql), _bf(qr), kv8, sc, T, T, torch.from_numpy(idx3).to(DEV), err)
    assert err.item() & lib.KV8_ERR_INDEX
    ref, bad = oracle.attn_select(ql, qr, q_o, s_o, T, T, idx3, synth.SM_SCALE)
    assert bad == 4  # -1 and 500 in sequence 0; 1<<30 and -7 in sequence 2
    parity(got, ref, "out of range")
    # every index invalid: output 0
    idx4 = np.full((B, 4), -3, dtype=np.int32)
    got = _sel(lib, _bf(ql), _bf(qr), kv8, sc, T, T, torch.from_numpy(idx4).to(DEV))
    assert np.all(got == 0)


def test_select_ragged_ns(lib, oracle):
    B, T, H = 2, 6000, 128
    q_o, s_o, ql, qr, rng = _small(oracle, B, T, H, 3)
    kv8, sc = torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)
    for NS in [129, 4096, 1000]:
        idx = np.stack([np.sort(rng.choice(T, NS, replace=False)) for _ in range(B)]).astype(np.int32)
        got = _sel(lib, _bf(ql), _bf(qr), kv8, sc, T, T, torch.from_numpy(idx).to(DEV))
        heads = [0, 63, 127]
        parity(got[:, heads], oracle.attn_select(ql[:, heads], qr[:, heads], q_o, s_o, T, T, idx,
                                                 synth.SM_SCALE)[0], f"NS={NS}")


def test_select_f32_queries(lib, oracle):
    # f32 queries keep full precision on the CUDA-core kernel
    B, T, H = 2, 400, 20
    rng = np.random.default_rng(4)
    rows = synth.latent_rows(rng, B * T, 0.1, 10.0)
    q_o, s_o = oracle.quant_rows(rows)
    q = synth.normal_f32(rng, (B, H, 576))
    ql, qr = np.ascontiguousarray(q[..., :512]), np.ascontiguousarray(q[..., 512:])
    idx = rng.integers(0, T, size=(B, 300)).astype(np.int32)
    got = _sel(lib, torch.from_numpy(ql).to(DEV), torch.from_numpy(qr).to(DEV), torch.from_numpy(q_o).to(DEV),
               torch.from_numpy(s_o).to(DEV), T, T, torch.from_numpy(idx).to(DEV))
    parity(got, oracle.attn_select(ql, qr, q_o, s_o, T, T, idx, synth.SM_SCALE)[0], "f32 queries")


def test_select_partitions_with_no_valid_row(lib, oracle):
    # whole partitions whose indices are all out of range, next to partitions with valid rows
    B, T, H = 2, 3000, 128
    q_o, s_o, ql, qr, rng = _small(oracle, B, T, H, 5)
    NS = 1024
    idx = rng.integers(0, T, size=(B, NS)).astype(np.int32)
    idx[0, :512] = -5          # the first half of sequence 0's list
    idx[1, 700:] = T + 3       # the tail of sequence 1's list
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _sel(lib, _bf(ql), _bf(qr), torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV), T, T,
               torch.from_numpy(idx).to(DEV), err)
    assert err.item() & lib.KV8_ERR_INDEX
    heads = [1, 64, 100]
    ref, bad = oracle.attn_select(ql[:, heads], qr[:, heads], q_o, s_o, T, T, idx, synth.SM_SCALE)
    assert bad == 512 + (NS - 700)
    parity(got[:, heads], ref, "partitions without valid rows")


def test_select_repeated_calls_identical(lib, oracle):
    """Repeated selection decodes give bit-identical outputs (a race between the row copies, the score
    and the context product would show up as a mismatch); several tiles per partition."""
    B, T, H = 2, 5000, 128
    q_o, s_o, ql, qr, rng = _small(oracle, B, T, H, 6)
    kv8, sc = torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)
    for NS in (700, 4096):
        idx = np.stack([rng.choice(T, NS, replace=True) for _ in range(B)]).astype(np.int32)
        tidx = torch.from_numpy(idx).to(DEV)
        first = _sel(lib, _bf(ql), _bf(qr), kv8, sc, T, T, tidx)
        for _ in range(10):
            assert np.array_equal(_sel(lib, _bf(ql), _bf(qr), kv8, sc, T, T, tidx), first), f"NS={NS}"
        heads = [0, 77, 127]
        parity(first[:, heads], oracle.attn_select(ql[:, heads], qr[:, heads], q_o, s_o, T, T, idx,
                                                   synth.SM_SCALE)[0], f"NS={NS}")


def test_select_more_sequences_than_one_wave(lib, oracle):
    """B = 90 sequences x 2 head halves: more CTAs than SMs (one partition per sequence, the grid in two
    waves behind the query prep); ragged lists of 200 positions; sampled heads of every sequence."""
    B, T, H, NS = 90, 500, 128, 200
    q_o, s_o, ql, qr, rng = _small(oracle, B, T, H, 9)
    kv8, sc = torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)
    idx = np.stack([np.sort(rng.choice(T, NS, replace=False)) for _ in range(B)]).astype(np.int32)
    got = _sel(lib, _bf(ql), _bf(qr), kv8, sc, T, T, torch.from_numpy(idx).to(DEV))
    heads = [0, 64, 127]
    ref, n_bad = oracle.attn_select(ql[:, heads], qr[:, heads], q_o, s_o, T, T, idx, synth.SM_SCALE)
    assert n_bad == 0
    parity(got[:, heads], ref, "90 sequences, sampled heads")
