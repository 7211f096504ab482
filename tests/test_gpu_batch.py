"""GPU batched dense decode (B sequences, each its own cache and length) and the scatter append of one
fresh row per sequence, vs the oracle.

Each sequence's output must match the oracle's single-sequence decode over that sequence's own rows;
the appended rows must be bit-exact.  Edge cases: ragged lengths (1, T_max, in between), a length 0
(zero output), a length above T_max (clamped), H = 65 and 16, f32 queries (CUDA-core path), a scatter
destination outside the cache (skipped and reported); very unequal lengths, all lengths zero, and 70 and 80
sequences (one partition each; 80 sequences take more than one wave of CTAs).
"""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_cache, parity, parity_per_head

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _setup(oracle, B, T_max, stride, seed):
    rng = np.random.default_rng(seed)
    rows = synth.latent_rows(rng, (B - 1) * stride + T_max, 0.1, 10.0)
    q_o, s_o = oracle_cache(oracle, rows)
    return rng, rows, q_o, s_o


def _decode(lib, q_lat, q_rope, kv8, sc, T_max, stride, lens, bf16):
    B, H = q_lat.shape[0], q_lat.shape[1]
    ql, qr = torch.from_numpy(q_lat).to(DEV), torch.from_numpy(q_rope).to(DEV)
    if bf16:
        ql, qr = ql.to(torch.bfloat16), qr.to(torch.bfloat16)
    ws = torch.empty(lib.mla_batch_decode8_workspace_bytes(B, H, T_max) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty((B, H, 512), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.mla_absorb_batch_decode8(ql, qr, kv8, sc, T_max, stride, torch.tensor(lens, dtype=torch.int32, device=DEV),
                                 synth.SM_SCALE, ws, out, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("H,bf16", [(128, True), (65, True), (16, False), (128, False)])
def test_batch_decode_ragged_lengths(lib, oracle, H, bf16):
    B, T_max, stride = 4, 5000, 5003
    lens = [5000, 1, 2345, 129]
    rng, rows, q_o, s_o = _setup(oracle, B, T_max, stride, 40 + H)
    kv8, sc = torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)
    # each sequence's newest row is appended on the GPU, one scatter call for all of them
    dst = np.array([b * stride + lens[b] - 1 for b in range(B)], dtype=np.int64)
    kv8[torch.from_numpy(dst).to(DEV)] = 0
    sc[torch.from_numpy(dst).to(DEV)] = 0
    lib.kv8_quant_rows_scatter(torch.from_numpy(rows[dst]).to(DEV), torch.from_numpy(dst).to(DEV), kv8, sc)
    torch.cuda.synchronize()
    assert np.array_equal(kv8.cpu().numpy()[dst], q_o[dst]) and np.array_equal(sc.cpu().numpy()[dst], s_o[dst])
    q = rng.standard_normal((B, H, 576)).astype(np.float32)
    if bf16:
        q = synth.to_bf16_values(q)
    got = _decode(lib, q[..., :512].copy(), q[..., 512:].copy(), kv8, sc, T_max, stride, lens, bf16)
    for b in range(B):
        lo = b * stride
        ref = oracle.attn_decode(q[b, :, :512], q[b, :, 512:], q_o[lo:lo + lens[b]], s_o[lo:lo + lens[b]], synth.SM_SCALE)
        parity(got[b], ref, f"sequence {b} (len {lens[b]})")


def test_batch_decode_empty_and_clamped_lengths(lib, oracle):
    B, H, T_max, stride = 3, 32, 700, 700
    lens = [0, 10_000, 300]  # no rows -> zeros; more than T_max -> all T_max rows
    rng, rows, q_o, s_o = _setup(oracle, B, T_max, stride, 41)
    q = synth.to_bf16_values(rng.standard_normal((B, H, 576)).astype(np.float32))
    got = _decode(lib, q[..., :512].copy(), q[..., 512:].copy(), torch.from_numpy(q_o).to(DEV),
                  torch.from_numpy(s_o).to(DEV), T_max, stride, lens, True)
    assert not got[0].any()
    for b, n in ((1, T_max), (2, 300)):
        lo = b * stride
        parity(got[b], oracle.attn_decode(q[b, :, :512], q[b, :, 512:], q_o[lo:lo + n], s_o[lo:lo + n], synth.SM_SCALE),
               f"sequence {b}")


@pytest.mark.parametrize("B,T_max,lens_kind", [(5, 3000, "unequal"), (4, 600, "zeros"), (70, 256, "ragged"),
                                               (80, 200, "ragged")])
def test_batch_decode_many_and_unequal_sequences(lib, oracle, B, T_max, lens_kind):
    H, stride = 128, T_max
    rng, rows, q_o, s_o = _setup(oracle, B, T_max, stride, 43 + B)
    if lens_kind == "unequal":
        lens = [T_max, 1, 0, 17, T_max // 3]
    elif lens_kind == "zeros":
        lens = [0] * B
    else:
        lens = [int(x) for x in rng.integers(0, T_max + 1, B)]
        lens[0] = T_max
    q = synth.to_bf16_values(rng.standard_normal((B, H, 576)).astype(np.float32))
    got = _decode(lib, q[..., :512].copy(), q[..., 512:].copy(), torch.from_numpy(q_o).to(DEV),
                  torch.from_numpy(s_o).to(DEV), T_max, stride, lens, True)
    heads = [0, 77, 127]
    for b in range(B):
        n = min(lens[b], T_max)
        if n == 0:
            assert not got[b].any()
            continue
        if B > 8 and b % 7:
            continue  # many sequences: a sample of them against the oracle
        lo = b * stride
        ref = oracle.attn_decode(q[b, heads, :512], q[b, heads, 512:], q_o[lo:lo + n], s_o[lo:lo + n], synth.SM_SCALE)
        parity(got[b][heads], ref, f"sequence {b} of {B} (len {n})")


def test_scatter_out_of_range_destination_is_skipped(lib, oracle):
    rng = np.random.default_rng(42)
    x = synth.latent_rows(rng, 3, 0.1, 10.0)
    kv8 = torch.zeros((10, 576), dtype=torch.uint8, device=DEV)
    sc = torch.zeros(10, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    dst = torch.tensor([2, 10, 7], dtype=torch.int64, device=DEV)  # row 10 is outside the 10-row cache
    lib.kv8_quant_rows_scatter(torch.from_numpy(x).to(DEV), dst, kv8, sc, err_word=err)
    torch.cuda.synchronize()
    q_o, s_o = oracle.quant_rows(x)
    k = kv8.cpu().numpy()
    assert np.array_equal(k[2], q_o[0]) and np.array_equal(k[7], q_o[2])
    assert not np.delete(k, [2, 7], axis=0).any()
    assert err.item() == 1  # KV8_ERR_INDEX


def test_batch_decode_eight_sequences(lib, oracle):
    B, H, T_max = 8, 128, 16384
    lens = [T_max - 997 * b for b in range(B)]
    rng, rows, q_o, s_o = _setup(oracle, B, T_max, T_max, 43)
    q = synth.to_bf16_values(rng.standard_normal((B, H, 576)).astype(np.float32))
    got = _decode(lib, q[..., :512].copy(), q[..., 512:].copy(), torch.from_numpy(q_o).to(DEV),
                  torch.from_numpy(s_o).to(DEV), T_max, T_max, lens, True)
    heads = list(range(0, H, 11))
    for b in range(B):
        lo = b * T_max
        # every head of the longest and the shortest sequence, each head on its own scale; sampled heads of
        # the others
        hs = list(range(H)) if b in (0, B - 1) else heads
        ref = oracle.attn_decode(q[b, hs, :512], q[b, hs, 512:], q_o[lo:lo + lens[b]], s_o[lo:lo + lens[b]],
                                 synth.SM_SCALE)
        if b in (0, B - 1):
            parity_per_head(got[b], ref, f"batch sequence {b} every head")
        else:
            parity(got[b][hs], ref, f"sequence {b}")
