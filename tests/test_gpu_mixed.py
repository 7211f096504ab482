"""GPU decode over the mixed-precision cache (448 e4m3 no-position values + row scale, 64 bf16 RoPE values)
vs the oracle.

The cache's e4m3 bytes come from the oracle's quantizer (the GPU's width-448 quantizer is checked
bit-exact separately).  Both sides quantize the query's no-position part the same way (the row
quantizer), so the comparison is of the attention itself, at the attention tolerance.  Edge cases:
T = 1 and T around the 128-row tile, several tiles per partition, H not a multiple of the 64-head
half, f32 queries (the RoPE query then enters as bf16 hi + lo).
"""
import numpy as np
import pytest
import torch

import synth
from helpers import parity, parity_per_head

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _cache(oracle, nope, rope):
    k8, ks = oracle.quant_rows_w(nope, 448)
    return k8, ks, torch.from_numpy(k8).to(DEV), torch.from_numpy(ks).to(DEV), \
        torch.from_numpy(rope).to(DEV).to(torch.bfloat16)


def _run(lib, qn, qr, tk8, tks, tkr, bf16, sm=synth.SM_SCALE, err=None):
    H, T = qn.shape[0], tk8.shape[0]
    tq = torch.from_numpy(np.ascontiguousarray(qn)).to(DEV)
    tr = torch.from_numpy(np.ascontiguousarray(qr)).to(DEV)
    if bf16:
        tq, tr = tq.to(torch.bfloat16), tr.to(torch.bfloat16)
    ws = torch.empty(lib.mla_mixed_decode8_workspace_bytes(H, T) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty((H, 512), dtype=torch.float32, device=DEV)
    lib.mla_absorb_mixed_decode8(tq, tr, tk8, tks, tkr, sm, ws, out, err_word=err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_quant_rows_width_448_bit_exact(lib, oracle):
    rng = np.random.default_rng(60)
    x = (rng.standard_normal((500, 448)) * 10.0 ** rng.uniform(-4, 4, (500, 1))).astype(np.float32)
    x[3] = 0.0
    x[4] = rng.standard_normal(448).astype(np.float32) * np.float32(1e-39)
    q = torch.empty((500, 448), dtype=torch.uint8, device=DEV)
    s = torch.empty(500, dtype=torch.float32, device=DEV)
    lib.kv8_quant_rows_w(torch.from_numpy(x).to(DEV), q, s)
    torch.cuda.synchronize()
    q_o, s_o = oracle.quant_rows_w(x, 448)
    assert np.array_equal(q.cpu().numpy(), q_o) and np.array_equal(s.cpu().numpy().view(np.uint32), s_o.view(np.uint32))


@pytest.mark.parametrize("T,H,bf16", [(1, 128, True), (63, 5, True), (64, 128, True), (65, 33, False),
                                      (127, 64, True), (128, 65, True), (129, 128, False), (257, 1, True),
                                      (1000, 128, True), (5000, 16, False), (40000, 128, True),
                                      (40000, 97, False)])
def test_mixed_decode_parity(lib, oracle, T, H, bf16):
    rng = np.random.default_rng(T * 7 + H)
    nope = (rng.standard_normal((T, 448)) * 10.0 ** rng.uniform(-1, 1, (T, 1))).astype(np.float32)
    rope = synth.to_bf16_values(rng.standard_normal((T, 64)).astype(np.float32))
    k8, ks, tk8, tks, tkr = _cache(oracle, nope, rope)
    q = rng.standard_normal((H, 512)).astype(np.float32)
    if bf16:
        q = synth.to_bf16_values(q)
    qn, qr = np.ascontiguousarray(q[:, :448]), np.ascontiguousarray(q[:, 448:])
    got = _run(lib, qn, qr, tk8, tks, tkr, bf16)
    parity(got, oracle.attn_mixed_decode(qn, qr, k8, ks, rope, synth.SM_SCALE), f"T={T} H={H}")


def test_mixed_decode_workload_every_head(lib, oracle):
    """The full mixed-cache workload in the benchmark's launch configuration: every head against the
    oracle, each head on its own scale."""
    w = synth.WORKLOADS["mixed_dec"]
    nope, rope = synth.mixed_rows_for(w)
    k8, ks, tk8, tks, tkr = _cache(oracle, nope, rope)
    qn, qr = synth.mixed_queries_for(w)
    got = _run(lib, qn, qr, tk8, tks, tkr, True)
    parity_per_head(got, oracle.attn_mixed_decode(qn, qr, k8, ks, rope, synth.SM_SCALE), "mixed_dec every head")


def test_mixed_decode_error_word_stays_clear(lib, oracle):
    rng = np.random.default_rng(61)
    T, H = 3000, 128
    nope = rng.standard_normal((T, 448)).astype(np.float32)
    rope = synth.to_bf16_values(rng.standard_normal((T, 64)).astype(np.float32))
    k8, ks, tk8, tks, tkr = _cache(oracle, nope, rope)
    q = synth.to_bf16_values(rng.standard_normal((H, 512)).astype(np.float32))
    qn, qr = np.ascontiguousarray(q[:, :448]), np.ascontiguousarray(q[:, 448:])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _run(lib, qn, qr, tk8, tks, tkr, True, err=err)
    assert int(err.item()) == 0
    parity(got, oracle.attn_mixed_decode(qn, qr, k8, ks, rope, synth.SM_SCALE), "err word run")
