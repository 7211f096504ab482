"""GPU causal prefill vs the oracle.

Small chunk: every query and head.  Full workload (S = 1024 queries at 64512..65535 over T = 65536
rows, H = 128): the 1024 fresh rows are quantized on the GPU in-run (checked bit-exact), then 64
queries -- the first, the last and 62 spread between -- are compared with the oracle on every head
(each head on its own scale); the last query also equals a full-T decode on the GPU.
"""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_cache, parity, parity_per_head

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _prefill(lib, ql, qr, pos0, kv8, sc, T):
    S, H = ql.shape[0], ql.shape[1]
    out = torch.empty((S, H, 512), dtype=torch.float32, device=DEV)
    lib.mla_absorb_prefill8(ql, qr, pos0, kv8, sc, T, synth.SM_SCALE, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("f32", [True, False])
def test_prefill_small_every_query(lib, oracle, f32):
    rng = np.random.default_rng(11)
    T, S, H = 300, 8, 20
    pos0 = T - S
    rows = synth.latent_rows(rng, T, 0.1, 10.0)
    q_o, s_o = oracle.quant_rows(rows)
    q = synth.normal_f32(rng, (S, H, 576))
    if not f32:
        q = synth.to_bf16_values(q)
    ql, qr = np.ascontiguousarray(q[..., :512]), np.ascontiguousarray(q[..., 512:])
    tq = (lambda v: torch.from_numpy(v).to(DEV)) if f32 else (lambda v: torch.from_numpy(v).to(DEV).to(torch.bfloat16))
    got = _prefill(lib, tq(ql), tq(qr), pos0, torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV), T)
    ref = oracle.attn_prefill(ql, qr, pos0 + np.arange(S), q_o, s_o, synth.SM_SCALE)
    parity(got, ref, "prefill small")


def test_prefill_positions_at_zero(lib, oracle):
    """pos0 = 0: query 0 sees one row (its own), query i sees i+1 rows."""
    rng = np.random.default_rng(12)
    T, S, H = 70, 70, 3
    rows = synth.latent_rows(rng, T, 0.1, 10.0)
    q_o, s_o = oracle.quant_rows(rows)
    q = synth.to_bf16_values(synth.normal_f32(rng, (S, H, 576)))
    ql, qr = np.ascontiguousarray(q[..., :512]), np.ascontiguousarray(q[..., 512:])
    bf = lambda v: torch.from_numpy(v).to(DEV).to(torch.bfloat16)
    got = _prefill(lib, bf(ql), bf(qr), 0, torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV), T)
    parity(got, oracle.attn_prefill(ql, qr, np.arange(S), q_o, s_o, synth.SM_SCALE), "pos0=0")
    tab = oracle.e4m3_table()
    np.testing.assert_allclose(got[0, 0], tab[q_o[0, :512]] * np.float64(s_o[0]), rtol=1e-6)


def test_prefill_full_workload_sampled(lib, oracle):
    w = synth.WORKLOADS["prefill"]
    rows = synth.rows_for(w)
    q_o, s_o = oracle_cache(oracle, rows)
    kv8 = torch.from_numpy(q_o).to(DEV)
    sc = torch.from_numpy(s_o).to(DEV)
    kv8[w.pos0:].fill_(0)
    sc[w.pos0:].fill_(0)
    fresh = torch.from_numpy(rows[w.pos0:].copy()).to(DEV)
    lib.kv8_quant_rows(fresh, kv8[w.pos0:], sc[w.pos0:])
    torch.cuda.synchronize()
    assert np.array_equal(kv8.cpu().numpy(), q_o)
    ql, qr = synth.queries_for(w)
    bf = lambda v: torch.from_numpy(v).to(DEV).to(torch.bfloat16)
    tql, tqr = bf(ql), bf(qr)
    got = _prefill(lib, tql, tqr, w.pos0, kv8, sc, w.T)
    assert np.all(np.isfinite(got))
    # 64 queries (the first, the last and 62 spread between) x every head, each head on its own scale
    qs = sorted({0, w.S - 1} | set(np.linspace(1, w.S - 2, 62).astype(int).tolist()))
    assert len(qs) == 64
    ref = oracle.attn_prefill(ql[qs], qr[qs], w.pos0 + np.array(qs), q_o, s_o, synth.SM_SCALE)
    parity_per_head(got[qs], ref, "prefill 64 queries every head")
    # the last query attends the whole cache: equal to decode over all T rows
    ws = torch.empty(lib.mla_decode8_workspace_bytes(w.H, w.T) // 4, dtype=torch.float32, device=DEV)
    dec = torch.empty((w.H, 512), dtype=torch.float32, device=DEV)
    lib.mla_absorb_decode8(tql[-1], tqr[-1], kv8, sc, w.T, synth.SM_SCALE, ws, dec)
    torch.cuda.synchronize()
    parity(got[-1], dec.cpu().numpy(), "last query vs decode")
