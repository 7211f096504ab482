"""GPU absorb projections through an fmt=8 kv_b vs the oracle.

The weights are synthetic fmt=8 bytes and block scales (synth.kvb_fmt8).  Every kernel shape is
covered: the weight-streaming kernels (S <= 8, three instantiations) and the tiled ones (S > 8,
ragged last tile), H = 128 and a ragged H, f32 and bf16 queries and q_lat.  The prefill shape
(S = 1024) is checked on sampled rows; a chain q_nope -> q_lat -> split-T decode -> merge ->
output projection is checked against the oracle's chain.
"""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_cache, parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")

F32_TOL = 2e-5  # f32 sums of exactly decoded weights vs double: relative to max |oracle|


def _close(got, ref, tol, what):
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64)).max() / max(np.abs(ref).max(), 1e-30)
    l2 = np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-30)
    assert err <= tol and l2 <= tol, f"{what}: max err {err:.2e}, rel-L2 {l2:.2e} (tolerance {tol:.0e})"


def _weights(H, seed):
    w8, sc = synth.kvb_fmt8(H, seed=seed)
    return w8, sc, torch.from_numpy(w8).to(DEV), torch.from_numpy(sc).to(DEV)


@pytest.mark.parametrize("S,H", [(1, 128), (3, 128), (8, 5), (9, 128), (64, 7), (65, 128), (130, 16)])
@pytest.mark.parametrize("q_bf16,out_bf16", [(False, False), (True, False), (True, True)])
def test_q_absorb_parity(lib, oracle, S, H, q_bf16, out_bf16):
    w8, sc, tw8, tsc = _weights(H, 11)
    q = synth.normal_f32(np.random.default_rng(S * 131 + H), (S, H, 128))
    if q_bf16:
        q = synth.to_bf16_values(q)
    tq = torch.from_numpy(q).to(DEV)
    if q_bf16:
        tq = tq.to(torch.bfloat16)
    out = torch.empty((S, H, 512), dtype=torch.bfloat16 if out_bf16 else torch.float32, device=DEV)
    lib.mla_q_absorb8(tq, tw8, tsc, out)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    ref = oracle.q_absorb(q, w8, sc)
    if out_bf16:
        # the f32 sum rounded once to bf16: within one bf16 half-step of the exact value (plus the f32 sum's error)
        bound = 2.0 ** -8 * np.abs(ref) + F32_TOL * np.abs(ref).max()
        assert np.all(np.abs(got - ref) <= bound), "bf16 q_lat outside one rounding of the oracle"
    else:
        _close(got, ref, F32_TOL, f"q_absorb S={S} H={H}")


@pytest.mark.parametrize("S,H", [(1, 128), (2, 128), (5, 3), (8, 128), (9, 128), (64, 128), (100, 9)])
def test_out_project_parity(lib, oracle, S, H):
    w8, sc, tw8, tsc = _weights(H, 12)
    x = synth.normal_f32(np.random.default_rng(S * 17 + H), (S, H, 512))
    out = torch.empty((S, H, 128), dtype=torch.float32, device=DEV)
    lib.mla_out_project8(torch.from_numpy(x).to(DEV), tw8, tsc, out)
    torch.cuda.synchronize()
    _close(out.cpu().numpy(), oracle.out_project(x, w8, sc), F32_TOL, f"out_project S={S} H={H}")


def test_projections_prefill_shape_sampled_rows(lib, oracle):
    """S = 1024 query rows of H = 128 heads (the prefill chunk): rows 0, 1, 63, 64, 511, 1023 checked."""
    S, H = 1024, 128
    w8, sc, tw8, tsc = _weights(H, 13)
    w = synth.WORKLOADS["prefill"]
    q = synth.q_nope_for(w)
    tq = torch.from_numpy(q).to(DEV).to(torch.bfloat16)
    q_lat = torch.empty((S, H, 512), dtype=torch.float32, device=DEV)
    lib.mla_q_absorb8(tq, tw8, tsc, q_lat)
    x = synth.normal_f32(np.random.default_rng(5), (S, H, 512))
    o = torch.empty((S, H, 128), dtype=torch.float32, device=DEV)
    lib.mla_out_project8(torch.from_numpy(x).to(DEV), tw8, tsc, o)
    torch.cuda.synchronize()
    rows = [0, 1, 63, 64, 511, 1023]
    _close(q_lat.cpu().numpy()[rows], oracle.q_absorb(q[rows], w8, sc), F32_TOL, "q_absorb prefill rows")
    _close(o.cpu().numpy()[rows], oracle.out_project(x[rows], w8, sc), F32_TOL, "out_project prefill rows")


def test_absorbed_layer_chain(lib, oracle):
    """q_nope -> q_lat (bf16) -> split-T decode over the 16k cache -> merge -> output projection, against
    the oracle's chain from the same q_lat values."""
    w = synth.WORKLOADS["dec16k"]
    H, T = w.H, w.T
    w8, sc, tw8, tsc = _weights(H, 14)
    rows = synth.rows_for(w)
    q_o, s_o = oracle_cache(oracle, rows)
    kv8, ks = torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)
    q_nope = synth.q_nope_for(w, 1)[0]
    _, q_rope = synth.queries_for(w, 1)
    q_lat = torch.empty((H, 512), dtype=torch.bfloat16, device=DEV)
    lib.mla_q_absorb8(torch.from_numpy(q_nope).to(DEV).to(torch.bfloat16), tw8, tsc, q_lat)
    ws = torch.empty(lib.mla_decode8_workspace_bytes(H, T) // 4, dtype=torch.float32, device=DEV)
    ctx = torch.empty((H, 512), dtype=torch.float32, device=DEV)
    lib.mla_absorb_decode8(q_lat, torch.from_numpy(q_rope[0]).to(DEV).to(torch.bfloat16), kv8, ks, T,
                           synth.SM_SCALE, ws, ctx)
    out = torch.empty((H, 128), dtype=torch.float32, device=DEV)
    lib.mla_out_project8(ctx, tw8, tsc, out)
    torch.cuda.synchronize()
    q_lat_v = q_lat.float().cpu().numpy()  # the bf16 query the decode saw (checked above against the oracle)
    heads = list(range(0, H, 7))
    ref_ctx = oracle.attn_decode(q_lat_v[heads], q_rope[0][heads], q_o, s_o, synth.SM_SCALE)
    parity(ctx.cpu().numpy()[heads], ref_ctx, "decode of the absorbed query")
    # output projection of the oracle's context for the sampled heads: a kv_b holding just those heads
    sel8 = w8.reshape(H, 256, 512)[heads].reshape(len(heads) * 256, 512)
    selsc = sc.reshape(H, 2, 4)[heads].reshape(len(heads) * 2, 4)
    ref_out = oracle.out_project(ref_ctx[None], sel8, selsc)[0]
    parity(out.cpu().numpy()[heads], ref_out, "output projection of the decoded context")
