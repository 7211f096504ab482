"""GPU quantizer and encoder vs the oracle: bit-exact bytes and scales.

- kv8_encode_e4m3 over all 2^32 f32 bit patterns: the GPU's change points (patterns where the code
  differs from the previous pattern's) must be exactly the oracle's list, with equal codes on both
  sides of each; between change points both are constant, so they agree on every pattern.
- kv8_quant_rows on every row of every workload, and on edge rows (zero, signed zero, subnormal
  amax, NaN/inf elements, huge and tiny amax), including a fresh row appended at an offset.
"""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_cache

pytestmark = pytest.mark.gpu


def test_encoder_all_f32_patterns(lib, oracle):
    expected = oracle.encode_change_points().astype(np.int64)
    dev = torch.device("cuda")
    chunk = 1 << 28
    out = torch.empty(chunk, dtype=torch.uint8, device=dev)
    found, codes_at, codes_before = [], [], []
    prev_last = None
    first_code = None
    for c in range(16):
        base = c * chunk
        start = base - (1 << 32) if base >= (1 << 31) else base
        bits = torch.arange(start, start + chunk, dtype=torch.int32, device=dev)
        lib.kv8_encode_e4m3(bits.view(torch.float32), out)
        if c == 0:
            first_code = int(out[0].item())
        d = torch.nonzero(out[1:] != out[:-1]).flatten() + 1
        pos = d.cpu().numpy().astype(np.int64)
        if prev_last is not None and int(out[0].item()) != prev_last:
            found.append(base)
            codes_at.append(int(out[0].item()))
            codes_before.append(prev_last)
        if pos.size:
            at = out[d].cpu().numpy()
            before = out[d - 1].cpu().numpy()
            found.extend((base + pos).tolist())
            codes_at.extend(at.tolist())
            codes_before.extend(before.tolist())
        prev_last = int(out[-1].item())
        del bits
    torch.cuda.synchronize()
    assert first_code == oracle.e4m3_encode(0.0) == 0
    assert np.array_equal(np.array(found, dtype=np.int64), expected), (len(found), len(expected))

    def enc_bits(p):
        return oracle.e4m3_encode(np.array([p & 0xFFFFFFFF], dtype=np.uint32).view(np.float32)[0])

    for p, a, b in zip(found, codes_at, codes_before):
        assert a == enc_bits(p) and b == enc_bits(p - 1), hex(p)


def _gpu_quant(lib, rows: np.ndarray):
    dev = torch.device("cuda")
    x = torch.from_numpy(np.ascontiguousarray(rows)).to(dev)
    q = torch.empty((rows.shape[0], 576), dtype=torch.uint8, device=dev)
    s = torch.empty(rows.shape[0], dtype=torch.float32, device=dev)
    lib.kv8_quant_rows(x, q, s)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("key", ["tiny", "dec16k", "dec262k", "dsa", "prefill"])
def test_quant_rows_every_row_of_every_workload(lib, oracle, key):
    w = synth.WORKLOADS[key]
    chunk = 65536
    for seq in range(w.B):
        for start in range(0, w.T, chunk):
            rows = synth.rows_for(w, seq, start, min(chunk, w.T - start))
            qg, sg = _gpu_quant(lib, rows)
            qo, so = oracle_cache(oracle, rows)
            assert np.array_equal(sg.view(np.uint32), so.view(np.uint32)), (key, seq, start)
            bad = np.nonzero(np.any(qg != qo, axis=1))[0]
            assert bad.size == 0, (key, seq, start + int(bad[0]) if bad.size else None)


def _edge_rows():
    rng = np.random.default_rng(99)
    rows = []
    z = np.zeros(576, np.float32)
    rows.append(z.copy())                                     # all +0
    r = z.copy(); r[::3] = -0.0; rows.append(r)               # signed zeros
    rows.append((rng.standard_normal(576) * 1e-39).astype(np.float32))   # subnormal amax
    rows.append((rng.standard_normal(576) * 1e-44).astype(np.float32))   # amax a few subnormal ulps
    r = np.zeros(576, np.float32); r[7] = np.float32(1.4e-45); rows.append(r)  # one smallest subnormal
    r = (rng.standard_normal(576) * 1e-37).astype(np.float32); rows.append(r)  # amax just under 448/FLT_MAX
    r = (rng.standard_normal(576) * 3e37).astype(np.float32); rows.append(r)   # huge amax
    r = rng.standard_normal(576).astype(np.float32); r[5] = np.nan; r[9] = -np.nan; rows.append(r)
    r = rng.standard_normal(576).astype(np.float32); r[1] = np.inf; r[2] = -np.inf; rows.append(r)
    r = np.zeros(576, np.float32); r[3] = np.inf; r[4] = -0.0; r[5] = np.nan; rows.append(r)  # amax 0, inf
    r = np.full(576, np.nan, np.float32); rows.append(r)      # all NaN
    r = rng.standard_normal(576).astype(np.float32); r[100] = 448.0; r[200] = -448.0; rows.append(r)
    r = (rng.standard_normal(576) * 10.0 ** rng.uniform(-8, 8, 576)).astype(np.float32); rows.append(r)  # wide range
    r = np.full(576, np.float32(3.4028235e38)); r[::2] *= -1; rows.append(r)  # FLT_MAX
    return np.stack(rows)


def test_quant_rows_edge_rows(lib, oracle):
    rows = _edge_rows()
    qg, sg = _gpu_quant(lib, rows)
    qo, so = oracle.quant_rows(rows)
    assert np.array_equal(sg.view(np.uint32), so.view(np.uint32))
    assert np.array_equal(qg, qo)


def test_quant_rows_append_at_offset_and_empty(lib, oracle):
    dev = torch.device("cuda")
    T = 37
    rows = synth.latent_rows(np.random.default_rng(5), T, 0.1, 10.0)
    kv8 = torch.full((T, 576), 0xAB, dtype=torch.uint8, device=dev)
    sc = torch.full((T,), -1.0, dtype=torch.float32, device=dev)
    x = torch.from_numpy(rows).to(dev)
    lib.kv8_quant_rows(x[:T - 1], kv8, sc)
    lib.kv8_quant_rows(x[T - 1:], kv8[T - 1:], sc[T - 1:])   # the fresh row of a decode step
    lib.kv8_quant_rows(x[:0], kv8, sc, n=0)                   # nothing to do
    torch.cuda.synchronize()
    qo, so = oracle.quant_rows(rows)
    assert np.array_equal(kv8.cpu().numpy(), qo)
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), so.view(np.uint32))


def test_encoder_ragged_lengths(lib, oracle):
    dev = torch.device("cuda")
    rng = np.random.default_rng(6)
    for n in [1, 2, 3, 5, 1023, 4097]:
        y = (rng.standard_normal(n) * 100).astype(np.float32)
        out = torch.full((n + 8,), 0xCD, dtype=torch.uint8, device=dev)
        lib.kv8_encode_e4m3(torch.from_numpy(y).to(dev), out[:n])
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert np.array_equal(got[:n], oracle.encode_array(y))
        assert np.all(got[n:] == 0xCD)  # nothing written past n
