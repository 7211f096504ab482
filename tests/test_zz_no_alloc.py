"""The no-allocation decode entry point against the oracle and against the workspace entry point.

Some callers cannot allocate device memory for the split-T workspace (a plugin inside a host program
whose memory pool owns the GPU, a caller from another language runtime without the host's allocator,
a loop that must not take cudaMalloc's implicit device synchronisation).  mla_absorb_decode8_noalloc
serves them: its partials live in a fixed device array inside the library.  Here two calls in a row,
on different caches and queries, each match the oracle and mla_absorb_decode8 (with a caller-allocated
workspace) within the parity tolerance; an explicit partition count that fits is used as given; a
request larger than the array and bad sizes are refused before anything is enqueued.

This file is collected last, so a failure here comes after every other test has run.
"""
import numpy as np
import pytest
import torch

import synth
from helpers import parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _case(oracle, T, H, seed):
    rng = np.random.default_rng(seed)
    rows = synth.latent_rows(rng, T, 0.1, 10.0)
    q_o, s_o = oracle.quant_rows(rows)
    q = synth.to_bf16_values(synth.normal_f32(rng, (H, 576)))
    ql = torch.from_numpy(np.ascontiguousarray(q[:, :512])).to(DEV).to(torch.bfloat16)
    qr = torch.from_numpy(np.ascontiguousarray(q[:, 512:])).to(DEV).to(torch.bfloat16)
    ref = oracle.attn_decode(np.ascontiguousarray(q[:, :512]), np.ascontiguousarray(q[:, 512:]), q_o, s_o,
                             synth.SM_SCALE)
    return (ql, qr, torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)), ref


def _with_workspace(lib, ql, qr, kv8, sc, T, P_req=0):
    H = ql.shape[0]
    ws = torch.empty(lib.mla_decode8_workspace_bytes(H, T, P_req) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty((H, 512), dtype=torch.float32, device=DEV)
    lib.mla_absorb_decode8(ql, qr, kv8, sc, T, synth.SM_SCALE, ws, out, P_req=P_req)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_noalloc_matches_oracle_and_workspace_entry_on_two_calls(lib, oracle):
    # first call: automatic partitions would need more than the fixed array, so fewer are used
    T1, H1 = 16384, 128
    a, ref1 = _case(oracle, T1, H1, seed=1)
    out1 = torch.full((H1, 512), float("nan"), dtype=torch.float32, device=DEV)
    lib.mla_absorb_decode8_noalloc(*a, T1, synth.SM_SCALE, out1)
    # second call right after, on another cache and other queries
    T2, H2 = 3001, 64
    b, ref2 = _case(oracle, T2, H2, seed=2)
    out2 = torch.full((H2, 512), float("nan"), dtype=torch.float32, device=DEV)
    lib.mla_absorb_decode8_noalloc(*b, T2, synth.SM_SCALE, out2)
    torch.cuda.synchronize()
    got1, got2 = out1.cpu().numpy(), out2.cpu().numpy()
    parity(got1, ref1, "no-alloc call 1 vs oracle")
    parity(got2, ref2, "no-alloc call 2 vs oracle")
    parity(got1, _with_workspace(lib, *a, T1), "no-alloc call 1 vs workspace entry")
    parity(got2, _with_workspace(lib, *b, T2), "no-alloc call 2 vs workspace entry")


def test_noalloc_explicit_partition_count_that_fits(lib, oracle):
    T, H, P = 3001, 64, 8
    a, ref = _case(oracle, T, H, seed=3)
    out = torch.full((H, 512), float("nan"), dtype=torch.float32, device=DEV)
    for _ in range(2):  # twice: the array keeps the previous call's partials, which must not leak in
        lib.mla_absorb_decode8_noalloc(*a, T, synth.SM_SCALE, out, P_req=P)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        parity(got, ref, "no-alloc P_req=8 vs oracle")
        assert np.array_equal(got, _with_workspace(lib, *a, T, P_req=P)), "same partitions, same kernels: identical"


def test_noalloc_refuses_requests_beyond_the_array_and_bad_sizes(lib):
    H, T = 128, 262144
    need = lib.mla_decode8_workspace_bytes(H, T, 100)
    assert need > (16 << 20)
    # validation happens before any launch: small placeholder tensors are never read
    ql = torch.zeros((H, 512), dtype=torch.bfloat16, device=DEV)
    qr = torch.zeros((H, 64), dtype=torch.bfloat16, device=DEV)
    kv8 = torch.zeros((16, 576), dtype=torch.uint8, device=DEV)
    sc = torch.zeros(16, dtype=torch.float32, device=DEV)
    out = torch.zeros((H, 512), dtype=torch.float32, device=DEV)
    with pytest.raises(lib.Kv8Error) as e:
        lib.mla_absorb_decode8_noalloc(ql, qr, kv8, sc, T, synth.SM_SCALE, out, P_req=100)
    assert e.value.code == lib.KV8_EWORKSPACE
    for bad_T in (0, (1 << 20) + 1):
        with pytest.raises(lib.Kv8Error) as e:
            lib.mla_absorb_decode8_noalloc(ql, qr, kv8, sc, bad_T, synth.SM_SCALE, out)
        assert e.value.code == lib.KV8_EINVAL
    with pytest.raises(lib.Kv8Error) as e:
        lib.mla_absorb_decode8_noalloc(torch.zeros((129, 512), dtype=torch.bfloat16, device=DEV),
                                       torch.zeros((129, 64), dtype=torch.bfloat16, device=DEV), kv8, sc, 16,
                                       synth.SM_SCALE, out)
    assert e.value.code == lib.KV8_EINVAL
