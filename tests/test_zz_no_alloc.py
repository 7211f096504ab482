"""The no-allocation decode entry point against the workspace entry point.

Some callers cannot allocate device memory for the split-T workspace (a plugin inside a host program
whose memory pool owns the GPU, a caller from another language runtime without the host's allocator,
a loop that must not take cudaMalloc's implicit device synchronisation).  mla_absorb_decode8_noalloc
serves them: its partials live in a fixed device array inside the library.  Here two calls in a row,
on different caches and queries, each match mla_absorb_decode8 (with a caller-allocated workspace)
within the parity tolerance, and a request larger than the array is refused.

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
    return ql, qr, torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV)


def _with_workspace(lib, ql, qr, kv8, sc, T):
    H = ql.shape[0]
    ws = torch.empty(lib.mla_decode8_workspace_bytes(H, T) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty((H, 512), dtype=torch.float32, device=DEV)
    lib.mla_absorb_decode8(ql, qr, kv8, sc, T, synth.SM_SCALE, ws, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_noalloc_matches_workspace_entry_on_two_calls(lib, oracle):
    # first call: automatic partitions would need more than the fixed array, so fewer are used
    T1, H1 = 16384, 128
    a = _case(oracle, T1, H1, seed=1)
    out1 = torch.full((H1, 512), float("nan"), dtype=torch.float32, device=DEV)
    lib.mla_absorb_decode8_noalloc(*a, T1, synth.SM_SCALE, out1)
    # second call right after, on another cache and other queries
    T2, H2 = 3001, 64
    b = _case(oracle, T2, H2, seed=2)
    out2 = torch.full((H2, 512), float("nan"), dtype=torch.float32, device=DEV)
    lib.mla_absorb_decode8_noalloc(*b, T2, synth.SM_SCALE, out2)
    torch.cuda.synchronize()
    parity(out1.cpu().numpy(), _with_workspace(lib, *a, T1), "no-alloc call 1 vs workspace entry")
    parity(out2.cpu().numpy(), _with_workspace(lib, *b, T2), "no-alloc call 2 vs workspace entry")


def test_noalloc_refuses_requests_beyond_the_array(lib):
    H, T = 128, 262144
    need = lib.mla_decode8_workspace_bytes(H, T, 100)
    assert need > (16 << 20)
    ql = torch.zeros((H, 512), dtype=torch.bfloat16, device=DEV)
    qr = torch.zeros((H, 64), dtype=torch.bfloat16, device=DEV)
    kv8 = torch.zeros((T, 576), dtype=torch.uint8, device=DEV)
    sc = torch.zeros(T, dtype=torch.float32, device=DEV)
    out = torch.zeros((H, 512), dtype=torch.float32, device=DEV)
    with pytest.raises(lib.Kv8Error) as e:
        lib.mla_absorb_decode8_noalloc(ql, qr, kv8, sc, T, synth.SM_SCALE, out, P_req=100)
    assert e.value.code == lib.KV8_EWORKSPACE
