"""The timeout path of the bounded waits, on the GPU: a wait that nothing completes gives up at its limit,
reports KV8_ERR_TIMEOUT through the caller's error word and returns; the context stays usable (a decode
right after it matches the oracle).  No fault, trap or hang is involved: the wait is the library's own
bounded mbarrier wait, run on a barrier that no thread or copy ever completes."""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_cache, parity

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")


def _timeout(lib, limit_ns):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.kv8_wait_selftest(limit_ns, err, st)
    torch.cuda.synchronize()
    return int(err.item()), int(st.item())


def test_bounded_wait_gives_up_and_reports(lib):
    err, st = _timeout(lib, 2_000_000)  # 2 ms
    assert err & lib.KV8_ERR_TIMEOUT
    assert st == 2


def test_limits_outside_the_documented_range_are_rejected(lib):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for bad in (10, 2_000_000_000):
        with pytest.raises(RuntimeError):
            lib.kv8_wait_selftest(bad, err, st)
    with pytest.raises(RuntimeError):
        lib.kv8_wait_selftest(1_000_000, None, st)


def test_context_usable_after_a_timeout(lib, oracle):
    _timeout(lib, 1_000_000)
    rng = np.random.default_rng(91)
    T, H = 700, 16
    rows = rng.standard_normal((T, 576)).astype(np.float32)
    q_o, s_o = oracle_cache(oracle, rows)
    q = synth.to_bf16_values(rng.standard_normal((H, 576)).astype(np.float32))
    ql, qr = np.ascontiguousarray(q[:, :512]), np.ascontiguousarray(q[:, 512:])
    ws = torch.empty(lib.mla_decode8_workspace_bytes(H, T, 0) // 4, dtype=torch.float32, device=DEV)
    out = torch.empty((H, 512), dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.mla_absorb_decode8(torch.from_numpy(ql).to(DEV).to(torch.bfloat16), torch.from_numpy(qr).to(DEV).to(torch.bfloat16),
                           torch.from_numpy(q_o).to(DEV), torch.from_numpy(s_o).to(DEV), T, synth.SM_SCALE, ws, out,
                           err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    parity(out.cpu().numpy(), oracle.attn_decode(ql, qr, q_o, s_o, synth.SM_SCALE), "decode after a timeout")
