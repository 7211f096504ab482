"""The C ABI library loads and exports every symbol include/kv8mla.h declares; host-side argument
validation rejects bad arguments before any launch.  CPU only (no CUDA call is made)."""
import ctypes
import os
import re

import pytest

import fp8_latent_kv_gb300 as kv
from fp8_latent_kv_gb300 import build as kvbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kv8mla.h")


@pytest.fixture(scope="module")
def lib():
    kvbuild.build()
    return kv.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"^KV8_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["kv8_quant_rows", "mla_absorb_decode8", "mla_absorb_sel8", "mla_absorb_prefill8", "mla_lse_merge8",
              "mla_decode8_partial", "kv8_encode_e4m3", "kv8_strerror"]:
        assert n in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) == set(kv.SIGNATURES)


def test_strerror(lib):
    for code in [kv.KV8_OK, kv.KV8_EINVAL, kv.KV8_EWORKSPACE, kv.KV8_ECUDA, kv.KV8_EUNSUPPORTED]:
        assert len(kv.kv8_strerror(code)) > 0
    assert "unknown" in kv.kv8_strerror(-99)


def test_partitions_and_workspace_sizes(lib):
    assert kv.mla_decode8_partitions(128, 262144) == 76
    assert kv.mla_decode8_partitions(16, 256) == 2
    assert kv.mla_decode8_partitions(64, 262144) == 152   # one 64-head half: a CTA per partition
    assert kv.mla_decode8_partitions(65, 262144) == 76
    assert kv.mla_decode8_partitions(128, 1) == 1
    assert kv.mla_decode8_partitions(128, 5, P_req=9) == 5
    assert kv.mla_decode8_partitions(128, 1000, P_req=7) == 7
    P = kv.mla_decode8_partitions(128, 262144)
    ws = kv.mla_decode8_workspace_bytes(128, 262144)
    assert ws >= P * 128 * 514 * 4                      # the partial sets come first
    assert ws - P * 128 * 514 * 4 < 256 * 1024          # plus a small staging area
    # selection: 8 items x 2 head halves leave 9 CTAs per item -> 16 tiles as 8 partitions of 2;
    # partial sets, then 2 query images + 128 head factors per item and the row-scale maxima
    assert kv.mla_sel8_workspace_bytes(8, 128, 2048) == 8 * 8 * 128 * 514 * 4 + 8 * (2 * 73728 + 512) + 256
    # one item, 64 heads: up to 152 partitions of one tile
    assert kv.mla_sel8_workspace_bytes(1, 64, 4096) == 1 * 32 * 64 * 514 * 4 + (2 * 73728 + 512) + 256


def _rc(fn, *args):
    return fn(*args)


def test_validation_rejects_before_launch(lib):
    fake = 0x100000  # 16-byte aligned, never dereferenced: validation fails first
    mis = fake + 4
    EINVAL, EWS = kv.KV8_EINVAL, kv.KV8_EWORKSPACE
    sz = ctypes.c_size_t(0)
    # sizes
    assert lib.mla_decode8_workspace_bytes(0, 10, 0, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_decode8_workspace_bytes(129, 10, 0, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_decode8_workspace_bytes(16, 0, 0, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_decode8_workspace_bytes(16, (1 << 20) + 1, 0, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_decode8_workspace_bytes(16, 10, -1, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_sel8_workspace_bytes(1, 16, 0, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_sel8_workspace_bytes(1, 16, 4097, ctypes.addressof(sz)) == EINVAL
    # decode: null / misaligned / bad dtype / workspace
    args = dict(q_lat=fake, q_rope=fake, dt=kv.KV8_BF16, H=16, kv8=fake, sc=fake, T=100, sm=0.07, P=0, ws=fake,
                ws_bytes=1 << 30, err=None, out=fake, st=None)

    def dec(**kw):
        a = dict(args, **kw)
        return lib.mla_absorb_decode8(a["q_lat"], a["q_rope"], a["dt"], a["H"], a["kv8"], a["sc"], a["T"], a["sm"],
                                      a["P"], a["ws"], a["ws_bytes"], a["err"], a["out"], a["st"])

    assert dec(q_lat=None) == EINVAL
    assert dec(q_rope=mis) == EINVAL
    assert dec(kv8=mis) == EINVAL
    assert dec(dt=7) == EINVAL
    assert dec(H=0) == EINVAL
    assert dec(T=0) == EINVAL
    assert dec(sm=float("nan")) == EINVAL
    assert dec(sm=float("inf")) == EINVAL
    assert dec(out=mis) == EINVAL
    assert dec(ws_bytes=16) == EWS
    # selection
    assert lib.mla_absorb_sel8(fake, fake, kv.KV8_BF16, 2, 16, fake, fake, 100, 50, fake, 10, 0.07, fake, 1 << 30,
                               None, fake, None) == EINVAL  # seq_stride_rows < T
    assert lib.mla_absorb_sel8(fake, fake, kv.KV8_BF16, 2, 16, fake, fake, 100, 100, fake, 4097, 0.07, fake, 1 << 30,
                               None, fake, None) == EINVAL  # NS > 4096
    assert lib.mla_absorb_sel8(fake, fake, kv.KV8_BF16, 2, 16, fake, fake, 100, 100, fake, 10, 0.07, fake, 8, None,
                               fake, None) == EWS
    # prefill
    assert lib.mla_absorb_prefill8(fake, fake, kv.KV8_BF16, 8, 16, 95, fake, fake, 100, 0.07, None, fake,
                                   None) == EINVAL  # pos0 + S > T
    assert lib.mla_absorb_prefill8(fake, fake, kv.KV8_BF16, 0, 16, 0, fake, fake, 100, 0.07, None, fake,
                                   None) == EINVAL
    assert lib.mla_absorb_prefill8(fake, fake, kv.KV8_BF16, 4, 16, -1, fake, fake, 100, 0.07, None, fake,
                                   None) == EINVAL
    # quantizer / encoder
    assert lib.kv8_quant_rows(fake, -1, fake, fake, None) == EINVAL
    assert lib.kv8_quant_rows(mis, 3, fake, fake, None) == EINVAL
    assert lib.kv8_quant_rows(None, 0, None, None, None) == kv.KV8_OK  # nothing to do
    assert lib.kv8_encode_e4m3(mis, 5, fake, None) == EINVAL
    assert lib.mla_lse_merge8(fake, 1, 0, 16, fake, None) == EINVAL
