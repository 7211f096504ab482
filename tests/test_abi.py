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


def test_validation_of_the_later_calls(lib):
    """Batched, mixed-cache, projection, indexer, scatter and copy calls reject bad scalars, alignment and
    workspace before any CUDA call."""
    fake = 0x100000
    mis4, mis2 = fake + 4, fake + 2  # 4-byte but not 8/16-byte aligned; 2-byte aligned
    EINVAL, EWS, OK = kv.KV8_EINVAL, kv.KV8_EWORKSPACE, kv.KV8_OK
    BF, F32 = kv.KV8_BF16, kv.KV8_F32
    sz = ctypes.c_size_t(0)
    # quantizers
    assert lib.kv8_quant_rows_w(fake, 3, 100, fake, fake, None) == EINVAL      # unsupported width
    assert lib.kv8_quant_rows_w(fake, -1, 128, fake, fake, None) == EINVAL
    assert lib.kv8_quant_rows_w(None, 0, 448, None, None, None) == OK         # nothing to do
    assert lib.kv8_quant_rows_w(mis4, 3, 128, fake, fake, None) == EINVAL
    assert lib.kv8_quant_rows_scatter(fake, -1, fake, fake, fake, 10, None, None) == EINVAL
    assert lib.kv8_quant_rows_scatter(fake, 2, fake, fake, fake, -1, None, None) == EINVAL
    assert lib.kv8_quant_rows_scatter(None, 0, None, None, None, 10, None, None) == OK
    assert lib.kv8_quant_rows_scatter(fake, 2, mis4, fake, fake, 10, None, None) == EINVAL  # int64 rows need 8 B
    # batched decode
    assert lib.mla_batch_decode8_workspace_bytes(0, 16, 100, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_batch_decode8_workspace_bytes(2, 129, 100, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_batch_decode8_workspace_bytes(2, 16, 0, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_batch_decode8_workspace_bytes(2, 16, 100, None) == EINVAL

    def bat(**kw):
        a = dict(ql=fake, qr=fake, dt=BF, B=2, H=16, kv8=fake, sc=fake, T=100, stride=100, lens=fake, sm=0.07,
                 ws=fake, wsb=1 << 30, err=None, out=fake)
        a.update(kw)
        return lib.mla_absorb_batch_decode8(a["ql"], a["qr"], a["dt"], a["B"], a["H"], a["kv8"], a["sc"], a["T"],
                                            a["stride"], a["lens"], a["sm"], a["ws"], a["wsb"], a["err"], a["out"],
                                            None)
    assert bat(stride=99) == EINVAL       # caches of two sequences would overlap
    assert bat(lens=mis2) == EINVAL
    assert bat(dt=7) == EINVAL
    assert bat(sm=float("nan")) == EINVAL
    assert bat(wsb=64) == EWS
    # mixed-precision cache
    assert lib.mla_mixed_decode8_workspace_bytes(0, 100, ctypes.addressof(sz)) == EINVAL
    assert lib.mla_mixed_decode8_workspace_bytes(16, 0, ctypes.addressof(sz)) == EINVAL

    def mix(**kw):
        a = dict(qn=fake, qr=fake, dt=BF, H=16, k8=fake, ks=fake, kr=fake, T=100, sm=0.07, ws=fake, wsb=1 << 30,
                 err=None, out=fake)
        a.update(kw)
        return lib.mla_absorb_mixed_decode8(a["qn"], a["qr"], a["dt"], a["H"], a["k8"], a["ks"], a["kr"], a["T"],
                                            a["sm"], a["ws"], a["wsb"], a["err"], a["out"], None)
    assert mix(k8=mis4) == EINVAL
    assert mix(kr=mis4) == EINVAL
    assert mix(H=129) == EINVAL
    assert mix(sm=float("inf")) == EINVAL
    assert mix(wsb=64) == EWS
    # absorb projections
    assert lib.mla_q_absorb8(fake, BF, 0, 16, fake, fake, fake, BF, None, None) == EINVAL
    assert lib.mla_q_absorb8(fake, BF, 4, 129, fake, fake, fake, BF, None, None) == EINVAL
    assert lib.mla_q_absorb8(fake, BF, 4, 16, fake, fake, fake, 7, None, None) == EINVAL
    assert lib.mla_q_absorb8(fake, BF, 4, 16, fake, fake, mis4, F32, None, None) == EINVAL
    assert lib.mla_out_project8(fake, 0, 16, fake, fake, fake, None, None) == EINVAL
    assert lib.mla_out_project8(fake, 4, 16, fake, fake, mis4, None, None) == EINVAL
    # DSA indexer
    assert lib.dsa_index_workspace_bytes(0, ctypes.addressof(sz)) == EINVAL

    def idx(**kw):
        a = dict(q=fake, dt=BF, w=fake, B=2, HI=64, k8=fake, ks=fake, T=1000, stride=1000, NS=64, ws=fake,
                 wsb=1 << 30, sc=fake, idx=fake)
        a.update(kw)
        return lib.dsa_index_topk8(a["q"], a["dt"], a["w"], a["B"], a["HI"], a["k8"], a["ks"], a["T"], a["stride"],
                                   a["NS"], a["ws"], a["wsb"], a["sc"], a["idx"], None, None)
    assert idx(HI=8) == EINVAL            # fewer than 16 heads
    assert idx(HI=40) == EINVAL           # not a multiple of 16
    assert idx(NS=0) == EINVAL
    assert idx(NS=4097) == EINVAL
    assert idx(T=0) == EINVAL
    assert idx(dt=7) == EINVAL
    assert idx(k8=mis4) == EINVAL
    assert idx(wsb=64) == EWS
    # copies: nothing to copy, a null pointer, overlapping ranges
    assert lib.kv8_copy(None, None, 0, None) == OK
    assert lib.kv8_copy(None, fake, 16, None) == EINVAL
    assert lib.kv8_copy(fake, fake + 8, 16, None) == EINVAL
