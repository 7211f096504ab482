"""kv8_copy: kernel copies between device memory and page-locked host memory, any size and alignment,
nothing written outside the range; pageable host memory and overlapping ranges are refused on the
host before anything is enqueued."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda")

SIZES = [1, 15, 16, 17, 4096, 150003, 1 << 22]


@pytest.mark.parametrize("kind", ["h2d", "d2h", "d2d"])
@pytest.mark.parametrize("off", [0, 3, 16])
def test_copy_bytes_exact(lib, kind, off):
    rng = np.random.default_rng(7 + off)
    for n in SIZES:
        data = rng.integers(1, 256, n + 32, dtype=np.uint8)
        src_h = torch.from_numpy(data).pin_memory()
        if kind == "h2d":
            src, dst = src_h, torch.zeros(n + 32, dtype=torch.uint8, device=DEV)
        elif kind == "d2h":
            src, dst = src_h.to(DEV), torch.zeros(n + 32, dtype=torch.uint8).pin_memory()
        else:
            src, dst = src_h.to(DEV), torch.zeros(n + 32, dtype=torch.uint8, device=DEV)
        lib.kv8_copy(dst[off:], src[off:], n)
        torch.cuda.synchronize()
        got = dst.cpu().numpy()
        assert np.array_equal(got[off:off + n], data[off:off + n]), f"{kind} n={n} off={off}"
        assert not got[:off].any() and not got[off + n:].any(), "bytes written outside the range"


def test_copy_typed_views_round_trip(lib):
    """The way a step uses it: f32 and bf16 views of one pinned buffer in, an f32 result out."""
    x = torch.randn(128, 512)
    h = x.pin_memory()
    d = torch.empty_like(x, device=DEV)
    lib.kv8_copy(d, h)
    back = torch.empty_like(x).pin_memory()
    lib.kv8_copy(back, d)
    torch.cuda.synchronize()
    assert torch.equal(back, x)
    hb = x.to(torch.bfloat16).pin_memory()
    db = torch.empty_like(hb, device=DEV)
    lib.kv8_copy(db, hb)
    torch.cuda.synchronize()
    assert torch.equal(db.cpu(), hb)


def test_copy_refuses_pageable_overlap_and_null(lib):
    import fp8_latent_kv_gb300 as kv
    d = torch.zeros(64, dtype=torch.uint8, device=DEV)
    pageable = torch.zeros(64, dtype=torch.uint8)  # ordinary (not page-locked) host memory
    assert not pageable.is_pinned()
    for dst, src, n in ((d, pageable, 64), (pageable, d, 64), (d[8:], d, 32), (d, d[8:], 32)):
        with pytest.raises(kv.Kv8Error) as e:
            lib.kv8_copy(dst, src, n)
        assert e.value.code == -1
    with pytest.raises(kv.Kv8Error):
        lib.kv8_copy(0, d, 16)
    lib.kv8_copy(d, d, 0)  # zero bytes: nothing to do, nothing checked
    torch.cuda.synchronize()
    assert not d.cpu().numpy().any()
