"""Shared helpers for the tests: parity check, cache building, workload fixtures."""
from __future__ import annotations

import os

import numpy as np

# Tolerance for attention outputs (the bar the method states): max|gpu - oracle| <= 1e-2 * max|oracle|
# and relative L2 <= 5e-3, over the compared outputs.
MAX_REL = 1e-2
L2_REL = 5e-3


def parity(got: np.ndarray, ref: np.ndarray, what: str = "") -> tuple[float, float]:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite GPU output"
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    nref = np.linalg.norm(ref)
    rel_l2 = np.linalg.norm(got - ref) / nref if nref > 0 else np.linalg.norm(got)
    assert err <= MAX_REL * scale + 1e-30, f"{what}: max|err| {err:.3e} > {MAX_REL} * {scale:.3e}"
    assert rel_l2 <= L2_REL, f"{what}: relative L2 {rel_l2:.3e} > {L2_REL}"
    return float(err / scale if scale > 0 else err), float(rel_l2)


def parity_per_head(got: np.ndarray, ref: np.ndarray, what: str = "", head_axis: int = -2) -> np.ndarray:
    """The attention bar applied to every head on its own (each head's error against that head's own
    largest output), on top of the aggregate check.  Returns [n_heads][2] (max-rel, relative L2).  With
    KV8_PARITY_REPORT set, appends a one-line summary per call to that file."""
    parity(got, ref, what)
    got = np.moveaxis(np.asarray(got, dtype=np.float64), head_axis, 0)
    ref = np.moveaxis(np.asarray(ref, dtype=np.float64), head_axis, 0)
    res = np.empty((got.shape[0], 2))
    for h in range(got.shape[0]):
        res[h] = parity(got[h], ref[h], f"{what} head {h}")
    path = os.environ.get("KV8_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(f"{what}: {got.shape[0]} heads x {got[0].size} outputs; per-head max-rel worst {res[:, 0].max():.2e} "
                    f"(head {int(res[:, 0].argmax())}), median {np.median(res[:, 0]):.2e}; per-head L2 worst "
                    f"{res[:, 1].max():.2e} (head {int(res[:, 1].argmax())}), median {np.median(res[:, 1]):.2e}\n")
    return res


def oracle_cache(oracle, rows: np.ndarray, chunk: int = 65536):
    """Quantize f32 rows with the oracle, in chunks: (bytes [n][576] u8, scales [n] f32)."""
    n = rows.shape[0]
    q = np.empty((n, 576), dtype=np.uint8)
    s = np.empty(n, dtype=np.float32)
    for i in range(0, n, chunk):
        q[i:i + chunk], s[i:i + chunk] = oracle.quant_rows(rows[i:i + chunk])
    return q, s
