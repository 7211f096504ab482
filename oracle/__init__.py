"""Oracle: a plain, slow CPU reference of fp8 latent-KV absorbed MLA attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs may import this package.  The product library never does, and the
two share no code.  The arithmetic lives in ``kv8_oracle.c`` (double accumulation, f32 quantizer);
this module compiles it with gcc and marshals numpy arrays through ctypes.

Sources: the web page "KV8 long-context CUDA: fp8 device shadow, split-T kernels, DSA-aware gather"
(colibri pull request #300), first commit message (fp8 row format, codec, absorb loops) and second
commit message (split-T partials + log-sum-exp merge, DSA gather).

Parity pins: every function here is checked by ``tests/test_oracle_pins.py`` against closed forms,
invariants, brute force and an independent library routine (torch's float8_e4m3fn conversion).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kv8_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

D, KL, KR = 576, 512, 64


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (gcc, IEEE arithmetic, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        sig = {
            "kv8o_e4m3_decode": (ctypes.c_double, [ctypes.c_uint8]),
            "kv8o_e4m3_encode": (ctypes.c_uint8, [f32]),
            "kv8o_e4m3_encode_scan": (ctypes.c_uint8, [f32]),
            "kv8o_e4m3_table": (None, [P]),
            "kv8o_encode_array": (None, [P, i64, P]),
            "kv8o_encode_change_points": (i64, [P, i64]),
            "kv8o_quant_rows": (None, [P, i64, P, P]),
            "kv8o_dequant_rows": (None, [P, P, i64, P]),
            "kv8o_attn_decode": (None, [P, P, i32, P, P, i64, f32, P]),
            "kv8o_attn_decode_split": (None, [P, P, i32, P, P, i64, f32, i32, P, P, P, P]),
            "kv8o_attn_select": (None, [P, P, i32, i32, P, P, i64, i64, P, i32, f32, P, P]),
            "kv8o_attn_prefill": (None, [P, P, i32, i32, P, P, P, i64, f32, P]),
            "kv8o_q_absorb": (None, [P, i32, i32, P, P, P]),
            "kv8o_quant_rows_w": (None, [P, i64, i32, P, P]),
            "kv8o_attn_mixed_decode": (None, [P, P, P, i32, P, P, P, i64, f32, P]),
            "kv8o_index_scores": (None, [P, P, P, i32, i32, i32, P, P, i64, i64, P]),
            "kv8o_topk": (None, [P, i64, i32, P]),
            "kv8o_out_project": (None, [P, i32, i32, P, P, P]),
            "kv8o_num_threads": (i32, []),
            "kv8o_set_num_threads": (None, [i32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


# --------------------------------------------------------------------------------------------------
# e4m3 codec
# --------------------------------------------------------------------------------------------------
def e4m3_decode(b: int) -> float:
    return _load().kv8o_e4m3_decode(int(b) & 0xFF)


def e4m3_table() -> np.ndarray:
    out = np.zeros(256, dtype=np.float64)
    _load().kv8o_e4m3_table(_ptr(out))
    return out


def e4m3_encode(y: float) -> int:
    return int(_load().kv8o_e4m3_encode(float(np.float32(y))))


def e4m3_encode_scan(y: float) -> int:
    return int(_load().kv8o_e4m3_encode_scan(float(np.float32(y))))


def encode_array(y) -> np.ndarray:
    y = _f32(y).reshape(-1)
    out = np.empty(y.size, dtype=np.uint8)
    _load().kv8o_encode_array(_ptr(y), y.size, _ptr(out))
    return out


def encode_change_points() -> np.ndarray:
    cap = 1024
    out = np.zeros(cap, dtype=np.uint32)
    n = _load().kv8o_encode_change_points(_ptr(out), cap)
    assert 0 <= n <= cap
    return out[:n].copy()


def quant_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Rows x [n][576] f32 -> (bytes [n][576] u8, scale [n] f32)."""
    x = _f32(x).reshape(-1, D)
    n = x.shape[0]
    q = np.empty((n, D), dtype=np.uint8)
    s = np.empty(n, dtype=np.float32)
    _load().kv8o_quant_rows(_ptr(x), n, _ptr(q), _ptr(s))
    return q, s


def quant_rows_w(x, width: int) -> tuple[np.ndarray, np.ndarray]:
    """Rows of any width [n][width] f32 -> (bytes [n][width] u8, scale [n] f32): the row quantizer above."""
    x = _f32(x).reshape(-1, width)
    n = x.shape[0]
    q = np.empty((n, width), dtype=np.uint8)
    s = np.empty(n, dtype=np.float32)
    _load().kv8o_quant_rows_w(_ptr(x), n, int(width), _ptr(q), _ptr(s))
    return q, s


def dequant_rows(q, s) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8).reshape(-1, D)
    s = _f32(s).reshape(-1)
    out = np.empty((q.shape[0], D), dtype=np.float64)
    _load().kv8o_dequant_rows(_ptr(q), _ptr(s), q.shape[0], _ptr(out))
    return out


# --------------------------------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------------------------------
def _split_q(q_lat, q_rope, lead):
    ql = _f32(q_lat).reshape(*lead, KL)
    qr = _f32(q_rope).reshape(*lead, KR)
    return ql, qr


def attn_decode(q_lat, q_rope, kv8, scale, sm_scale) -> np.ndarray:
    """One query, H heads over all rows of kv8 [T][576]; returns [H][512] f32."""
    H = int(np.asarray(q_lat).size // KL)
    ql, qr = _split_q(q_lat, q_rope, (H,))
    kv8 = np.ascontiguousarray(kv8, dtype=np.uint8).reshape(-1, D)
    scale = _f32(scale).reshape(-1)
    T = kv8.shape[0]
    assert scale.size == T
    out = np.empty((H, KL), dtype=np.float32)
    _load().kv8o_attn_decode(_ptr(ql), _ptr(qr), H, _ptr(kv8), _ptr(scale), T, float(np.float32(sm_scale)),
                             _ptr(out))
    return out


def attn_decode_split(q_lat, q_rope, kv8, scale, sm_scale, P: int):
    """Split-T form: returns (out [H][512] f32, cl_part [P][H][512], m_part [P][H], z_part [P][H])."""
    H = int(np.asarray(q_lat).size // KL)
    ql, qr = _split_q(q_lat, q_rope, (H,))
    kv8 = np.ascontiguousarray(kv8, dtype=np.uint8).reshape(-1, D)
    scale = _f32(scale).reshape(-1)
    T = kv8.shape[0]
    cl = np.zeros((P, H, KL), dtype=np.float64)
    m = np.zeros((P, H), dtype=np.float64)
    z = np.zeros((P, H), dtype=np.float64)
    out = np.empty((H, KL), dtype=np.float32)
    _load().kv8o_attn_decode_split(_ptr(ql), _ptr(qr), H, _ptr(kv8), _ptr(scale), T, float(np.float32(sm_scale)),
                                   int(P), _ptr(cl), _ptr(m), _ptr(z), _ptr(out))
    return out, cl, m, z


def attn_select(q_lat, q_rope, kv8, scale, T: int, seq_stride_rows: int, idx, sm_scale):
    """B sequences with their own T-row caches; idx [B][NS] int32.  Returns (out [B][H][512], n_bad)."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    B, NS = idx.shape
    H = int(np.asarray(q_lat).size // (B * KL))
    ql, qr = _split_q(q_lat, q_rope, (B, H))
    kv8 = np.ascontiguousarray(kv8, dtype=np.uint8).reshape(-1, D)
    scale = _f32(scale).reshape(-1)
    assert kv8.shape[0] >= (B - 1) * seq_stride_rows + T
    out = np.empty((B, H, KL), dtype=np.float32)
    bad = np.zeros(1, dtype=np.int64)
    _load().kv8o_attn_select(_ptr(ql), _ptr(qr), B, H, _ptr(kv8), _ptr(scale), int(T), int(seq_stride_rows),
                             _ptr(idx), NS, float(np.float32(sm_scale)), _ptr(out), _ptr(bad))
    return out, int(bad[0])


def attn_prefill(q_lat, q_rope, pos, kv8, scale, sm_scale) -> np.ndarray:
    """nq queries at absolute positions pos [nq]; q [nq][H][...]; returns [nq][H][512] f32."""
    pos = np.ascontiguousarray(pos, dtype=np.int64).reshape(-1)
    nq = pos.size
    H = int(np.asarray(q_lat).size // (nq * KL))
    ql, qr = _split_q(q_lat, q_rope, (nq, H))
    kv8 = np.ascontiguousarray(kv8, dtype=np.uint8).reshape(-1, D)
    scale = _f32(scale).reshape(-1)
    T = kv8.shape[0]
    out = np.empty((nq, H, KL), dtype=np.float32)
    _load().kv8o_attn_prefill(_ptr(ql), _ptr(qr), nq, H, _ptr(pos), _ptr(kv8), _ptr(scale), T,
                              float(np.float32(sm_scale)), _ptr(out))
    return out


NOPE, VH, BLK = 128, 128, 128


def _kvb(w8, w_scale, H):
    w8 = np.ascontiguousarray(w8, dtype=np.uint8).reshape(H * (NOPE + VH), KL)
    w_scale = _f32(w_scale).reshape(-1)
    assert w_scale.size == (H * (NOPE + VH) // BLK) * (KL // BLK), "one scale per 128x128 block"
    return w8, w_scale


def q_absorb(q_nope, w8, w_scale) -> np.ndarray:
    """q_lat [..., H, 512] f32 = each head's 128 no-position query values through its W_UK rows of the
    fmt=8 kv_b (w8 [H*256][512] e4m3 bytes, w_scale [H*2][4] block scales); double accumulation."""
    q = _f32(q_nope)
    H = q.shape[-2]
    S = int(q.size // (H * NOPE))
    w8, w_scale = _kvb(w8, w_scale, H)
    out = np.empty(q.shape[:-1] + (KL,), dtype=np.float32)
    _load().kv8o_q_absorb(_ptr(q), S, H, _ptr(w8), _ptr(w_scale), _ptr(out))
    return out


def out_project(ctx, w8, w_scale) -> np.ndarray:
    """out [..., H, 128] f32 = each head's 512-wide context through its W_UV rows of the fmt=8 kv_b."""
    x = _f32(ctx)
    H = x.shape[-2]
    S = int(x.size // (H * KL))
    w8, w_scale = _kvb(w8, w_scale, H)
    out = np.empty(x.shape[:-1] + (VH,), dtype=np.float32)
    _load().kv8o_out_project(_ptr(x), S, H, _ptr(w8), _ptr(w_scale), _ptr(out))
    return out


def index_scores(q8, q_scale, w, k8, k_scale, T: int, seq_stride_rows: int) -> np.ndarray:
    """Indexer scores [B][T] (double): q8 [B][HI][DI] u8, q_scale [B][HI], w [B][HI] f32, k8 [rows][DI] u8,
    k_scale [rows] f32; item b's position t reads key row b * seq_stride_rows + t."""
    q8 = np.ascontiguousarray(q8, dtype=np.uint8)
    B, HI, DI = q8.shape
    q_scale = _f32(q_scale).reshape(B, HI)
    w = _f32(w).reshape(B, HI)
    k8 = np.ascontiguousarray(k8, dtype=np.uint8).reshape(-1, DI)
    k_scale = _f32(k_scale).reshape(-1)
    assert (B - 1) * seq_stride_rows + T <= k8.shape[0] and k_scale.size == k8.shape[0]
    out = np.empty((B, T), dtype=np.float64)
    _load().kv8o_index_scores(_ptr(q8), _ptr(q_scale), _ptr(w), B, HI, DI, _ptr(k8), _ptr(k_scale), int(T),
                              int(seq_stride_rows), _ptr(out))
    return out


def topk(scores, k: int) -> np.ndarray:
    """Indices of the k largest scores (smaller index first among equals), ascending, int32."""
    s = np.ascontiguousarray(scores, dtype=np.float64).reshape(-1)
    kk = min(int(k), s.size)
    out = np.empty(kk, dtype=np.int32)
    _load().kv8o_topk(_ptr(s), s.size, int(k), _ptr(out))
    return out


MX_NOPE, MX_ROPE = 448, 64


def attn_mixed_decode(q_nope, q_rope, k8, k_scale, k_rope, sm_scale) -> np.ndarray:
    """Mixed-precision cache decode: q_nope [H][448] and q_rope [H][64] (f32 holding bf16 values); the cache's
    k8 [T][448] e4m3 bytes, k_scale [T] f32, k_rope [T][64] (f32 holding bf16 values).  q_nope is quantized
    per head by the row quantizer first.  Returns out [H][512] f32."""
    qn = _f32(q_nope).reshape(-1, MX_NOPE)
    H = qn.shape[0]
    q8, qs = quant_rows_w(qn, MX_NOPE)
    qr = _f32(q_rope).reshape(H, MX_ROPE)
    k8 = np.ascontiguousarray(k8, dtype=np.uint8).reshape(-1, MX_NOPE)
    T = k8.shape[0]
    ks = _f32(k_scale).reshape(T)
    kr = _f32(k_rope).reshape(T, MX_ROPE)
    out = np.empty((H, MX_NOPE + MX_ROPE), dtype=np.float32)
    _load().kv8o_attn_mixed_decode(_ptr(q8), _ptr(qs), _ptr(qr), H, _ptr(k8), _ptr(ks), _ptr(kr), T,
                                   float(np.float32(sm_scale)), _ptr(out))
    return out


def num_threads() -> int:
    return int(_load().kv8o_num_threads())


def set_num_threads(n: int) -> None:
    _load().kv8o_set_num_threads(int(n))
