"""Python binding of libkv8mla.so: fp8 latent-KV absorbed MLA attention for GB300 (sm_103a).

Argument marshalling only: every step runs in the library's CUDA kernels.  Functions carry the C ABI
names (include/kv8mla.h) and take torch CUDA tensors; the stream defaults to torch's current stream.
A nonzero return code raises Kv8Error.  There is no fallback: if the library is missing or fails to
load, `load()` raises.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkv8mla.so")

KV8_ROW_BYTES, KV8_KL, KV8_KR = 576, 512, 64
KV8_MAX_HEADS, KV8_MAX_ROWS, KV8_MAX_SELECT = 128, 1 << 20, 4096
KV8_OK, KV8_EINVAL, KV8_EWORKSPACE, KV8_ECUDA, KV8_EUNSUPPORTED = 0, -1, -2, -3, -4
KV8_ERR_INDEX, KV8_ERR_TIMEOUT = 1, 2
KV8_F32, KV8_BF16 = 0, 1

# (restype, argtypes) for every exported symbol of include/kv8mla.h
_P, _I, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "kv8_encode_e4m3": (_I, [_P, _I64, _P, _P]),
    "kv8_quant_rows": (_I, [_P, _I64, _P, _P, _P]),
    "mla_decode8_partitions": (_I, [_I, _I64, _I, _P]),
    "mla_decode8_workspace_bytes": (_I, [_I, _I64, _I, _P]),
    "mla_decode8_partial": (_I, [_P, _P, _I, _I, _P, _P, _I64, _F, _I, _P, _SZ, _P, _P]),
    "mla_lse_merge8": (_I, [_P, _I, _I, _I, _P, _P]),
    "mla_absorb_decode8": (_I, [_P, _P, _I, _I, _P, _P, _I64, _F, _I, _P, _SZ, _P, _P, _P]),
    "mla_sel8_workspace_bytes": (_I, [_I, _I, _I, _P]),
    "mla_absorb_sel8": (_I, [_P, _P, _I, _I, _I, _P, _P, _I64, _I64, _P, _I, _F, _P, _SZ, _P, _P, _P]),
    "mla_absorb_prefill8": (_I, [_P, _P, _I, _I, _I, _I64, _P, _P, _I64, _F, _P, _P, _P]),
    "mla_absorb_decode8_noalloc": (_I, [_P, _P, _I, _I, _P, _P, _I64, _F, _I, _P, _P, _P]),
    "mla_q_absorb8": (_I, [_P, _I, _I, _I, _P, _P, _P, _I, _P, _P]),
    "kv8_quant_rows_w": (_I, [_P, _I64, _I, _P, _P, _P]),
    "kv8_quant_rows_scatter": (_I, [_P, _I64, _P, _P, _P, _I64, _P, _P]),
    "mla_mixed_decode8_workspace_bytes": (_I, [_I, _I64, _P]),
    "mla_absorb_mixed_decode8": (_I, [_P, _P, _I, _I, _P, _P, _P, _I64, _F, _P, _SZ, _P, _P, _P]),
    "mla_batch_decode8_workspace_bytes": (_I, [_I, _I, _I64, _P]),
    "mla_absorb_batch_decode8": (_I, [_P, _P, _I, _I, _I, _P, _P, _I64, _I64, _P, _F, _P, _SZ, _P, _P, _P]),
    "dsa_index_workspace_bytes": (_I, [_I, _P]),
    "dsa_index_topk8": (_I, [_P, _I, _P, _I, _I, _P, _P, _I64, _I64, _I, _P, _SZ, _P, _P, _P, _P]),
    "mla_out_project8": (_I, [_P, _I, _I, _P, _P, _P, _P, _P]),
    "kv8_copy": (_I, [_P, _P, _SZ, _P]),
    "kv8_wait_selftest": (_I, [ctypes.c_uint64, _P, _P, _P]),
    "kv8_strerror": (ctypes.c_char_p, [_I]),
}

_lib = None


class Kv8Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        msg = _lib.kv8_strerror(code).decode() if _lib is not None else str(code)
        super().__init__(f"{fn} returned {code}: {msg}")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libkv8mla.so (build it first with fp8_latent_kv_gb300.build / __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first (python -m fp8_latent_kv_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> None:
    if rc != KV8_OK:
        raise Kv8Error(fn, rc)


def _qdtype(q) -> int:
    import torch
    if q.dtype == torch.bfloat16:
        return KV8_BF16
    if q.dtype == torch.float32:
        return KV8_F32
    raise TypeError(f"queries must be float32 or bfloat16, got {q.dtype}")


def kv8_encode_e4m3(y, out, stream=None) -> None:
    _check("kv8_encode_e4m3", load().kv8_encode_e4m3(_ptr(y), y.numel(), _ptr(out), _stream(stream)))


def kv8_quant_rows(x, kv8, kv_scale, n: int | None = None, stream=None) -> None:
    """x [n][576] f32 -> kv8 [n][576] u8 (or a view starting at the first row to write), kv_scale [n]."""
    n = x.shape[0] if n is None else n
    _check("kv8_quant_rows", load().kv8_quant_rows(_ptr(x), n, _ptr(kv8), _ptr(kv_scale), _stream(stream)))


def mla_decode8_partitions(H: int, T: int, P_req: int = 0) -> int:
    out = ctypes.c_int(0)
    _check("mla_decode8_partitions", load().mla_decode8_partitions(H, T, P_req, ctypes.addressof(out)))
    return out.value


def mla_decode8_workspace_bytes(H: int, T: int, P_req: int = 0) -> int:
    out = ctypes.c_size_t(0)
    _check("mla_decode8_workspace_bytes", load().mla_decode8_workspace_bytes(H, T, P_req, ctypes.addressof(out)))
    return out.value


def mla_decode8_partial(q_lat, q_rope, kv8, kv_scale, T: int, sm_scale: float, workspace, P_req: int = 0,
                        err_word=None, stream=None) -> None:
    H = q_lat.shape[-2]
    _check("mla_decode8_partial", load().mla_decode8_partial(
        _ptr(q_lat), _ptr(q_rope), _qdtype(q_lat), H, _ptr(kv8), _ptr(kv_scale), T, sm_scale, P_req,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err_word), _stream(stream)))


def mla_mixed_decode8_workspace_bytes(H: int, T: int) -> int:
    out = ctypes.c_size_t(0)
    _check("mla_mixed_decode8_workspace_bytes", load().mla_mixed_decode8_workspace_bytes(H, T, ctypes.addressof(out)))
    return out.value


def mla_absorb_mixed_decode8(q_nope, q_rope, k8, k_scale, k_rope, sm_scale: float, workspace, out, err_word=None,
                             stream=None) -> None:
    """Mixed-cache decode: q_nope [H][448], q_rope [H][64] (f32 or bf16); k8 [T][448] uint8, k_scale [T] f32,
    k_rope [T][64] bf16 -> out [H][512] f32."""
    H = q_nope.shape[-2]
    T = k8.shape[0]
    _check("mla_absorb_mixed_decode8", load().mla_absorb_mixed_decode8(
        _ptr(q_nope), _ptr(q_rope), _qdtype(q_nope), H, _ptr(k8), _ptr(k_scale), _ptr(k_rope), T, sm_scale,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err_word), _ptr(out), _stream(stream)))


def kv8_quant_rows_scatter(x, dst_rows, kv8, kv_scale, err_word=None, stream=None) -> None:
    """Quantize rows x [n][576] f32 into cache rows dst_rows [n] (int64 tensor) of kv8 [rows][576] / kv_scale."""
    n = x.numel() // 576
    _check("kv8_quant_rows_scatter", load().kv8_quant_rows_scatter(
        _ptr(x), n, _ptr(dst_rows), _ptr(kv8), _ptr(kv_scale), kv8.shape[0], _ptr(err_word), _stream(stream)))


def mla_batch_decode8_workspace_bytes(B: int, H: int, T_max: int) -> int:
    out = ctypes.c_size_t(0)
    _check("mla_batch_decode8_workspace_bytes", load().mla_batch_decode8_workspace_bytes(B, H, T_max,
                                                                                         ctypes.addressof(out)))
    return out.value


def mla_absorb_batch_decode8(q_lat, q_rope, kv8, kv_scale, T_max: int, seq_stride_rows: int, lens, sm_scale: float,
                             workspace, out, err_word=None, stream=None) -> None:
    """B sequences, sequence b attending its first lens[b] rows of cache rows b*seq_stride_rows.. (lens: int32
    CUDA tensor [B]) -> out [B][H][512] f32."""
    B, H = q_lat.shape[0], q_lat.shape[1]
    _check("mla_absorb_batch_decode8", load().mla_absorb_batch_decode8(
        _ptr(q_lat), _ptr(q_rope), _qdtype(q_lat), B, H, _ptr(kv8), _ptr(kv_scale), T_max, seq_stride_rows,
        _ptr(lens), sm_scale, _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err_word),
        _ptr(out), _stream(stream)))


def kv8_quant_rows_w(x, q, scale, stream=None) -> None:
    """Rows x [n][width] f32 (width 576 or 128) -> q [n][width] uint8 e4m3, scale [n] f32."""
    width = x.shape[-1]
    n = x.numel() // width
    _check("kv8_quant_rows_w", load().kv8_quant_rows_w(_ptr(x), n, width, _ptr(q), _ptr(scale), _stream(stream)))


def dsa_index_workspace_bytes(B: int) -> int:
    out = ctypes.c_size_t(0)
    _check("dsa_index_workspace_bytes", load().dsa_index_workspace_bytes(B, ctypes.addressof(out)))
    return out.value


def dsa_index_topk8(q_idx, w, k8, k_scale, T: int, seq_stride_rows: int, NS: int, workspace, scores, idx,
                    err_word=None, stream=None) -> None:
    """DSA indexer: q_idx [B][HI][128] (f32/bf16), w [B][HI] f32, index keys k8 [rows][128] uint8 + k_scale
    [rows] f32 -> scores [B][T] f32 and idx [B][NS] int32 (top positions, ascending)."""
    B, HI = q_idx.shape[0], q_idx.shape[1]
    _check("dsa_index_topk8", load().dsa_index_topk8(
        _ptr(q_idx), _qdtype(q_idx), _ptr(w), B, HI, _ptr(k8), _ptr(k_scale), T, seq_stride_rows, NS,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(scores), _ptr(idx), _ptr(err_word),
        _stream(stream)))


def mla_q_absorb8(q_nope, w8, w_scale, q_lat, err_word=None, stream=None) -> None:
    """q_lat [S][H][512] (f32 or bf16 tensor) = q_nope [S][H][128] (f32 or bf16) through the key rows of
    the fmt=8 kv_b (w8 [H*256][512] uint8, w_scale [H*2][4] f32)."""
    H = q_nope.shape[-2]
    S = q_nope.numel() // (H * 128)
    _check("mla_q_absorb8", load().mla_q_absorb8(_ptr(q_nope), _qdtype(q_nope), S, H, _ptr(w8), _ptr(w_scale),
                                                 _ptr(q_lat), _qdtype(q_lat), _ptr(err_word), _stream(stream)))


def mla_out_project8(ctx, w8, w_scale, out, err_word=None, stream=None) -> None:
    """out [S][H][128] f32 = ctx [S][H][512] f32 through the value rows of the fmt=8 kv_b."""
    H = ctx.shape[-2]
    S = ctx.numel() // (H * 512)
    _check("mla_out_project8", load().mla_out_project8(_ptr(ctx), S, H, _ptr(w8), _ptr(w_scale), _ptr(out),
                                                       _ptr(err_word), _stream(stream)))


def kv8_wait_selftest(limit_ns: int, err_word, wait_status, stream=None) -> None:
    """Diagnostic: a bounded wait that nothing completes; sets KV8_ERR_TIMEOUT in err_word and 2 in wait_status
    (both int32 device tensors) after limit_ns."""
    _check("kv8_wait_selftest", load().kv8_wait_selftest(limit_ns, _ptr(err_word), _ptr(wait_status), _stream(stream)))


def kv8_copy(dst, src, nbytes: int | None = None, stream=None) -> None:
    """Copy nbytes (default: all of src) from src to dst with a kernel; either may be a CUDA tensor or a
    pinned (page-locked) CPU tensor."""
    n = src.numel() * src.element_size() if nbytes is None else int(nbytes)
    _check("kv8_copy", load().kv8_copy(_ptr(dst), _ptr(src), n, _stream(stream)))


def mla_lse_merge8(workspace, B: int, P: int, H: int, out, stream=None) -> None:
    _check("mla_lse_merge8", load().mla_lse_merge8(_ptr(workspace), B, P, H, _ptr(out), _stream(stream)))


def mla_absorb_decode8(q_lat, q_rope, kv8, kv_scale, T: int, sm_scale: float, workspace, out, P_req: int = 0,
                       err_word=None, stream=None) -> None:
    H = q_lat.shape[-2]
    _check("mla_absorb_decode8", load().mla_absorb_decode8(
        _ptr(q_lat), _ptr(q_rope), _qdtype(q_lat), H, _ptr(kv8), _ptr(kv_scale), T, sm_scale, P_req,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err_word), _ptr(out), _stream(stream)))


def mla_sel8_workspace_bytes(B: int, H: int, NS: int) -> int:
    out = ctypes.c_size_t(0)
    _check("mla_sel8_workspace_bytes", load().mla_sel8_workspace_bytes(B, H, NS, ctypes.addressof(out)))
    return out.value


def mla_absorb_sel8(q_lat, q_rope, kv8, kv_scale, T: int, seq_stride_rows: int, idx, sm_scale: float, workspace,
                    out, err_word=None, stream=None) -> None:
    B, NS = idx.shape
    H = q_lat.shape[-2]
    _check("mla_absorb_sel8", load().mla_absorb_sel8(
        _ptr(q_lat), _ptr(q_rope), _qdtype(q_lat), B, H, _ptr(kv8), _ptr(kv_scale), T, seq_stride_rows, _ptr(idx),
        NS, sm_scale, _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err_word), _ptr(out),
        _stream(stream)))


def mla_absorb_prefill8(q_lat, q_rope, pos0: int, kv8, kv_scale, T: int, sm_scale: float, out, err_word=None,
                        stream=None) -> None:
    S, H = q_lat.shape[0], q_lat.shape[1]
    _check("mla_absorb_prefill8", load().mla_absorb_prefill8(
        _ptr(q_lat), _ptr(q_rope), _qdtype(q_lat), S, H, pos0, _ptr(kv8), _ptr(kv_scale), T, sm_scale,
        _ptr(err_word), _ptr(out), _stream(stream)))


def mla_absorb_decode8_noalloc(q_lat, q_rope, kv8, kv_scale, T: int, sm_scale: float, out, P_req: int = 0,
                               err_word=None, stream=None) -> None:
    """Decode without a workspace argument: the partials live in the library's fixed device array."""
    H = q_lat.shape[-2]
    _check("mla_absorb_decode8_noalloc", load().mla_absorb_decode8_noalloc(
        _ptr(q_lat), _ptr(q_rope), _qdtype(q_lat), H, _ptr(kv8), _ptr(kv_scale), T, sm_scale, P_req,
        _ptr(err_word), _ptr(out), _stream(stream)))


def kv8_strerror(code: int) -> str:
    return load().kv8_strerror(code).decode()
