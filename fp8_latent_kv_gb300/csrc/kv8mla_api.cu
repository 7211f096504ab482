// kv8mla_api.cu -- the C ABI (include/kv8mla.h): host-side validation and launches.
//
// Every entry point validates its scalars and pointers before enqueuing anything, returns a
// KV8_E* code instead of falling back, allocates nothing and never synchronises (page "B1 Mixed
// FP8/BF16 FMHA first pass", "Intentional first-pass limits": unsupported shapes are a hard error).
#include "internal.h"

#include <math.h>

namespace kv8 {
namespace {

inline bool aligned(const void *p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int status(cudaError_t e) { return e == cudaSuccess ? KV8_OK : KV8_ECUDA; }

inline bool valid_q(const void *q_lat, const void *q_rope, int q_dtype) {
    return aligned(q_lat, 16) && aligned(q_rope, 16) && (q_dtype == KV8_F32 || q_dtype == KV8_BF16);
}

inline bool valid_cache(const uint8_t *kv8, const float *kv_scale, int64_t T) {
    return aligned(kv8, 16) && aligned(kv_scale, 4) && T >= 1 && T <= KV8_MAX_ROWS;
}

// The address the current device's kernels use for p: device memory of the current device as is,
// page-locked host memory through its mapping; null for anything a kernel cannot reach (pageable
// host memory, another device's memory, an unknown pointer).
const void *device_view(const void *p) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();  // clear the error the query left
        return nullptr;
    }
    switch (at.type) {
        case cudaMemoryTypeDevice: return at.device == dev ? p : nullptr;
        case cudaMemoryTypeManaged: return p;
        case cudaMemoryTypeHost: return at.devicePointer;
        default: return nullptr;
    }
}

}  // namespace

size_t decode_partial_bytes(int P, int H) {
    return ((PartialView::floats(1, P, H) * sizeof(float)) + 255) & ~(size_t)255;
}

size_t sel_partial_bytes(int B, int P, int H) {
    return ((PartialView::floats(B, P, H) * sizeof(float)) + 255) & ~(size_t)255;
}

int device_sm_count() {
    // a property of the GPU, so it may be kept per device id; with no visible device (host-only size
    // queries) the answer is GB300's 152
    constexpr int kMaxDev = 64;
    static int cache[kMaxDev] = {0};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        (void)cudaGetLastError();
        return 152;
    }
    if (dev < kMaxDev && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 152;
    }
    if (dev < kMaxDev) cache[dev] = n;
    return n;
}

int decode_partitions(int H, int64_t T, int P_req) {
    if (T < 1) return 1;
    if (P_req > 0) {
        int64_t p = P_req < T ? P_req : T;
        return (int)(p > 65535 ? 65535 : p);
    }
    // automatic: one wave of tensor-core CTAs on the current device (one per SM: a CTA per partition
    // and 64-head half), at least 128 rows per partition
    const int64_t sms = device_sm_count();
    const int64_t cap = H > 64 ? sms / 2 : sms;
    const int64_t p = (T + 127) / 128;
    return (int)(p < cap ? p : (cap < 1 ? 1 : cap));
}

int batch_partitions(int B, int H, int64_t T_max) {
    // one wave of tensor-core CTAs on the current device (one per SM): B items x P partitions x head
    // halves, at least 128 rows per partition
    const int64_t n_half = H > 64 ? 2 : 1;
    int64_t cap = device_sm_count() / ((int64_t)B * n_half);
    if (cap < 1) cap = 1;
    const int64_t p = (T_max + 127) / 128;
    return (int)(p < cap ? p : cap);
}

size_t decode_partial_bytes_b(int B, int P, int H) {
    return ((PartialView::floats(B, P, H) * sizeof(float)) + 255) & ~(size_t)255;
}

int select_partitions(int B, int H, int NS) {
    // one wave of tensor-core CTAs on the current device (one per SM): B items x P partitions x head
    // halves, with the list's 128-row tiles spread evenly over the partitions
    const int64_t n_half = H > 64 ? 2 : 1;
    const int64_t tiles = (NS + 127) / 128;
    int64_t cap = device_sm_count() / ((int64_t)B * n_half);
    if (cap < 1) cap = 1;
    const int64_t per = (tiles + cap - 1) / cap;
    const int64_t p = (tiles + per - 1) / per;
    return (int)(p < 1 ? 1 : p);
}

}  // namespace kv8

using namespace kv8;

extern "C" {

const char *kv8_strerror(int code) {
    switch (code) {
        case KV8_OK: return "ok";
        case KV8_EINVAL: return "invalid argument (null pointer, size, alignment or limit)";
        case KV8_EWORKSPACE: return "workspace too small";
        case KV8_ECUDA: return "CUDA launch failed";
        case KV8_EUNSUPPORTED: return "unsupported device or shape";
        default: return "unknown kv8 error code";
    }
}

int mla_mixed_decode8_workspace_bytes(int H, int64_t T, size_t *bytes) {
    if (H < 1 || H > KV8_MAX_HEADS || T < 1 || T > KV8_MAX_ROWS || !bytes) return KV8_EINVAL;
    // partial sets first (the documented layout), then staging for the query prep
    const int P = mixed_partitions(H, T);
    *bytes = decode_partial_bytes(P, H) + mixed_scratch_bytes(H, P);
    return KV8_OK;
}

int mla_absorb_mixed_decode8(const void *q_nope, const void *q_rope, int q_dtype, int H, const uint8_t *k8,
                             const float *k_scale, const void *k_rope, int64_t T, float sm_scale, void *workspace,
                             size_t ws_bytes, int *err_word, float *out, void *stream) {
    size_t need = 0;
    int rc = mla_mixed_decode8_workspace_bytes(H, T, &need);
    if (rc != KV8_OK) return rc;
    if (!valid_q(q_nope, q_rope, q_dtype) || !aligned(k8, 16) || !aligned(k_scale, 4) || !aligned(k_rope, 16) ||
        !isfinite(sm_scale) || !aligned(workspace, 16) || !aligned(out, 16))
        return KV8_EINVAL;
    if (ws_bytes < need) return KV8_EWORKSPACE;
    const int P = mixed_partitions(H, T);
    rc = status(launch_attn_mixed(q_nope, q_rope, q_dtype == KV8_BF16, H, k8, k_scale, k_rope, T, sm_scale * kLog2e, P,
                                  static_cast<float *>(workspace),
                                  static_cast<uint8_t *>(workspace) + decode_partial_bytes(P, H), err_word,
                                  (cudaStream_t)stream));
    if (rc != KV8_OK) return rc;
    return mla_lse_merge8(workspace, 1, P, H, out, stream);
}

int kv8_quant_rows_scatter(const float *x, int64_t n, const int64_t *dst_rows, uint8_t *kv8, float *kv_scale,
                           int64_t cache_rows, int *err_word, void *stream) {
    if (n < 0 || cache_rows < 0) return KV8_EINVAL;
    if (n == 0) return KV8_OK;
    if (!aligned(x, 16) || !aligned(dst_rows, 8) || !aligned(kv8, 16) || !aligned(kv_scale, 4)) return KV8_EINVAL;
    return status(launch_quant_rows_scatter(x, n, dst_rows, cache_rows, kv8, kv_scale, err_word, (cudaStream_t)stream));
}

int mla_batch_decode8_workspace_bytes(int B, int H, int64_t T_max, size_t *bytes) {
    if (B < 1 || H < 1 || H > KV8_MAX_HEADS || T_max < 1 || T_max > KV8_MAX_ROWS || !bytes) return KV8_EINVAL;
    const int P = batch_partitions(B, H, T_max);
    *bytes = decode_partial_bytes_b(B, P, H) + tc_scratch_bytes(B, P);
    return KV8_OK;
}

int mla_absorb_batch_decode8(const void *q_lat, const void *q_rope, int q_dtype, int B, int H, const uint8_t *kv8,
                             const float *kv_scale, int64_t T_max, int64_t seq_stride_rows, const int32_t *lens,
                             float sm_scale, void *workspace, size_t ws_bytes, int *err_word, float *out,
                             void *stream) {
    size_t need = 0;
    int rc = mla_batch_decode8_workspace_bytes(B, H, T_max, &need);
    if (rc != KV8_OK) return rc;
    if (!valid_q(q_lat, q_rope, q_dtype) || !valid_cache(kv8, kv_scale, T_max) || !aligned(lens, 4) ||
        !isfinite(sm_scale) || !aligned(workspace, 16) || !aligned(out, 16) || seq_stride_rows < 0 ||
        (B > 1 && seq_stride_rows < T_max))
        return KV8_EINVAL;
    if (ws_bytes < need) return KV8_EWORKSPACE;
    AttnArgs a{};
    a.q_lat = q_lat;
    a.q_rope = q_rope;
    a.q_bf16 = q_dtype == KV8_BF16;
    a.B = B;
    a.H = H;
    a.kv8 = kv8;
    a.kv_scale = kv_scale;
    a.T = T_max;
    a.seq_stride_rows = B > 1 ? seq_stride_rows : 0;
    a.idx = nullptr;
    a.lens = lens;
    a.pos0 = -1;
    a.sm_scale_log2 = sm_scale * kLog2e;
    a.P = batch_partitions(B, H, T_max);
    a.ws = static_cast<float *>(workspace);
    a.out = nullptr;
    a.err_word = err_word;
    a.tc_scratch = static_cast<uint8_t *>(workspace) + decode_partial_bytes_b(B, a.P, H);
    // bf16 queries: tensor cores (32-bit tensor-map row coordinates); f32 queries: CUDA cores
    const bool tc = a.q_bf16 && (int64_t)(B - 1) * a.seq_stride_rows + T_max <= 0x7fffffffLL;
    rc = status(tc ? launch_attn_tc(a, (cudaStream_t)stream) : launch_attn_simt(a, (cudaStream_t)stream));
    if (rc != KV8_OK) return rc;
    return mla_lse_merge8(workspace, B, a.P, H, out, stream);
}

int kv8_quant_rows_w(const float *x, int64_t n, int width, uint8_t *q, float *scale, void *stream) {
    if (n < 0 || (width != KV8_ROW_BYTES && width != KV8_IDX_D && width != KV8_MX_NOPE)) return KV8_EINVAL;
    if (n == 0) return KV8_OK;
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4)) return KV8_EINVAL;
    return status(launch_quant_rows_w(x, n, width, q, scale, (cudaStream_t)stream));
}

int dsa_index_workspace_bytes(int B, size_t *bytes) {
    if (B < 1 || !bytes) return KV8_EINVAL;
    *bytes = topk_workspace_bytes(B);
    return KV8_OK;
}

int dsa_index_topk8(const void *q_idx, int q_dtype, const float *w, int B, int HI, const uint8_t *k8,
                    const float *k_scale, int64_t T, int64_t seq_stride_rows, int NS, void *workspace,
                    size_t ws_bytes, float *scores, int32_t *idx, int *err_word, void *stream) {
    if (B < 1 || HI < 16 || HI > KV8_MAX_IDX_HEADS || HI % 16 != 0 || T < 1 || T > KV8_MAX_ROWS || NS < 1 ||
        NS > KV8_MAX_SELECT || seq_stride_rows < 0)
        return KV8_EINVAL;
    if ((int64_t)(B - 1) * seq_stride_rows + T >= (1LL << 31) - 128) return KV8_EINVAL;
    if ((q_dtype != KV8_F32 && q_dtype != KV8_BF16) || !aligned(q_idx, 16) || !aligned(w, 4) || !aligned(k8, 16) ||
        !aligned(k_scale, 4) || !aligned(scores, 16) || !aligned(idx, 16) || !aligned(workspace, 16))
        return KV8_EINVAL;
    if (ws_bytes < topk_workspace_bytes(B)) return KV8_EWORKSPACE;
    cudaError_t e = reset_topk_workspace(workspace, B, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = launch_index_scores(q_idx, q_dtype == KV8_BF16, w, B, HI, k8, k_scale, T, seq_stride_rows, scores, workspace,
                                err_word, (cudaStream_t)stream);
    if (e != cudaSuccess) return KV8_ECUDA;
    return status(launch_topk(scores, B, T, NS, idx, workspace, err_word, (cudaStream_t)stream));
}

int mla_q_absorb8(const void *q_nope, int q_dtype, int S, int H, const uint8_t *w8, const float *w_scale,
                  void *q_lat, int out_dtype, int *err_word, void *stream) {
    if (S < 1 || S > KV8_MAX_ROWS || H < 1 || H > KV8_MAX_HEADS) return KV8_EINVAL;
    if (!aligned(q_nope, 16) || !aligned(w8, 16) || !aligned(w_scale, 4) || !aligned(q_lat, 16)) return KV8_EINVAL;
    if ((q_dtype != KV8_F32 && q_dtype != KV8_BF16) || (out_dtype != KV8_F32 && out_dtype != KV8_BF16))
        return KV8_EINVAL;
    return status(launch_q_absorb(q_nope, q_dtype == KV8_BF16, S, H, w8, w_scale, q_lat, out_dtype == KV8_BF16,
                                  err_word, (cudaStream_t)stream));
}

int mla_out_project8(const float *ctx, int S, int H, const uint8_t *w8, const float *w_scale, float *out,
                     int *err_word, void *stream) {
    if (S < 1 || S > KV8_MAX_ROWS || H < 1 || H > KV8_MAX_HEADS) return KV8_EINVAL;
    if (!aligned(ctx, 16) || !aligned(w8, 16) || !aligned(w_scale, 4) || !aligned(out, 16)) return KV8_EINVAL;
    return status(launch_out_project(ctx, S, H, w8, w_scale, out, err_word, (cudaStream_t)stream));
}

int kv8_copy(void *dst, const void *src, size_t bytes, void *stream) {
    if (bytes == 0) return KV8_OK;
    if (!dst || !src) return KV8_EINVAL;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    if (d < s + bytes && s < d + bytes) return KV8_EINVAL;  // overlapping ranges
    void *dd = const_cast<void *>(device_view(dst));
    const void *ds = device_view(src);
    if (!dd || !ds) return KV8_EINVAL;
    return status(launch_copy(dd, ds, bytes, (cudaStream_t)stream));
}

int kv8_wait_selftest(uint64_t limit_ns, int *err_word, int *wait_status, void *stream) {
    if (limit_ns < 1000ull || limit_ns > 1000000000ull || !aligned(err_word, 4) || !aligned(wait_status, 4))
        return KV8_EINVAL;
    return status(launch_wait_selftest(limit_ns, err_word, wait_status, (cudaStream_t)stream));
}

int kv8_encode_e4m3(const float *y, int64_t n, uint8_t *out, void *stream) {
    if (n < 0) return KV8_EINVAL;
    if (n == 0) return KV8_OK;
    if (!aligned(y, 16) || !aligned(out, 4)) return KV8_EINVAL;
    return status(launch_encode(y, n, out, (cudaStream_t)stream));
}

int kv8_quant_rows(const float *x, int64_t n, uint8_t *kv8, float *kv_scale, void *stream) {
    if (n < 0) return KV8_EINVAL;
    if (n == 0) return KV8_OK;
    if (!aligned(x, 16) || !aligned(kv8, 16) || !aligned(kv_scale, 4)) return KV8_EINVAL;
    return status(launch_quant_rows(x, n, kv8, kv_scale, (cudaStream_t)stream));
}

int mla_decode8_partitions(int H, int64_t T, int P_req, int *P_out) {
    if (!P_out || H < 1 || H > KV8_MAX_HEADS || T < 1 || T > KV8_MAX_ROWS || P_req < 0) return KV8_EINVAL;
    *P_out = decode_partitions(H, T, P_req);
    return KV8_OK;
}

int mla_decode8_workspace_bytes(int H, int64_t T, int P_req, size_t *bytes) {
    int P = 0;
    int rc = mla_decode8_partitions(H, T, P_req, &P);
    if (rc != KV8_OK || !bytes) return rc != KV8_OK ? rc : KV8_EINVAL;
    // partial sets first (the documented layout), then staging for the tensor-core path
    *bytes = decode_partial_bytes(P, H) + tc_scratch_bytes(1, P);
    return KV8_OK;
}

int mla_decode8_partial(const void *q_lat, const void *q_rope, int q_dtype, int H, const uint8_t *kv8,
                        const float *kv_scale, int64_t T, float sm_scale, int P_req, void *workspace,
                        size_t ws_bytes, int *err_word, void *stream) {
    size_t need = 0;
    int rc = mla_decode8_workspace_bytes(H, T, P_req, &need);
    if (rc != KV8_OK) return rc;
    if (!valid_q(q_lat, q_rope, q_dtype) || !valid_cache(kv8, kv_scale, T) || !isfinite(sm_scale) ||
        !aligned(workspace, 16))
        return KV8_EINVAL;
    if (ws_bytes < need) return KV8_EWORKSPACE;
    AttnArgs a{};
    a.q_lat = q_lat;
    a.q_rope = q_rope;
    a.q_bf16 = q_dtype == KV8_BF16;
    a.B = 1;
    a.H = H;
    a.kv8 = kv8;
    a.kv_scale = kv_scale;
    a.T = T;
    a.seq_stride_rows = 0;
    a.idx = nullptr;
    a.NS = 0;
    a.pos0 = -1;
    a.sm_scale_log2 = sm_scale * kLog2e;
    a.P = decode_partitions(H, T, P_req);
    a.ws = static_cast<float *>(workspace);
    a.out = nullptr;
    a.err_word = err_word;
    a.tc_scratch = static_cast<uint8_t *>(workspace) + decode_partial_bytes(a.P, H);
    // bf16 queries: tensor cores; f32 queries keep full f32 precision on the CUDA cores
    return status(a.q_bf16 ? launch_attn_tc(a, (cudaStream_t)stream) : launch_attn_simt(a, (cudaStream_t)stream));
}

int mla_lse_merge8(const void *workspace, int B, int P, int H, float *out, void *stream) {
    if (!aligned(workspace, 16) || !aligned(out, 16) || B < 1 || B > 65535 || P < 1 || P > 65535 || H < 1 ||
        H > KV8_MAX_HEADS)
        return KV8_EINVAL;
    return status(launch_lse_merge(static_cast<const float *>(workspace), B, P, H, out, (cudaStream_t)stream));
}

int mla_absorb_decode8(const void *q_lat, const void *q_rope, int q_dtype, int H, const uint8_t *kv8,
                       const float *kv_scale, int64_t T, float sm_scale, int P_req, void *workspace,
                       size_t ws_bytes, int *err_word, float *out, void *stream) {
    if (!aligned(out, 16)) return KV8_EINVAL;
    int rc = mla_decode8_partial(q_lat, q_rope, q_dtype, H, kv8, kv_scale, T, sm_scale, P_req, workspace, ws_bytes,
                                 err_word, stream);
    if (rc != KV8_OK) return rc;
    return mla_lse_merge8(workspace, 1, decode_partitions(H, T, P_req), H, out, stream);
}

int mla_sel8_workspace_bytes(int B, int H, int NS, size_t *bytes) {
    if (!bytes || B < 1 || B > 65535 || H < 1 || H > KV8_MAX_HEADS || NS < 1 || NS > KV8_MAX_SELECT)
        return KV8_EINVAL;
    const int P = select_partitions(B, H, NS);
    // partial sets first, then staging for the tensor-core path
    *bytes = sel_partial_bytes(B, P, H) + tc_scratch_bytes(B, P);
    return KV8_OK;
}

int mla_absorb_sel8(const void *q_lat, const void *q_rope, int q_dtype, int B, int H, const uint8_t *kv8,
                    const float *kv_scale, int64_t T, int64_t seq_stride_rows, const int32_t *idx, int NS,
                    float sm_scale, void *workspace, size_t ws_bytes, int *err_word, float *out, void *stream) {
    size_t need = 0;
    int rc = mla_sel8_workspace_bytes(B, H, NS, &need);
    if (rc != KV8_OK) return rc;
    if (!valid_q(q_lat, q_rope, q_dtype) || !valid_cache(kv8, kv_scale, T) || !aligned(idx, 4) ||
        !isfinite(sm_scale) || !aligned(workspace, 16) || !aligned(out, 16) || seq_stride_rows < 0 ||
        (B > 1 && seq_stride_rows < T))
        return KV8_EINVAL;
    if (ws_bytes < need) return KV8_EWORKSPACE;
    AttnArgs a{};
    a.q_lat = q_lat;
    a.q_rope = q_rope;
    a.q_bf16 = q_dtype == KV8_BF16;
    a.B = B;
    a.H = H;
    a.kv8 = kv8;
    a.kv_scale = kv_scale;
    a.T = T;
    a.seq_stride_rows = B > 1 ? seq_stride_rows : 0;
    a.idx = idx;
    a.NS = NS;
    a.pos0 = -1;
    a.sm_scale_log2 = sm_scale * kLog2e;
    a.P = select_partitions(B, H, NS);
    a.ws = static_cast<float *>(workspace);
    a.out = nullptr;
    a.err_word = err_word;
    a.tc_scratch = static_cast<uint8_t *>(workspace) + sel_partial_bytes(B, a.P, H);
    // bf16 queries: tensor cores (row gathers address all items' caches with 32-bit row coordinates);
    // f32 queries, or caches spanning 2^31 rows or more: CUDA cores
    const bool tc = a.q_bf16 && (int64_t)(B - 1) * a.seq_stride_rows + T <= 0x7fffffffLL;
    rc = status(tc ? launch_attn_tc(a, (cudaStream_t)stream) : launch_attn_simt(a, (cudaStream_t)stream));
    if (rc != KV8_OK) return rc;
    return mla_lse_merge8(workspace, B, a.P, H, out, stream);
}

int mla_absorb_prefill8(const void *q_lat, const void *q_rope, int q_dtype, int S, int H, int64_t pos0,
                        const uint8_t *kv8, const float *kv_scale, int64_t T, float sm_scale, int *err_word,
                        float *out, void *stream) {
    if (!valid_q(q_lat, q_rope, q_dtype) || !valid_cache(kv8, kv_scale, T) || !aligned(out, 16) ||
        !isfinite(sm_scale) || S < 1 || S > 65535 || H < 1 || H > KV8_MAX_HEADS || pos0 < 0 || pos0 + S > T)
        return KV8_EINVAL;
    AttnArgs a{};
    a.q_lat = q_lat;
    a.q_rope = q_rope;
    a.q_bf16 = q_dtype == KV8_BF16;
    a.B = S;
    a.H = H;
    a.kv8 = kv8;
    a.kv_scale = kv_scale;
    a.T = T;
    a.seq_stride_rows = 0;
    a.idx = nullptr;
    a.NS = 0;
    a.pos0 = pos0;
    a.sm_scale_log2 = sm_scale * kLog2e;
    a.P = 1;
    a.ws = nullptr;
    a.out = out;
    a.err_word = err_word;
    return status(a.q_bf16 ? launch_attn_tc(a, (cudaStream_t)stream) : launch_attn_simt(a, (cudaStream_t)stream));
}

}  // extern "C"
