// internal.h -- host-side launchers behind the C ABI (not exported).
#pragma once

#include "common.cuh"

#include <cudaTypedefs.h>

namespace kv8 {

// One attention problem set: B batch items (decode: 1; selection: B sequences; prefill: S queries),
// each with H heads, attending a list of rows of a cache, split into P partitions.
struct AttnArgs {
    const void *q_lat;        // [B][H][512]
    const void *q_rope;       // [B][H][64]
    int q_bf16;               // 1: bf16 queries, 0: f32
    int B, H;
    const uint8_t *kv8;       // cache rows [*][576]
    const float *kv_scale;    // [*]
    int64_t T;                // rows in each batch item's cache
    int64_t seq_stride_rows;  // rows between consecutive batch items' caches (selection), else 0
    const int32_t *idx;       // selection lists [B][NS], or nullptr for a dense row range
    int NS;                   // selection length
    int64_t pos0;             // causal prefill: item i attends rows [0, pos0 + i]; -1 = not causal
    const int32_t *lens;      // batched dense decode: item i attends its rows [0, lens[i]) (device; clamped
                              // to [0, T]), or null
    float sm_scale_log2;      // sm_scale * log2(e)
    int P;                    // partitions per batch item
    float *ws;                // partial sets (PartialView layout), or nullptr when `out` is written directly
    float *out;               // [B][H][512] normalised output (used when ws == nullptr; requires P == 1)
    int *err_word;            // optional device error word
    void *tc_scratch;         // decode / selection on the tensor cores: staging for the prepared queries
                              // (tc_scratch_bytes(B, P)); null for prefill
};

cudaError_t launch_quant_rows(const float *x, int64_t n, uint8_t *q, float *scale, cudaStream_t st);
cudaError_t launch_quant_rows_scatter(const float *x, int64_t n, const int64_t *dst, int64_t cache_rows, uint8_t *q,
                                      float *scale, int *err_word, cudaStream_t st);
cudaError_t launch_quant_rows_w(const float *x, int64_t n, int width, uint8_t *q, float *scale, cudaStream_t st);
// the scores also fill each item's pass-0 top-k histogram in topk_ws (zeroed first by reset_topk_workspace)
cudaError_t launch_index_scores(const void *q, int q_bf16, const float *w, int B, int HI, const uint8_t *k8,
                                const float *k_scale, int64_t T, int64_t seq_stride_rows, float *scores,
                                void *topk_ws, int *err_word, cudaStream_t st);
size_t topk_workspace_bytes(int B);
cudaError_t reset_topk_workspace(void *ws, int B, cudaStream_t st);
cudaError_t launch_topk(const float *scores, int B, int64_t T, int NS, int32_t *idx, void *ws, int *err_word,
                        cudaStream_t st);
cudaError_t launch_encode(const float *y, int64_t n, uint8_t *out, cudaStream_t st);
cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t st);
// tcgen05 kernel for bf16 queries: a dense (optionally causal) row range, or selection lists (which
// need tc_scratch and (B-1)*seq_stride_rows + T < 2^31).
cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t st);
size_t tc_scratch_bytes(int B, int P);
cudaError_t launch_q_absorb(const void *q_nope, int q_bf16, int S, int H, const uint8_t *w8, const float *w_scale,
                            void *q_lat, int out_bf16, int *err_word, cudaStream_t st);
cudaError_t launch_out_project(const float *ctx, int S, int H, const uint8_t *w8, const float *w_scale, float *out,
                               int *err_word, cudaStream_t st);
cudaError_t launch_q_absorb_tc(const void *q_nope, int q_bf16, int S, int H, const uint8_t *w8, const float *w_scale,
                               void *q_lat, int out_bf16, int *err_word, cudaStream_t st);
cudaError_t launch_out_project_tc(const float *ctx, int S, int H, const uint8_t *w8, const float *w_scale, float *out,
                                  int *err_word, cudaStream_t st);
// diagnostic: one CTA's bounded wait on an mbarrier nothing completes (see kv8_wait_selftest)
cudaError_t launch_wait_selftest(uint64_t limit_ns, int *err_word, int *status, cudaStream_t st);
// the driver's cuTensorMapEncodeTiled, looked up once; null if unavailable
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
int mixed_partitions(int H, int64_t T);
cudaError_t launch_attn_mixed(const void *q_nope, const void *q_rope, int q_bf16, int H, const uint8_t *k8,
                              const float *k_scale, const void *k_rope, int64_t T, float sm_scale_log2, int P,
                              float *ws, void *scratch, int *err_word, cudaStream_t st);
// staging for the mixed decode's query prep (query images, score factors, row-scale maxima)
size_t mixed_scratch_bytes(int H, int P);
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t st);
cudaError_t launch_lse_merge(const float *ws, int B, int P, int H, float *out, cudaStream_t st);

// Partition policy shared by the workspace queries and the launchers: one wave of CTAs on the current
// device, from its multiprocessor count (152 when no device is visible).
int device_sm_count();
int decode_partitions(int H, int64_t T, int P_req);
int select_partitions(int B, int H, int NS);
int batch_partitions(int B, int H, int64_t T_max);
size_t decode_partial_bytes_b(int B, int P, int H);

}  // namespace kv8
