/*
 * kv8mla.h -- C ABI of the fp8 latent-KV absorbed MLA attention library (libkv8mla.so, sm_103a).
 *
 * The operations follow two web pages:
 *   [KV8]  "KV8 long-context CUDA: fp8 device shadow, split-T kernels, DSA-aware gather"
 *          (colibri pull request #300): first commit message (fp8 row format, c/kv_fp8.h codec,
 *          absorb attention, CUDA wrappers coli_cuda_attention_absorb8 / _absorb_batch8) and second
 *          commit message (device-resident shadow, split-T partial blocks + log-sum-exp merge,
 *          DSA gather attention_absorb_sel_kernel8 with NS <= 4096, batch cap lifted to 1M rows).
 *   [B1]   "B1 Mixed FP8/BF16 FMHA first pass", sections "New files" (C ABI launcher driven from
 *          Python through ctypes) and "Intentional first-pass limits" (an unsupported shape is an
 *          error code; there is no fallback path).
 *   [FMT8] "feat: fmt=8 (fp8-e4m3) decode on the kv_b absorb path, CPU and CUDA" (colibri pull
 *          request #1102): kv_b_proj as raw e4m3 bytes with one f32 scale per 128x128 block.
 *
 * Cache layout (one layer).  Row t of the latent cache is KV8_ROW_BYTES = 576 e4m3 bytes:
 * bytes 0..511 are Lc (kv_lora latent), bytes 512..575 are Rc (qk_rope key), followed in a separate
 * array by one f32 scale s_t = amax_t / 448 covering the whole row.  kv8 is [T][576] u8 row-major,
 * kv_scale is [T] f32.  The attended value of row t, head h:
 *     score[h,t] = sm_scale * s_t * ( q_lat[h].e4m3(Lc8_t) + q_rope[h].e4m3(Rc8_t) )
 *     cl[h]      = sum_t softmax_t(score[h,:]) * s_t * e4m3(Lc8_t)            (512 f32 per head)
 * (The latent row serves as key and as value, and the row scale is applied outside the dot product:
 * [KV8] first commit.)
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers owned by the caller (unless stated).  The library allocates no
 *     memory, keeps no state between calls, never synchronises the device, and has no CPU
 *     fallback: an unsupported argument is an error code.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are asynchronous:
 *     a return of KV8_OK means the kernels were enqueued; results are valid once the stream has
 *     reached that point.
 *   - Validation happens on the host before any launch: on any error nothing is enqueued.
 *   - Device buffers must be 16-byte aligned (TMA and vector loads).  Inputs and outputs must not
 *     overlap, except where stated.
 *   - Return values: KV8_OK (0) or a negative KV8_E* code.  kv8_strerror() names it.
 *   - Device-side conditions (a selected index out of range, a wait that timed out) are OR-ed
 *     into *err_word (a device int, optional: may be NULL) as KV8_ERR_* bits; the caller clears it
 *     beforehand and reads it after synchronising.
 */
#ifndef KV8MLA_H
#define KV8MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KV8_API __attribute__((visibility("default")))
#else
#define KV8_API
#endif

#define KV8_ROW_BYTES 576      /* e4m3 bytes per cache row: Lc then Rc */
#define KV8_KL 512             /* kv_lora rank: latent width, also the context width */
#define KV8_KR 64              /* qk_rope width */
#define KV8_MAX_HEADS 128      /* query heads per call */
#define KV8_MAX_ROWS (1 << 20) /* rows per cache: the 1M cap of [KV8] second commit */
#define KV8_MAX_SELECT 4096    /* selected rows per sequence: NS <= 4096 ([KV8] second commit) */
#define KV8_NOPE 128           /* per-head no-position query / key width (kv_b_proj key rows per head) */
#define KV8_VHEAD 128          /* per-head value width (kv_b_proj value rows per head) */
#define KV8_KVB_BLOCK 128      /* fmt=8 scale block edge: one f32 scale per 128x128 weight block */
#define KV8_IDX_D 128          /* DSA indexer: index key / index query head width */
#define KV8_MAX_IDX_HEADS 128  /* DSA indexer: index heads per query (a multiple of 16) */
#define KV8_MX_NOPE 448        /* mixed cache: no-position values per row (e4m3 + row scale) */
#define KV8_MX_ROPE 64         /* mixed cache: RoPE values per row (bf16) */

/* return codes */
#define KV8_OK 0
#define KV8_EINVAL (-1)       /* null pointer, bad size, misalignment, or value outside the limits */
#define KV8_EWORKSPACE (-2)   /* workspace smaller than the matching *_workspace_bytes() */
#define KV8_ECUDA (-3)        /* a CUDA launch or attribute call failed */
#define KV8_EUNSUPPORTED (-4) /* the device is not sm_103 (or the shape has no kernel) */

/* bits OR-ed into *err_word by the device */
#define KV8_ERR_INDEX 1u    /* a selected row index was outside [0, T): that entry was skipped */
#define KV8_ERR_TIMEOUT 2u  /* a bounded wait in a kernel gave up: that output is not valid */

/* query element types */
#define KV8_F32 0
#define KV8_BF16 1

/* -----------------------------------------------------------------------------------------------
 * kv8_encode_e4m3 -- the element encoder of the row quantizer, without scaling.
 * [KV8] first commit, c/kv_fp8.h item: round to nearest, ties to even; saturate at +-448 (inf
 * included); keep the sign of zero (so -0.0 and negative values that round to zero give 0x80);
 * store NaN as 0x00.
 *   y   [n] f32 in, out [n] u8 out (byte i encodes y[i]).  n >= 0 (n == 0 enqueues nothing).
 *   Alignment: y 16-byte aligned, out 4-byte aligned.
 * --------------------------------------------------------------------------------------------- */
KV8_API int kv8_encode_e4m3(const float *y, int64_t n, uint8_t *out, void *stream);

/* -----------------------------------------------------------------------------------------------
 * kv8_quant_rows -- quantize n f32 rows into cache rows ([KV8] first commit: the producer
 * quantizes the fresh normed/roped row; per-row quantizer with a subnormal-amax guard).
 *   x        [n][576] f32 in (Lc then Rc for each row)
 *   kv8      [n][576] u8 out: pass the cache base + 576*t to write rows t..t+n-1
 *   kv_scale [n] f32 out:     pass the scale base + t
 * Per row, in f32 with IEEE round-to-nearest: amax = max |x_i| over finite x_i; scale = amax/448;
 * y_i = x_i * (448/amax), or, when 448/amax overflows (subnormal amax), (x_i*2^64)*(448/(amax*2^64));
 * when amax == 0, y_i = x_i.  byte_i = kv8_encode_e4m3(y_i).  Bit-exact with the oracle.
 *   n >= 0.  x and kv8 16-byte aligned, kv_scale 4-byte aligned.
 * --------------------------------------------------------------------------------------------- */
KV8_API int kv8_quant_rows(const float *x, int64_t n, uint8_t *kv8, float *kv_scale, void *stream);

/* kv8_quant_rows_w -- the same row quantizer for rows of `width` elements: width = KV8_ROW_BYTES (cache
 * rows, as kv8_quant_rows), KV8_IDX_D (DSA index keys) or KV8_MX_NOPE (mixed-cache no-position parts).  x [n][width] f32 -> q [n][width] e4m3,
 * scale [n] f32.  Any other width is KV8_EINVAL. */
KV8_API int kv8_quant_rows_w(const float *x, int64_t n, int width, uint8_t *q, float *scale, void *stream);

/* -----------------------------------------------------------------------------------------------
 * Split-T decode ([KV8] second commit: flash-decoding style partial online-softmax blocks
 * (cl[K], m, z) plus a log-sum-exp merge kernel; the cache is device-resident, only new rows are
 * uploaded).  One query of H heads over rows 0..T-1.
 *
 * Partition p of P covers rows [floor(T*p/P), floor(T*(p+1)/P)).  The workspace begins with the
 * partial sets (f32), for B batch items (B = 1 for decode):
 *     cl [B][P][H][512]   unnormalised context of each partition, relative to its m
 *     m  [B][P][H]        the partition's reference: the max of score * log2(e) over its rows, or a
 *                         value at most 2 below it (the online softmax rescales lazily); -inf for a
 *                         partition without rows
 *     z  [B][P][H]        sum over the partition of 2^(score*log2(e) - m)
 * The decode workspace continues with the library's own staging (the prepared queries); its size
 * is included in mla_decode8_workspace_bytes.
 * mla_decode8_partitions:      the partition count P the library uses for (H, T, P_req):
 *                              P_req = 0 picks automatically (one CTA per SM of the current device,
 *                              N SMs (152 on GB300; 152 when no device is visible): min(ceil(T/128),
 *                              N/2 for H > 64, else N)), P_req > 0 is clamped to [1, T].  The count
 *                              depends on the device current at the call: size and launch on one device.
 * mla_decode8_workspace_bytes: workspace bytes for (H, T, P_req).
 * --------------------------------------------------------------------------------------------- */
KV8_API int mla_decode8_partitions(int H, int64_t T, int P_req, int *P_out);
KV8_API int mla_decode8_workspace_bytes(int H, int64_t T, int P_req, size_t *bytes);

/* mla_decode8_partial -- the partial kernel alone (fills the workspace for P partitions).
 *   q_lat [H][512], q_rope [H][64] of type q_dtype (KV8_F32 or KV8_BF16), 16-byte aligned.
 *   H in [1, 128]; T in [1, KV8_MAX_ROWS]; kv8 [T][576], kv_scale [T].
 *   sm_scale: finite.  err_word: optional (KV8_ERR_TIMEOUT).
 *   workspace: >= mla_decode8_workspace_bytes(H, T, P_req) bytes. */
KV8_API int mla_decode8_partial(const void *q_lat, const void *q_rope, int q_dtype, int H, const uint8_t *kv8,
                        const float *kv_scale, int64_t T, float sm_scale, int P_req, void *workspace,
                        size_t ws_bytes, int *err_word, void *stream);

/* mla_lse_merge8 -- the log-sum-exp merge of B*H partial sets into out [B][H][512] f32:
 *   M = max_p m_p;  w_p = 2^(m_p - M) (0 when m_p = -inf);  Z = sum_p w_p z_p;
 *   out = sum_p w_p cl_p / Z   (0 when Z == 0, i.e. no row was attended).
 * workspace as written by the partial kernels; P in [1, 65535]. */
KV8_API int mla_lse_merge8(const void *workspace, int B, int P, int H, float *out, void *stream);

/* mla_absorb_decode8 -- partial + merge on one stream: out [H][512] f32 = cl for each head. */
KV8_API int mla_absorb_decode8(const void *q_lat, const void *q_rope, int q_dtype, int H, const uint8_t *kv8,
                       const float *kv_scale, int64_t T, float sm_scale, int P_req, void *workspace,
                       size_t ws_bytes, int *err_word, float *out, void *stream);

/* -----------------------------------------------------------------------------------------------
 * mla_absorb_sel8 -- DSA gather decode ([KV8] second commit: attention_absorb_sel_kernel8 attends
 * the selected rows straight from the device cache by absolute index, NS <= 4096; when a
 * selection is active decode attends exactly the selection).
 *   B sequences; sequence b's cache is rows [b*seq_stride_rows, b*seq_stride_rows + T) of
 *   kv8 / kv_scale (seq_stride_rows >= T, or 0 when B == 1).
 *   q_lat [B][H][512], q_rope [B][H][64] (q_dtype); idx [B][NS] int32 absolute row indices into
 *   the sequence's own cache (any order; duplicates attend twice).  An index outside [0, T) is
 *   skipped and sets KV8_ERR_INDEX in *err_word.  out [B][H][512] f32.
 *   NS in [1, KV8_MAX_SELECT]; T in [1, KV8_MAX_ROWS]; H in [1, 128]; B >= 1.
 *   workspace >= mla_sel8_workspace_bytes(B, H, NS): the B x P partial sets, then staging for the
 *   prepared bf16 queries.  P spreads the list's 128-row tiles over one wave of CTAs, one per SM (B items x
 *   P x ceil(H/64)).  bf16 queries run on the tensor cores, which gather the selected rows from all
 *   items' caches with 32-bit row coordinates; f32 queries, and caches with
 *   (B-1)*seq_stride_rows + T >= 2^31 rows, run on the CUDA cores.
 * --------------------------------------------------------------------------------------------- */
KV8_API int mla_sel8_workspace_bytes(int B, int H, int NS, size_t *bytes);
KV8_API int mla_absorb_sel8(const void *q_lat, const void *q_rope, int q_dtype, int B, int H, const uint8_t *kv8,
                    const float *kv_scale, int64_t T, int64_t seq_stride_rows, const int32_t *idx, int NS,
                    float sm_scale, void *workspace, size_t ws_bytes, int *err_word, float *out, void *stream);

/* -----------------------------------------------------------------------------------------------
 * mla_absorb_prefill8 -- causal prefill of S new queries ([KV8] first and second commits: the
 * batch/prefill absorb path, coli_cuda_attention_absorb_batch8, tiled streaming, cap 1M rows).
 * Query i sits at position pos0 + i and attends rows 0..pos0+i (row index = position); its own
 * fresh row must already be quantized into the cache (kv8_quant_rows).
 *   q_lat [S][H][512], q_rope [S][H][64] (q_dtype); out [S][H][512] f32.
 *   S >= 1; pos0 >= 0; pos0 + S <= T <= KV8_MAX_ROWS; H in [1, 128].
 * --------------------------------------------------------------------------------------------- */
KV8_API int mla_absorb_prefill8(const void *q_lat, const void *q_rope, int q_dtype, int S, int H, int64_t pos0,
                        const uint8_t *kv8, const float *kv_scale, int64_t T, float sm_scale, int *err_word,
                        float *out, void *stream);

/* -----------------------------------------------------------------------------------------------
 * mla_absorb_decode8_noalloc -- mla_absorb_decode8 for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists for users of this library.
 *
 * Some callers cannot call cudaMalloc or reach an allocator for the workspace that the split-T
 * partials need: a plugin loaded into a host program whose memory pool already owns the GPU's
 * memory, a caller from another language runtime with no handle on the host's caching allocator,
 * or a latency-critical loop that must not take cudaMalloc's implicit device synchronisation.
 * This entry point keeps the partials in a fixed array of KV8_NOALLOC_SCRATCH_BYTES that is part of
 * the library's device image: every GPU that loads the library holds it until the process exits.
 * Apart from that module load (below), neither this call nor anything it calls allocates memory.
 *
 * Arguments as mla_absorb_decode8, without workspace / ws_bytes.  P_req == 0 picks the automatic
 * partition count, lowered if needed until the partials fit the array; an explicit P_req whose
 * partials do not fit returns KV8_EWORKSPACE (nothing is enqueued).
 * Every call looks up the array's address in the current device's context (a cheap host query; no
 * address is kept between calls, so a context that was reset and created again is handled).  The
 * first call in a context also loads the library's device module, which places the array: that step
 * can allocate device memory and synchronise, and it fails with KV8_ECUDA if the device has no room
 * left.  A caller whose memory pool takes the whole GPU should therefore make one warm-up call per
 * device at set-up time, before the pool grows and before any stream capture.
 * All calls share the one array and it keeps the last call's contents (each call writes every
 * partial it reads, so nothing needs clearing): calls whose kernels overlap on the GPU (two streams,
 * or two host threads) race on it and must be ordered by the caller.
 * --------------------------------------------------------------------------------------------- */
#define KV8_NOALLOC_SCRATCH_BYTES (16u << 20) /* 16 MiB per device */
KV8_API int mla_absorb_decode8_noalloc(const void *q_lat, const void *q_rope, int q_dtype, int H,
                                       const uint8_t *kv8, const float *kv_scale, int64_t T, float sm_scale,
                                       int P_req, int *err_word, float *out, void *stream);

/* -----------------------------------------------------------------------------------------------
 * mla_absorb_mixed_decode8 -- decode over the mixed-precision cache ([B1] "B1 Mixed FP8/BF16 FMHA first
 * pass": the no-position part of each KV row stored as e4m3 with a per-row f32 scale, the RoPE part as
 * bf16, the query's no-position part quantized from bf16 to e4m3 before the attention; head width
 * 512 = KV8_MX_NOPE + KV8_MX_ROPE; the row is both key and value).  For each head h:
 *     (q8[h], q_scale[h]) = the row quantizer (amax/448) applied to q_nope[h]
 *     score[h][t] = sm_scale * ( q_scale[h] * k_scale[t] * e4m3(q8[h]).e4m3(k8[t]) + q_rope[h].k_rope[t] )
 *     out[h] = sum_t softmax_t(score[h]) * [ k_scale[t] * e4m3(k8[t]) , k_rope[t] ]        (512 f32)
 *   q_nope [H][448], q_rope [H][64] of type q_dtype; k8 [T][448] e4m3 (kv8_quant_rows_w, width 448),
 *   k_scale [T] f32, k_rope [T][64] bf16; out [H][512] f32.  H in [1, 128]; T in [1, KV8_MAX_ROWS].
 *   workspace: >= mla_mixed_decode8_workspace_bytes(H, T) (split-T partial sets as for mla_decode8_partial,
 *   merged by mla_lse_merge8 inside the call; then staging for the query prep).  k8 and k_rope 16-byte aligned.  err_word: optional
 *   (KV8_ERR_TIMEOUT).  Runs on the tensor cores: the no-position product as e4m3 x e4m3 and the RoPE
 *   product as bf16 x bf16 (an f32 RoPE query as bf16 hi + lo), f32 accumulation; the softmax weights
 *   enter the value product as e4m3 hi + lo (no-position values) and bf16 (RoPE values).
 * --------------------------------------------------------------------------------------------- */
KV8_API int mla_mixed_decode8_workspace_bytes(int H, int64_t T, size_t *bytes);
KV8_API int mla_absorb_mixed_decode8(const void *q_nope, const void *q_rope, int q_dtype, int H, const uint8_t *k8,
                                     const float *k_scale, const void *k_rope, int64_t T, float sm_scale,
                                     void *workspace, size_t ws_bytes, int *err_word, float *out, void *stream);

/* -----------------------------------------------------------------------------------------------
 * mla_absorb_batch_decode8 -- one decode step for B sequences at once, each with its own cache and length
 * ([KV8] second commit: a device-resident cache per sequence to which each step appends the new rows;
 * the split-T partials and log-sum-exp merge as for one sequence).
 *   Sequence b's cache is rows b*seq_stride_rows .. b*seq_stride_rows + T_max - 1 of kv8 / kv_scale; it
 *   attends its first lens[b] rows (lens: device int32 [B], clamped to [0, T_max]; 0 rows give a zero
 *   output).  q_lat [B][H][512], q_rope [B][H][64] of type q_dtype; out [B][H][512] f32.
 *   B >= 1; H in [1, 128]; T_max in [1, KV8_MAX_ROWS]; seq_stride_rows >= T_max when B > 1.
 *   workspace: >= mla_batch_decode8_workspace_bytes(B, H, T_max) bytes (partial sets [B][P][H] first, as
 *   for one sequence, then the prepared queries).  err_word: optional (KV8_ERR_TIMEOUT).
 * kv8_quant_rows_scatter -- kv8_quant_rows writing input row r to cache row dst_rows[r] (device int64 [n]),
 *   e.g. one fresh row appended to each sequence; a destination outside [0, cache_rows) is skipped and sets
 *   KV8_ERR_INDEX in *err_word (optional).
 * --------------------------------------------------------------------------------------------- */
KV8_API int mla_batch_decode8_workspace_bytes(int B, int H, int64_t T_max, size_t *bytes);
KV8_API int mla_absorb_batch_decode8(const void *q_lat, const void *q_rope, int q_dtype, int B, int H,
                                     const uint8_t *kv8, const float *kv_scale, int64_t T_max, int64_t seq_stride_rows,
                                     const int32_t *lens, float sm_scale, void *workspace, size_t ws_bytes,
                                     int *err_word, float *out, void *stream);
KV8_API int kv8_quant_rows_scatter(const float *x, int64_t n, const int64_t *dst_rows, uint8_t *kv8,
                                   float *kv_scale, int64_t cache_rows, int *err_word, void *stream);

/* -----------------------------------------------------------------------------------------------
 * Absorb projections through kv_b_proj stored as fmt=8 ([FMT8] "feat: fmt=8 (fp8-e4m3) decode on
 * the kv_b absorb path, CPU and CUDA": raw e4m3 bytes plus one f32 scale per 128x128 block,
 * block-row-major; the absorbed attention of [KV8] first commit works in the 512-wide latent).
 *   w8 [H*256][512] e4m3 bytes: head h's rows 256h..256h+127 are W_UK (no-position key part,
 *      KV8_NOPE), rows 256h+128..256h+255 are W_UV (value part, KV8_VHEAD).
 *   w_scale [H*2][4] f32: block (r, c) covers rows 128r.., columns 128c..; the weight is
 *      W[o][i] = e4m3(w8[o][i]) * w_scale[(o/128)*4 + i/128].
 * mla_q_absorb8:    q_lat[s][h][c] = sum_{j<128} q_nope[s][h][j] * W[256h + j][c]      (c < 512)
 *   q_nope [S][H][128] of type q_dtype; q_lat [S][H][512] of type out_dtype (KV8_F32 / KV8_BF16;
 *   bf16 rounds the f32 sum to nearest even) -- the query the decode / selection / prefill calls take.
 * mla_out_project8: out[s][h][v] = sum_{c<512} W[256h + 128 + v][c] * ctx[s][h][c]     (v < 128)
 *   ctx [S][H][512] f32 (a normalised context, e.g. mla_lse_merge8's out); out [S][H][128] f32.
 * Sums in f32 over exactly decoded weights; the block scale is applied per 128-column block.  Up to 8
 * rows run on the CUDA cores (the weights read once); more on the tensor cores (kind::f16: every e4m3
 * weight is a bf16; f32 activations as bf16 hi + lo pieces).  err_word: optional (KV8_ERR_TIMEOUT).
 * S in [1, KV8_MAX_ROWS]; H in [1, 128]; all buffers 16-byte aligned; outputs must not overlap inputs.
 * The kernels are programmatic dependents of the kernel launched before them on the stream: they start
 * reading w8 and w_scale while that kernel finishes, and q_nope / ctx only after it has completed.  So
 * w8 and w_scale must not be written by the kernel launched just before this call on the same stream.
 * --------------------------------------------------------------------------------------------- */
KV8_API int mla_q_absorb8(const void *q_nope, int q_dtype, int S, int H, const uint8_t *w8, const float *w_scale,
                          void *q_lat, int out_dtype, int *err_word, void *stream);
KV8_API int mla_out_project8(const float *ctx, int S, int H, const uint8_t *w8, const float *w_scale, float *out,
                             int *err_word, void *stream);

/* -----------------------------------------------------------------------------------------------
 * dsa_index_topk8 -- the DSA lightning indexer and its top-k ([B1] page, the commit adding
 * indexer_fp8_score_topk: an e4m3 index query of 64 heads x 128 quantized from bf16, e4m3 index keys
 * read as they are, the score dequantized by q_scale * k_scale, ReLU, weighted sum over the heads,
 * top-k).  For each of B queries b and each position t < T of its key rows t' = b*seq_stride_rows + t:
 *     I[b][t] = sum_h w[b][h] * max(0, q_scale[b][h] * k_scale[t'] * sum_i e4m3(q8[b][h][i]) e4m3(k8[t'][i]))
 * where (q8[b][h], q_scale[b][h]) is the row quantizer applied to q_idx[b][h] (amax/448 per head row).
 *   q_idx [B][HI][128] of type q_dtype (KV8_F32 / KV8_BF16); w [B][HI] f32 (either sign);
 *   k8 [rows][128] e4m3 and k_scale [rows] f32 as written by kv8_quant_rows_w(width = KV8_IDX_D).
 *   scores [B][T] f32 (written: I); idx [B][NS] int32 (written): the min(NS, T) positions with the
 *   largest scores, the smaller position first among equal scores, in ascending position order -- the
 *   selection list mla_absorb_sel8 takes.  When NS > T, idx[b][T..NS-1] is left as it was.
 *   HI a multiple of 16 in [16, KV8_MAX_IDX_HEADS]; T in [1, KV8_MAX_ROWS]; NS in [1, KV8_MAX_SELECT];
 *   seq_stride_rows >= 0 and (B-1)*seq_stride_rows + T < 2^31 - 128; buffers 16-byte aligned.
 *   workspace: >= dsa_index_workspace_bytes(B) bytes (the top-k's histograms and the barrier counters of
 *   the CTAs that share a query; zeroed by the call itself).  err_word: optional (KV8_ERR_TIMEOUT).
 *   The scores run on the tensor cores (e4m3 x e4m3, f32 sums); the top-k is one cooperative launch
 *   whose CTAs meet at time-bounded barriers (a barrier that gives up sets KV8_ERR_TIMEOUT).
 * --------------------------------------------------------------------------------------------- */
KV8_API int dsa_index_workspace_bytes(int B, size_t *bytes);
KV8_API int dsa_index_topk8(const void *q_idx, int q_dtype, const float *w, int B, int HI, const uint8_t *k8,
                            const float *k_scale, int64_t T, int64_t seq_stride_rows, int NS, void *workspace,
                            size_t ws_bytes, float *scores, int32_t *idx, int *err_word, void *stream);

/* -----------------------------------------------------------------------------------------------
 * kv8_copy -- copy `bytes` bytes from src to dst with a kernel (the SMs' loads and stores, not a
 * copy engine).  The pages have no counterpart to this call; it exists for users of this library:
 * on a GPU whose host memory is coherently attached (NVLink-C2C), it moves a step's small inputs
 * and outputs between page-locked host memory and the device with less fixed cost per transfer
 * than a copy-engine memcpy.
 *   dst, src: device memory of the current device, managed memory, or page-locked host memory
 *   (cudaHostAlloc / cudaMallocHost / cudaHostRegister), in any combination and any alignment
 *   (16-byte aligned pointers take the vector path).  The ranges must not overlap.
 *   Pageable host memory, another device's memory or an unknown pointer is KV8_EINVAL (checked
 *   with cudaPointerGetAttributes on the host; nothing is enqueued).  bytes == 0 enqueues nothing.
 *   Stream-ordered and asynchronous like every call.
 * --------------------------------------------------------------------------------------------- */
KV8_API int kv8_copy(void *dst, const void *src, size_t bytes, void *stream);

/* -----------------------------------------------------------------------------------------------
 * kv8_wait_selftest -- diagnostic of the timeout path.  One CTA waits on an mbarrier that nothing
 * completes, through the same bounded wait the library's tensor-core kernels use for their TMA, MMA and
 * softmax hand-offs.  After limit_ns (in [1000, 1e9] ns) the wait gives up: KV8_ERR_TIMEOUT is OR-ed into
 * *err_word, *wait_status is set to 2 (1 would mean the wait completed) and the kernel returns normally,
 * leaving the context usable.  err_word and wait_status: device ints (required).
 * --------------------------------------------------------------------------------------------- */
KV8_API int kv8_wait_selftest(uint64_t limit_ns, int *err_word, int *wait_status, void *stream);

/* Name of a return code (static string). */
KV8_API const char *kv8_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* KV8MLA_H */
