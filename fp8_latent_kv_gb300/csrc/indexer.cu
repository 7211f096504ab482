// indexer.cu -- the DSA lightning indexer: scores over e4m3 index keys, then top-k selection.
//
// Page "B1 Mixed FP8/BF16 FMHA first pass", the commit adding indexer_fp8_score_topk: the index query
// (64 heads of 128) is quantized from bf16 to e4m3, the index keys are read as e4m3, the score is
// dequantized with q_scale * k_scale, passed through a ReLU and summed over the heads with per-head
// weights, and the top-k positions become the selection.  Per query b and position t:
//     I[b][t] = k_scale[t'] * sum_h (w[b][h] * q_scale[b][h]) * max(0, sum_i q8[b][h][i] * k8[t'][i])
// (t' = b * seq_stride_rows + t; the scales are positive, so the ReLU commutes with them).
//
// score kernel: the scores are a dense e4m3 contraction (HI heads x 128 x T rows), so they run on the
// tensor cores: per 128-row key tile, S^T = K8 [Q8]^T with M = 128 rows, N = HI heads, K = 128 (four
// kind::f8f6f4 MMAs of K = 32) into one of four TMEM accumulators.  Warp 0 streams key tiles through
// six shared-memory stages with TMA, warp 1 issues the MMAs, warps 2..5 (one TMEM lane quadrant each)
// read a row's HI scores, apply the ReLU and weights and store the row's score.  The CTA quantizes its
// query's HI heads itself (same f32 steps as the row quantizer).  Every wait is bounded in time.
//
// top-k kernel: one CTA per query; a radix select over the scores' order-preserving 32-bit keys
// (11 + 11 + 10 bits) finds the k-th largest key, then an index-ordered pass keeps every larger score
// and, among scores equal to the k-th, the smallest positions -- written in ascending position order.
#include "internal.h"
#include "quant_row.cuh"
#include "sm100.cuh"

#include <cudaTypedefs.h>
#include <mutex>

namespace kv8 {
namespace {

using namespace sm100;

constexpr int kIdxD = KV8_IDX_D;  // 128 bytes per key row and per query head
constexpr int kITile = 128;       // key rows per tile (MMA M)
constexpr int kIStages = 6;
constexpr int kIAcc = 4;          // TMEM accumulator buffers
constexpr int kIThreads = 192;    // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr uint32_t kIStageBytes = kITile * kIdxD;  // 16 KB

struct IdxSmem {
    alignas(1024) uint8_t stage[kIStages][kIStageBytes];
    alignas(1024) uint8_t qimg[KV8_MAX_IDX_HEADS * kIdxD];  // B operand: HI rows of 128 bytes, 128B-swizzled
    alignas(16) float wq[KV8_MAX_IDX_HEADS];                // w[h] * q_scale[h]
    uint64_t full[kIStages], empty[kIStages], dfull[kIAcc], dempty[kIAcc], final_bar;
    uint32_t tmem_base;
    int abort_flag;
};

struct IdxArgs {
    const void *q;        // [B][HI][128] f32 or bf16
    int q_bf16;
    const float *w;       // [B][HI]
    int B, HI;
    const float *k_scale; // [rows]
    int64_t T, seq_stride_rows;
    int ctas_per_item;
    float *scores;        // [B][T]
    int *err_word;
};

__global__ void __launch_bounds__(kIThreads, 1) index_score_kernel(const __grid_constant__ CUtensorMap map_k, IdxArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    IdxSmem &sm = *reinterpret_cast<IdxSmem *>(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(smem) & 1023u) != 0) {  // swizzled operands need 1024-byte alignment
        if (tid == 0 && a.err_word) atomicOr(a.err_word, (int)KV8_ERR_TIMEOUT);
        return;
    }
    const int b = blockIdx.x / a.ctas_per_item, c = blockIdx.x - b * a.ctas_per_item;
    const int64_t n_tiles_item = (a.T + kITile - 1) / kITile;
    const int64_t i0 = n_tiles_item * c / a.ctas_per_item, i1 = n_tiles_item * (c + 1) / a.ctas_per_item;
    const int n_tiles = (int)(i1 - i0);
    const int HI = a.HI;
    const int64_t row_base = (int64_t)b * a.seq_stride_rows;
    // each accumulator starts at a power-of-two column: stride >= HI
    const uint32_t dstride = HI <= 16 ? 16u : HI <= 32 ? 32u : HI <= 64 ? 64u : 128u;
    const uint32_t ncols = dstride * kIAcc < 32u ? 32u : dstride * kIAcc;

    if (tid == 0) {
        for (int s = 0; s < kIStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int k = 0; k < kIAcc; ++k) {
            mbar_init(&sm.dfull[k], 1);
            mbar_init(&sm.dempty[k], 128);
        }
        mbar_init(&sm.final_bar, 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, ncols);
        tmem_relinquish();
    }
    // the query image: warps 2..5 quantize the HI heads of query b (one warp per head row at a time;
    // lane l takes elements 4l..4l+3), exactly as the row quantizer does
    if (warp >= 2) {
        for (int h = warp - 2; h < HI; h += 4) {
            float4 v;
            const int64_t e = ((int64_t)b * HI + h) * kIdxD + 4 * lane;
            if (a.q_bf16) {
                const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(a.q) + e));
                const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
                const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
                v = make_float4(f0.x, f0.y, f1.x, f1.y);
            } else {
                v = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(a.q) + e));
            }
            float amax = 0.f;
            amax = finite_abs_max(amax, v.x);
            amax = finite_abs_max(amax, v.y);
            amax = finite_abs_max(amax, v.z);
            amax = finite_abs_max(amax, v.w);
            amax = warp_max(amax);
            float pre, mul, qs;
            row_quant_factors(amax, pre, mul, qs);
            *reinterpret_cast<uint32_t *>(sm.qimg + sw128_offset(h, 4 * lane)) = enc4(scale4(v, pre, mul));
            if (lane == 0) sm.wq[h] = __ldg(a.w + (int64_t)b * HI + h) * qs;
        }
        fence_proxy_async_smem();  // the MMAs read the image through the async proxy
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ================================ TMA producer ================================
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&map_k);
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % kIStages;
                if (i >= kIStages &&
                    !mbar_wait(&sm.empty[s], ((i / kIStages) - 1) & 1, &sm.abort_flag, a.err_word))
                    break;
                mbar_arrive_expect_tx(&sm.full[s], kIStageBytes);
                tma_load_2d(sm.stage[s], &map_k, 0, (int32_t)(row_base + (i0 + i) * kITile), &sm.full[s]);
                issued = i + 1;
            }
            // every issued copy lands before the CTA ends
            for (int i = issued > kIStages ? issued - kIStages : 0; i < issued; ++i)
                mbar_wait(&sm.full[i % kIStages], (i / kIStages) & 1, nullptr, a.err_word, 200000000ull);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ================================ MMA issuer ================================
        if (lane == 0 && n_tiles > 0) {
            const uint32_t idesc = idesc_e4m3_f32(kITile, HI, false, false);
            const uint32_t qb = smem_u32(sm.qimg);
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % kIStages, buf = i % kIAcc;
                if (!mbar_wait(&sm.full[s], (i / kIStages) & 1, &sm.abort_flag, a.err_word)) break;
                if (i >= kIAcc && !mbar_wait(&sm.dempty[buf], ((i / kIAcc) - 1) & 1, &sm.abort_flag, a.err_word))
                    break;
                tc_fence_after_sync();
                const uint32_t st = smem_u32(sm.stage[s]);
                const uint32_t d = tmem + (uint32_t)buf * dstride;
#pragma unroll
                for (int kk = 0; kk < kIdxD / 32; ++kk)
                    mma_f8f6f4(d, smem_desc(st + kk * 32, 0, 1024, kSw128), smem_desc(qb + kk * 32, 0, 1024, kSw128),
                               idesc, kk > 0);
                mma_commit(&sm.empty[s]);
                mma_commit(&sm.dfull[buf]);
            }
            mma_commit(&sm.final_bar);
            mbar_wait(&sm.final_bar, 0, nullptr, a.err_word, 200000000ull);
        }
        __syncwarp();
    } else {
        // ================================ epilogue ================================
        const int q = warp & 3;  // TMEM lane quadrant
        const int r = q * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        bool ok = true;
        for (int i = 0; i < n_tiles && ok; ++i) {
            const int buf = i % kIAcc;
            ok = mbar_wait(&sm.dfull[buf], (i / kIAcc) & 1, &sm.abort_flag, a.err_word);
            if (!ok) break;
            tc_fence_after_sync();
            float acc = 0.f;
            for (int h0 = 0; h0 < HI; h0 += 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(tmem + lane_addr + (uint32_t)buf * dstride + (uint32_t)h0, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) acc = fmaf(sm.wq[h0 + j], fmaxf(__uint_as_float(v[j]), 0.f), acc);
            }
            tc_fence_before_sync();
            mbar_arrive(&sm.dempty[buf]);
            const int64_t t = (i0 + i) * kITile + r;
            if (t < a.T) a.scores[(int64_t)b * a.T + t] = __ldg(a.k_scale + row_base + t) * acc;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, ncols);
}

// ------------------------------------------------------------------------------------------------
// top-k: one CTA of 1024 threads per query
// ------------------------------------------------------------------------------------------------
constexpr int kKThreads = 1024;
constexpr int kKBins = 2048;

// order-preserving key: larger float -> larger unsigned key (-0 sorts just below +0)
__device__ __forceinline__ uint32_t fkey(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one value per thread (1024 threads); returns the exclusive prefix and
// writes the total to *total.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *warp_sums, uint32_t *total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const uint32_t before = (warp > 0 ? warp_sums[warp - 1] : 0u) + x - v;
    *total = warp_sums[31];
    __syncthreads();  // warp_sums may be reused by the caller's next scan
    return before;
}

__global__ void __launch_bounds__(kKThreads, 1) topk_kernel(const float *__restrict__ scores, int64_t T, int NS,
                                                           int32_t *__restrict__ idx) {
    __shared__ uint32_t hist[kKBins];
    __shared__ uint32_t warp_sums[32];
    __shared__ uint32_t sh_bin, sh_need;
    const int tid = threadIdx.x;
    const int b = blockIdx.x;
    const float *s = scores + (int64_t)b * T;
    int32_t *out = idx + (int64_t)b * NS;
    const uint32_t k = (uint32_t)((int64_t)NS < T ? NS : T);

    // ---- radix select: prefix / mask of the k-th largest key, `need` = how many of the keys equal to it
    // (after the last pass) still belong to the top k
    uint32_t prefix = 0, mask = 0, need = k;
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int p = 0; p < 3; ++p) {
        const int shift = shifts[p];
        const uint32_t nb = 1u << widths[p];
        for (int i = tid; i < kKBins; i += kKThreads) hist[i] = 0;
        __syncthreads();
        for (int64_t t = tid; t < T; t += kKThreads) {
            const uint32_t key = fkey(__ldg(s + t));
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
        }
        __syncthreads();
        // bins from the top: thread j holds bins nb-1-2j and nb-2-2j (in descending order)
        uint32_t c0 = 0, c1 = 0;
        const int j0 = (int)nb - 1 - 2 * tid, j1 = j0 - 1;
        if (j0 >= 0) c0 = hist[j0];
        if (j1 >= 0) c1 = hist[j1];
        uint32_t total;
        const uint32_t above = block_exclusive_scan(c0 + c1, warp_sums, &total);
        // the bin where the running count from the top reaches `need`
        if (j0 >= 0 && above < need && above + c0 >= need) {
            sh_bin = (uint32_t)j0;
            sh_need = need - above;
        } else if (j1 >= 0 && above + c0 < need && above + c0 + c1 >= need) {
            sh_bin = (uint32_t)j1;
            sh_need = need - above - c0;
        }
        __syncthreads();
        prefix |= sh_bin << shift;
        mask |= (nb - 1) << shift;
        need = sh_need;
        __syncthreads();
    }
    const uint32_t thr = prefix;  // the k-th largest key; `need` of the keys equal to it are taken

    // ---- index-ordered selection: thread j owns positions [j*C, (j+1)*C)
    const int64_t C = (T + kKThreads - 1) / kKThreads;
    const int64_t t0 = (int64_t)tid * C, t1 = t0 + C < T ? t0 + C : T;
    uint32_t n_gt = 0, n_eq = 0;
    for (int64_t t = t0; t < t1; ++t) {
        const uint32_t key = fkey(__ldg(s + t));
        n_gt += key > thr;
        n_eq += key == thr;
    }
    uint32_t tot;
    const uint32_t eq_before = block_exclusive_scan(n_eq, warp_sums, &tot);
    const uint32_t eq_take = eq_before >= need ? 0u : (need - eq_before < n_eq ? need - eq_before : n_eq);
    const uint32_t pos0 = block_exclusive_scan(n_gt + eq_take, warp_sums, &tot);
    uint32_t pos = pos0, eq_used = 0;
    for (int64_t t = t0; t < t1; ++t) {
        const uint32_t key = fkey(__ldg(s + t));
        if (key > thr || (key == thr && eq_used < eq_take)) {
            if (key == thr) ++eq_used;
            if (pos < k) out[pos] = (int32_t)t;
            ++pos;
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 index_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

cudaError_t launch_index_scores(const void *q, int q_bf16, const float *w, int B, int HI, const uint8_t *k8,
                                const float *k_scale, int64_t T, int64_t seq_stride_rows, float *scores,
                                int *err_word, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = index_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const int64_t rows = (int64_t)(B - 1) * seq_stride_rows + T;
    if (rows > 0x7fffffffLL - kITile) return cudaErrorInvalidValue;  // tensor-map row coordinates are 32-bit
    CUtensorMap m;
    const cuuint64_t dims[2] = {(cuuint64_t)kIdxD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kIdxD};
    const cuuint32_t box[2] = {(cuuint32_t)kIdxD, (cuuint32_t)kITile}, es[2] = {1, 1};
    if (encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(k8), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    IdxArgs a{};
    a.q = q;
    a.q_bf16 = q_bf16;
    a.w = w;
    a.B = B;
    a.HI = HI;
    a.k_scale = k_scale;
    a.T = T;
    a.seq_stride_rows = seq_stride_rows;
    a.ctas_per_item = B >= 152 ? 1 : 152 / B;  // one wave of CTAs (one per SM of a 152-SM part)
    a.scores = scores;
    a.err_word = err_word;
    const size_t smem = sizeof(IdxSmem);
    cudaError_t e = cudaFuncSetAttribute(index_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    index_score_kernel<<<(unsigned)(B * a.ctas_per_item), kIThreads, smem, st>>>(m, a);
    return cudaGetLastError();
}

cudaError_t launch_topk(const float *scores, int B, int64_t T, int NS, int32_t *idx, cudaStream_t st) {
    topk_kernel<<<(unsigned)B, kKThreads, 0, st>>>(scores, T, NS, idx);
    return cudaGetLastError();
}

}  // namespace kv8
