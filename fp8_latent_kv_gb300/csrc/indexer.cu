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
// twelve shared-memory stages with TMA, warp 1 issues the MMAs, warps 2..9 (two groups of four, one TMEM
// lane quadrant per warp, taking alternate tiles) read a row's HI scores, apply the ReLU and weights and
// store the row's score.  The CTA quantizes its query's HI heads itself (same f32 steps as the row
// quantizer).  Every wait is bounded in time.
//
// top-k kernel: a radix select over the scores' order-preserving 32-bit keys (11 + 11 + 10 bits) finds
// the k-th largest key, then an index-ordered pass keeps every larger score and, among scores equal to
// the k-th, the smallest positions -- written in ascending position order.  Each query's positions are
// split over several CTAs of one cooperative launch that meet at bounded barriers; the launch is a
// programmatic dependent of the score kernel.
#include "internal.h"
#include "quant_row.cuh"
#include "sm100.cuh"

#include <cudaTypedefs.h>

namespace kv8 {
namespace {

using namespace sm100;

constexpr int kIdxD = KV8_IDX_D;  // 128 bytes per key row and per query head
constexpr int kITile = 128;       // key rows per tile (MMA M)
constexpr int kIStages = 12;
constexpr int kIAcc = 4;          // TMEM accumulator buffers
constexpr int kIThreads = 320;    // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue (two groups of four)
constexpr uint32_t kIStageBytes = kITile * kIdxD;  // 16 KB

// top-k workspace layout and key order (the score kernel also builds the first radix pass's histogram)
constexpr int kKThreads = 512;
constexpr int kKBins = 2048;
constexpr int kKMaxC = 152;
constexpr int kKCache = 8192;  // a CTA's scores staged in shared memory when its range is this short
// unused dynamic shared memory that keeps the top-k at one CTA per SM: launched early behind the score
// kernel, its CTAs would otherwise pack four to each of the first SMs that score CTAs leave
constexpr int kKPadSmem = 80 * 1024;
// per-query workspace (u32): three pass histograms, per-CTA (above, equal) counts, barrier counter
constexpr int kKWsHist = 3 * kKBins;
constexpr int kKWsPerItem = kKWsHist + 2 * kKMaxC + 32;

// order-preserving key: larger float -> larger unsigned key (-0 sorts just below +0)
__device__ __forceinline__ uint32_t fkey(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct IdxSmem {
    alignas(1024) uint8_t stage[kIStages][kIStageBytes];
    alignas(1024) uint8_t qimg[KV8_MAX_IDX_HEADS * kIdxD];  // B operand: HI rows of 128 bytes, 128B-swizzled
    alignas(16) float wq[KV8_MAX_IDX_HEADS];                // w[h] * q_scale[h]
    uint32_t hist0[kKBins];                                 // the CTA's keys by their top 11 bits (radix pass 0)
    uint64_t full[kIStages], empty[kIStages], dfull[kIAcc], dempty[kIAcc], final_bar, qready;
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
    uint32_t *hist0;      // top-k workspace: each item's pass-0 histogram gets this kernel's counts, or null
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

    // The first epilogue group's warps load the query head rows and weights first, before any key tile
    // is requested: issued behind the key stream they would wait for it.  Lane j holds the weight of the
    // warp's j-th head row; lane l holds elements 4l..4l+3 of each row, as raw bits (f32: 16 bytes, bf16:
    // 8 bytes in .x and .y) converted only where they are quantized, so that every load is in flight at
    // once -- converting each row as it arrives took one memory round trip per row.
    constexpr int kRowsPerWarp = KV8_MAX_IDX_HEADS / 4;
    static_assert(kRowsPerWarp <= 32, "one head weight per lane");
    uint4 qraw[kRowsPerWarp];
    float w_lane = 0.f;
    if (warp >= 2 && warp < 6) {
        const int hw = warp - 2 + 4 * lane;
        if (lane < kRowsPerWarp && hw < a.HI) w_lane = __ldg(a.w + (int64_t)b * a.HI + hw);
#pragma unroll
        for (int j = 0; j < kRowsPerWarp; ++j) {
            const int h = warp - 2 + 4 * j;
            qraw[j] = make_uint4(0u, 0u, 0u, 0u);
            if (h < a.HI) {
                const int64_t e = ((int64_t)b * a.HI + h) * kIdxD + 4 * lane;
                if (a.q_bf16) {
                    const uint2 r2 = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(a.q) + e));
                    qraw[j] = make_uint4(r2.x, r2.y, 0u, 0u);
                } else {
                    qraw[j] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(a.q) + e));
                }
            }
        }
    }
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
        mbar_init(&sm.qready, 128);  // the first epilogue group has written the query image and weights
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, ncols);
        tmem_relinquish();
    }
    for (int i = tid; i < kKBins; i += kIThreads) sm.hist0[i] = 0u;
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    // the top-k kernel may be launched now: it waits for this grid to complete before it reads anything
    grid_launch_dependents();

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
            const bool q_ok = mbar_wait(&sm.qready, 0, &sm.abort_flag, a.err_word);
            for (int i = 0; i < n_tiles && q_ok; ++i) {
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
        // Two groups of four warps take alternate tiles (group g: tiles g, g + 2, ...; its accumulators
        // are buffers g and g + 2), so one group reads back a tile while the other waits for the next.
        // First the query image (its rows were loaded at the top of the kernel): warp w of the first group
        // quantizes head rows w-2, w+2, ... (lane l takes elements 4l..4l+3) with the row quantizer's f32
        // steps; the second group waits for it.
        const int grp = (warp - 2) >> 2;
        if (grp == 0) {
#pragma unroll
            for (int j = 0; j < kRowsPerWarp; ++j) {
                const int h = warp - 2 + 4 * j;
                if (h >= HI) break;
                float4 vj;
                if (a.q_bf16) {
                    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qraw[j].x));
                    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qraw[j].y));
                    vj = make_float4(f0.x, f0.y, f1.x, f1.y);
                } else {
                    vj = make_float4(__uint_as_float(qraw[j].x), __uint_as_float(qraw[j].y), __uint_as_float(qraw[j].z),
                                     __uint_as_float(qraw[j].w));
                }
                float amax = 0.f;
                amax = finite_abs_max(amax, vj.x);
                amax = finite_abs_max(amax, vj.y);
                amax = finite_abs_max(amax, vj.z);
                amax = finite_abs_max(amax, vj.w);
                amax = warp_max(amax);
                float pre, mul, qs;
                row_quant_factors(amax, pre, mul, qs);
                *reinterpret_cast<uint32_t *>(sm.qimg + sw128_offset(h, 4 * lane)) = enc4(scale4(vj, pre, mul));
                const float wj = __shfl_sync(0xffffffffu, w_lane, j);
                if (lane == 0) sm.wq[h] = wj * qs;
            }
            fence_proxy_async_smem();  // the MMAs read the image through the async proxy
            named_sync(1, 128);  // wq complete for this group's threads
            mbar_arrive(&sm.qready);
        }
        bool ok = grp == 0 || n_tiles <= 1 || mbar_wait(&sm.qready, 0, &sm.abort_flag, a.err_word);
        const int q = warp & 3;  // TMEM lane quadrant
        const int r = q * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        // the row's key scale, loaded one tile ahead so its latency hides behind the previous tile
        auto kscale = [&](int i) -> float {
            const int64_t t = (i0 + i) * kITile + r;
            return (i < n_tiles && t < a.T) ? __ldg(a.k_scale + row_base + t) : 0.f;
        };
        float ks_next = kscale(grp);
        for (int i = grp; i < n_tiles && ok; i += 2) {
            const int buf = i % kIAcc;
            const float ks = ks_next;
            ks_next = kscale(i + 2);
            ok = mbar_wait(&sm.dfull[buf], (i / kIAcc) & 1, &sm.abort_flag, a.err_word);
            if (!ok) break;
            tc_fence_after_sync();
            float acc = 0.f;
            for (int h0 = 0; h0 < HI; h0 += 64) {
                // up to 64 columns in flight, one wait
                uint32_t v[4][16];
                const uint32_t ta = tmem + lane_addr + (uint32_t)buf * dstride + (uint32_t)h0;
                const int nq = (HI - h0) >= 64 ? 4 : (HI - h0) / 16;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq)
                    if (qq < nq) tmem_ld_32x32b_x16(ta + 16u * qq, v[qq]);
                tmem_wait_ld();
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    if (qq >= nq) break;
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const float4 wq = *reinterpret_cast<const float4 *>(&sm.wq[h0 + 16 * qq + 4 * j4]);
                        acc = fmaf(wq.x, fmaxf(__uint_as_float(v[qq][4 * j4 + 0]), 0.f), acc);
                        acc = fmaf(wq.y, fmaxf(__uint_as_float(v[qq][4 * j4 + 1]), 0.f), acc);
                        acc = fmaf(wq.z, fmaxf(__uint_as_float(v[qq][4 * j4 + 2]), 0.f), acc);
                        acc = fmaf(wq.w, fmaxf(__uint_as_float(v[qq][4 * j4 + 3]), 0.f), acc);
                    }
                }
            }
            tc_fence_before_sync();
            mbar_arrive(&sm.dempty[buf]);
            const int64_t t = (i0 + i) * kITile + r;
            if (t < a.T) {
                const float sv = ks * acc;
                a.scores[(int64_t)b * a.T + t] = sv;
                atomicAdd(&sm.hist0[fkey(sv) >> 21], 1u);  // the top-k's first radix digit
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (a.hist0)
        for (int i = tid; i < kKBins; i += kIThreads)
            if (sm.hist0[i]) atomicAdd(&a.hist0[(int64_t)b * kKWsPerItem + i], sm.hist0[i]);
    if (warp == 1) tmem_dealloc(tmem, ncols);
}

// ------------------------------------------------------------------------------------------------
// top-k: C CTAs per query (a cooperative launch: all CTAs resident), CTA c owning positions
// [c*T/C, (c+1)*T/C).  Pass 0's histogram (the keys' top 11 bits) comes complete from the score kernel.
// Passes 1 and 2: a shared histogram of the CTA's candidates (plain shared atomics; grouping equal bins
// with __match_any_sync first was slower), added once into the query's global histogram; a barrier of the
// query's C CTAs.  After each pass every CTA finds the pass's bin from the global histogram.  The final pass counts keys above / equal to the k-th key
// per CTA, and after a last barrier each CTA writes its selected positions at their global offsets.
// ------------------------------------------------------------------------------------------------
// Block-wide exclusive scan of one value per thread; returns the prefix, *total gets the sum.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *warp_sums, uint32_t *total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < nw ? warp_sums[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const uint32_t before = (warp > 0 ? warp_sums[warp - 1] : 0u) + x - v;
    *total = warp_sums[nw - 1];
    __syncthreads();  // warp_sums is reused by the next scan
    return before;
}

// Barrier of the C CTAs of one query: arrive on the query's counter, wait (bounded) until it reaches
// `target`.  A wait that gives up sets KV8_ERR_TIMEOUT and returns false; the CTA then stops.
__device__ bool query_barrier(uint32_t *ctr, uint32_t target, int *err_word, int *abort_sh) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        const uint64_t t0 = globaltimer_ns();
        while (*reinterpret_cast<volatile uint32_t *>(ctr) < target) {
            if (globaltimer_ns() - t0 > 1000000000ull) {  // 1 s
                if (err_word) atomicOr(err_word, (int)KV8_ERR_TIMEOUT);
                *abort_sh = 1;
                break;
            }
            __nanosleep(100);
        }
        __threadfence();
    }
    __syncthreads();
    return *abort_sh == 0;
}

__global__ void __launch_bounds__(kKThreads) topk_kernel(const float *__restrict__ scores, int64_t T, int NS, int C,
                                                          int32_t *__restrict__ idx, uint32_t *__restrict__ ws,
                                                          int *err_word) {
    __shared__ uint32_t hist[kKBins];
    __shared__ uint32_t warp_sums[32];
    __shared__ uint32_t sh_bin, sh_need;
    __shared__ int abort_sh;
    __shared__ uint32_t keys_sh[kKCache];
    const int tid = threadIdx.x;
    const int b = blockIdx.x / C, c = blockIdx.x - b * C;
    const float *s = scores + (int64_t)b * T;
    int32_t *out = idx + (int64_t)b * NS;
    uint32_t *wsb = ws + (size_t)b * kKWsPerItem;
    uint32_t *ghist = wsb, *gcnt = wsb + kKWsHist, *gbar = wsb + kKWsHist + 2 * kKMaxC;
    const uint32_t k = (uint32_t)((int64_t)NS < T ? NS : T);
    const int64_t c0 = T * c / C, c1 = T * (c + 1) / C;
    if (tid == 0) abort_sh = 0;
    // launched as a programmatic dependent of the score kernel: its scores and pass-0 histogram are
    // complete and visible once this returns
    grid_dependency_wait();
    // the CTA's keys, staged once when they fit (every pass below reads them again)
    const bool cached = c1 - c0 <= kKCache;
    if (cached)
        for (int64_t t = c0 + tid; t < c1; t += kKThreads) keys_sh[t - c0] = fkey(__ldg(s + t));
    __syncthreads();
    auto key_at = [&](int64_t t) -> uint32_t { return cached ? keys_sh[t - c0] : fkey(__ldg(s + t)); };

    uint32_t prefix = 0, mask = 0, need = k;
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int p = 0; p < 3; ++p) {
        const int shift = shifts[p];
        const uint32_t nb = 1u << widths[p];
        // pass 0's histogram was built by the score kernel (complete: it ran before this grid)
        if (p > 0) {
            for (int i = tid; i < kKBins; i += kKThreads) hist[i] = 0;
            __syncthreads();
            for (int64_t t0 = c0; t0 < c1; t0 += kKThreads) {
                const int64_t t = t0 + tid;
                const bool in = t < c1;
                const uint32_t key = in ? key_at(t) : 0u;
                const bool cand = in && (key & mask) == prefix;
                if (cand) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
            }
            __syncthreads();
            for (int i = tid; i < (int)nb; i += kKThreads)
                if (hist[i]) atomicAdd(&ghist[p * kKBins + i], hist[i]);
            if (!query_barrier(gbar, (uint32_t)p * (uint32_t)C, err_word, &abort_sh)) return;
        }
        // the bin where the count from the top reaches `need`: thread j holds 4 bins in descending order
        uint32_t cnt[4], sum = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int bi = (int)nb - 1 - (4 * tid + u);
            cnt[u] = bi >= 0 ? __ldcg(&ghist[p * kKBins + bi]) : 0u;
            sum += cnt[u];
        }
        uint32_t total;
        uint32_t above = block_exclusive_scan(sum, warp_sums, &total);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int bi = (int)nb - 1 - (4 * tid + u);
            if (bi >= 0 && above < need && above + cnt[u] >= need) {
                sh_bin = (uint32_t)bi;
                sh_need = need - above;
            }
            above += cnt[u];
        }
        __syncthreads();
        prefix |= sh_bin << shift;
        mask |= (nb - 1) << shift;
        need = sh_need;
        __syncthreads();
    }
    const uint32_t thr = prefix;  // the k-th largest key; `need` of the keys equal to it are taken

    // ---- positions in order: thread j of CTA c owns a contiguous sub-range of the CTA's range
    const int64_t per = (c1 - c0 + kKThreads - 1) / kKThreads;
    const int64_t t0 = c0 + (int64_t)tid * per, t1 = t0 + per < c1 ? t0 + per : c1;
    uint32_t n_gt = 0, n_eq = 0;
    for (int64_t t = t0; t < t1; ++t) {
        const uint32_t key = key_at(t);
        n_gt += key > thr;
        n_eq += key == thr;
    }
    uint32_t cta_gt, cta_eq;
    const uint32_t gt_before = block_exclusive_scan(n_gt, warp_sums, &cta_gt);
    const uint32_t eq_before = block_exclusive_scan(n_eq, warp_sums, &cta_eq);
    if (tid == 0) {
        gcnt[2 * c] = cta_gt;
        gcnt[2 * c + 1] = cta_eq;
    }
    if (!query_barrier(gbar, 3u * (uint32_t)C, err_word, &abort_sh)) return;
    // over the query's earlier CTAs: every count loaded at once (a lane per CTA, all in flight), then a
    // warp sum -- a loop of dependent adds would wait for one round trip per earlier CTA
    if (tid < 32) {
        uint32_t g = 0, e = 0;
#pragma unroll
        for (int u = 0; u < (kKMaxC + 31) / 32; ++u) {
            const int cc = tid + 32 * u;
            const bool in = cc < c;
            const uint32_t gv = in ? __ldcg(&gcnt[2 * cc]) : 0u, ev = in ? __ldcg(&gcnt[2 * cc + 1]) : 0u;
            g += gv;
            e += ev;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            e += __shfl_xor_sync(0xffffffffu, e, o);
        }
        if (tid == 0) {
            warp_sums[0] = g;
            warp_sums[1] = e;
        }
    }
    __syncthreads();
    const uint32_t gt_prev = warp_sums[0], eq_prev = warp_sums[1];
    __syncthreads();  // warp_sums is reused by the next scan
    const uint32_t eq_all_before = eq_prev + eq_before;
    const uint32_t eq_take = eq_all_before >= need ? 0u : (need - eq_all_before < n_eq ? need - eq_all_before : n_eq);
    const uint32_t eq_taken_prev = eq_prev < need ? eq_prev : need;  // equals taken by earlier CTAs
    uint32_t tot;
    const uint32_t pos_in_cta = block_exclusive_scan(n_gt + eq_take, warp_sums, &tot);
    uint32_t pos = gt_prev + eq_taken_prev + pos_in_cta, eq_used = 0;
    (void)gt_before;
    for (int64_t t = t0; t < t1; ++t) {
        const uint32_t key = key_at(t);
        if (key > thr || (key == thr && eq_used < eq_take)) {
            if (key == thr) ++eq_used;
            if (pos < k) out[pos] = (int32_t)t;
            ++pos;
        }
    }
}

}  // namespace

cudaError_t launch_index_scores(const void *q, int q_bf16, const float *w, int B, int HI, const uint8_t *k8,
                                const float *k_scale, int64_t T, int64_t seq_stride_rows, float *scores,
                                void *topk_ws, int *err_word, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
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
    const int sms = device_sm_count();
    a.ctas_per_item = B >= sms ? 1 : sms / B;  // one wave of CTAs (one per SM of the current device)
    a.scores = scores;
    a.hist0 = static_cast<uint32_t *>(topk_ws);
    a.err_word = err_word;
    const size_t smem = sizeof(IdxSmem);
    cudaError_t e = cudaFuncSetAttribute(index_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    index_score_kernel<<<(unsigned)(B * a.ctas_per_item), kIThreads, smem, st>>>(m, a);
    return cudaGetLastError();
}

size_t topk_workspace_bytes(int B) { return (size_t)B * kKWsPerItem * sizeof(uint32_t); }

cudaError_t reset_topk_workspace(void *ws, int B, cudaStream_t st) {
    return cudaMemsetAsync(ws, 0, topk_workspace_bytes(B), st);
}

cudaError_t launch_topk(const float *scores, int B, int64_t T, int NS, int32_t *idx, void *ws, int *err_word,
                        cudaStream_t st) {
    cudaError_t e;
    const int cmax = min(kKMaxC, device_sm_count());  // one CTA per SM: the grid barriers need them all resident
    const int C = B >= cmax ? 1 : cmax / B;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * C));
    cfg.blockDim = dim3(kKThreads);
    cfg.dynamicSmemBytes = kKPadSmem;
    cfg.stream = st;
    e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kKPadSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;  // the CTAs of a query wait for one another
    attr[0].val.cooperative = C > 1 ? 1 : 0;
    // a programmatic dependent of the score kernel: its launch overlaps that kernel's tail
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, topk_kernel, scores, T, NS, C, idx, static_cast<uint32_t *>(ws), err_word);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kv8
