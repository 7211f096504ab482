// proj8_tc.cu -- the absorb projections for many query rows (prefill chunks) on the tensor cores.
//
// Same operations as proj8.cu (page "feat: fmt=8 (fp8-e4m3) decode on the kv_b absorb path, CPU and
// CUDA": kv_b as e4m3 bytes with one f32 scale per 128x128 block; head h's rows 256h.. are W_UK, rows
// 256h+128.. are W_UV):
//   q absorb:     q_lat[s][h][c] = sum_j q_nope[s][h][j] * W[256h + j][c]
//   out project:  out[s][h][v]   = sum_c W[256h + 128 + v][c] * ctx[s][h][c]
// Every e4m3 value is exactly a bf16, so the weights enter a tcgen05.mma.kind::f16 (bf16 x bf16, f32
// accumulate in TMEM) unchanged; the block scales are applied to the f32 sums.  bf16 queries are used as
// they are; f32 queries and the f32 context are split into bf16 hi + lo pieces (two MMAs each), so the
// products match f32 arithmetic to ~2^-17 relative.
//
// One CTA per head (256 threads, phases separated by block barriers): the head's weight block is decoded
// once into shared memory as K-major 128-byte-swizzled bf16 rows; 128-row tiles of the activations are
// staged the same way; one thread issues the MMAs, every thread waits on the commit (bounded), and the
// eight warps read the accumulators back (lane quadrant = warp % 4, column half = warp / 4).
#include "internal.h"
#include "sm100.cuh"

namespace kv8 {
namespace {

using namespace sm100;

constexpr int kNope = KV8_NOPE, kVH = KV8_VHEAD, kKvbRows = kNope + kVH, kBlk = 128, kNbc = kKL / kBlk;
constexpr int kPT = 128;          // activation rows per tile (MMA M)
constexpr int kPThreads = 256;
constexpr uint32_t kKB = 64;      // bf16 elements per 128-byte swizzled row segment (one K block)

__device__ __forceinline__ uint32_t bf16_bits(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// four e4m3 bytes -> two words of bf16 pairs (exact: e4m3 values are bf16 values)
__device__ __forceinline__ uint2 e4m3x4_to_bf16x4(uint32_t w) {
    float e0, e1, e2, e3;
    e4m3x4_to_f32(w, e0, e1, e2, e3);
    return make_uint2(bf16_bits(e0) | (bf16_bits(e1) << 16), bf16_bits(e2) | (bf16_bits(e3) << 16));
}

// byte offset of bf16 element (row, k) in K-major 128-byte-swizzled K blocks of `rows` rows each
__device__ __forceinline__ uint32_t kmajor_off(uint32_t row, uint32_t k, uint32_t rows) {
    return (k / kKB) * rows * 128u + sw128_offset(row, (k % kKB) * 2u);
}

// wait until the commit barrier's phase `parity` completes; bounded (a timeout sets the error word)
__device__ bool commit_wait(uint64_t *bar, uint32_t parity, int *err_word) {
    return mbar_wait(bar, parity, nullptr, err_word, 200000000ull);
}

// ------------------------------------------------------------------------------------------------
// q absorb: B = W_UK[h] as [512 c][128 j] (two K blocks of 512 rows x 128 B = 128 KB), A = a 128-row
// tile of q_nope (two K blocks of 128 rows x 128 B = 32 KB, bf16 hi only when the queries are bf16,
// hi then lo when f32), D = [128 rows][512 c] f32 = all 512 TMEM columns.
// ------------------------------------------------------------------------------------------------
struct QTcSmem {
    alignas(1024) uint8_t b[2][kKL * 128];        // W_UK^T, K blocks j 0..63 / 64..127
    alignas(1024) uint8_t a[2][2][kPT * 128];     // [piece][K block] query tile
    uint64_t mma_bar;
    uint32_t tmem_base;
};

__global__ void __launch_bounds__(kPThreads, 1) q_absorb_tc_kernel(const void *__restrict__ q_nope, int q_bf16, int S,
                                                                   int H, const uint8_t *__restrict__ w8,
                                                                   const float *__restrict__ w_scale,
                                                                   void *__restrict__ q_lat, int out_bf16,
                                                                   int *err_word) {
    extern __shared__ __align__(1024) uint8_t smem[];
    QTcSmem &sm = *reinterpret_cast<QTcSmem *>(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, h = blockIdx.x;
    if ((smem_u32(smem) & 1023u) != 0) {
        if (tid == 0 && err_word) atomicOr(err_word, (int)KV8_ERR_TIMEOUT);
        return;
    }
    if (tid == 0) {
        mbar_init(&sm.mma_bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    // a programmatic dependent: the weights (never written by the kernel before this one on the stream)
    // are decoded while that kernel finishes; the activations are read only after it has completed
    grid_launch_dependents();
    // W_UK[h] (e4m3 [128 j][512 c]) -> b[j / 64][c][j % 64] as bf16: item (j, c4) = 4 consecutive c;
    // each thread's loads go out 16 at a time
    static_assert(kNope * (kKL / 4) % (16 * kPThreads) == 0, "weight items split evenly");
    for (int base = tid; base < kNope * (kKL / 4); base += 16 * kPThreads) {
        uint32_t w[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int it = base + u * kPThreads, j = it / (kKL / 4), c4 = it - j * (kKL / 4);
            w[u] = __ldg(reinterpret_cast<const uint32_t *>(w8 + ((int64_t)h * kKvbRows + j) * kKL) + c4);
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int it = base + u * kPThreads, j = it / (kKL / 4), c4 = it - j * (kKL / 4);
            const uint2 v = e4m3x4_to_bf16x4(w[u]);
            const uint16_t e[4] = {(uint16_t)(v.x & 0xFFFFu), (uint16_t)(v.x >> 16), (uint16_t)(v.y & 0xFFFFu),
                                   (uint16_t)(v.y >> 16)};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint16_t *>(&sm.b[0][0] + kmajor_off(4 * c4 + k, j, kKL)) = e[k];
        }
    }
    const int n_pieces = q_bf16 ? 1 : 2;
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t idesc = idesc_bf16_f32(kPT, 256);
    const int q = warp & 3, col_half = warp >> 2;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    const int n_tiles = (S + kPT - 1) / kPT;
    // A query tile is 128 rows x 16 items of 8 values; thread tid takes items tid + 256 u (u < 8).  The
    // next tile's values are loaded into registers (raw: 8 bf16 = one uint4, or 8 f32 = two float4) while
    // the current tile's MMAs and epilogue run.
    constexpr int kQItems = kPT * (kNope / 8) / kPThreads;  // 8
    static_assert(kPT * (kNope / 8) == kQItems * kPThreads, "query items split evenly");
    uint4 raw[kQItems][2];
    auto load_tile = [&](int ti) {
#pragma unroll
        for (int u = 0; u < kQItems; ++u) {
            const int it = tid + u * kPThreads, r = it / (kNope / 8), j8 = it - r * (kNope / 8);
            const int srow = ti * kPT + r;
            raw[u][0] = raw[u][1] = make_uint4(0u, 0u, 0u, 0u);
            if (ti < n_tiles && srow < S) {
                const int64_t e = ((int64_t)srow * H + h) * kNope + 8 * j8;
                if (q_bf16) {
                    raw[u][0] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(q_nope) + e));
                } else {
                    raw[u][0] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(q_nope) + e));
                    raw[u][1] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(q_nope) + e) + 1);
                }
            }
        }
    };
    grid_dependency_wait();
    load_tile(0);
    bool ok = true;
    for (int ti = 0; ti < n_tiles && ok; ++ti) {
        const int s0 = ti * kPT;
        // ---- query tile -> a[piece][K block]: item (row, j8) = 8 consecutive j of one row
#pragma unroll
        for (int u = 0; u < kQItems; ++u) {
            const int it = tid + u * kPThreads, r = it / (kNope / 8), j8 = it - r * (kNope / 8);
            float v[8];
            if (q_bf16) {
                const uint32_t w4[4] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[k]));
                    v[2 * k] = f.x;
                    v[2 * k + 1] = f.y;
                }
            } else {
                v[0] = __uint_as_float(raw[u][0].x); v[1] = __uint_as_float(raw[u][0].y);
                v[2] = __uint_as_float(raw[u][0].z); v[3] = __uint_as_float(raw[u][0].w);
                v[4] = __uint_as_float(raw[u][1].x); v[5] = __uint_as_float(raw[u][1].y);
                v[6] = __uint_as_float(raw[u][1].z); v[7] = __uint_as_float(raw[u][1].w);
            }
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t h0 = bf16_bits(v[2 * k]), h1 = bf16_bits(v[2 * k + 1]);
                hi[k] = h0 | (h1 << 16);
                const float r0 = v[2 * k] - __bfloat162float(__ushort_as_bfloat16((uint16_t)h0));
                const float r1 = v[2 * k + 1] - __bfloat162float(__ushort_as_bfloat16((uint16_t)h1));
                lo[k] = bf16_bits(r0) | (bf16_bits(r1) << 16);
            }
            const uint32_t off = kmajor_off(r, 8 * j8, kPT);  // 16 bytes, one swizzle chunk
            *reinterpret_cast<uint4 *>(&sm.a[0][0][0] + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            if (n_pieces == 2) *reinterpret_cast<uint4 *>(&sm.a[1][0][0] + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        load_tile(ti + 1);  // in flight during this tile's MMAs and epilogue
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        tc_fence_after_sync();
        if (tid == 0) {
            for (int nh = 0; nh < 2; ++nh) {
                bool first = true;
                for (int pc = 0; pc < n_pieces; ++pc)
                    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = smem_desc(smem_u32(sm.a[pc][kb]) + kk * 32, 0, 1024, kSw128);
                            const uint64_t bd = smem_desc(smem_u32(sm.b[kb]) + nh * 256 * 128 + kk * 32, 0, 1024, kSw128);
                            mma_bf16(tmem + (uint32_t)nh * 256u, ad, bd, idesc, first ? 0u : 1u);
                            first = false;
                        }
            }
            mma_commit(&sm.mma_bar);
        }
        // one decision for the whole block: every thread must take the same path through the barriers
        ok = __syncthreads_and(commit_wait(&sm.mma_bar, (uint32_t)(ti & 1), err_word)) != 0;
        tc_fence_after_sync();
        // ---- epilogue: thread (row r, column half) -> 256 outputs, scaled per 128-column block
        const int r = q * 32 + lane, s = s0 + r;
        for (int c0 = col_half * 256; c0 < col_half * 256 + 256 && ok; c0 += 64) {
            uint32_t v[4][16];  // 64 columns (one scale block), one TMEM round trip
#pragma unroll
            for (int g = 0; g < 4; ++g) tmem_ld_32x32b_x16(tmem + lane_addr + (uint32_t)(c0 + 16 * g), v[g]);
            tmem_wait_ld();
            const float sc = __ldg(w_scale + (int64_t)(2 * h) * kNbc + c0 / kBlk);
            if (s < S) {
                const int64_t o = ((int64_t)s * H + h) * kKL + c0;
                if (out_bf16) {
                    uint4 *d = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(q_lat) + o);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint32_t pk[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            pk[k] = bf16_bits(__uint_as_float(v[g][2 * k]) * sc) | (bf16_bits(__uint_as_float(v[g][2 * k + 1]) * sc) << 16);
                        d[2 * g] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        d[2 * g + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                } else {
                    float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(q_lat) + o);
#pragma unroll
                    for (int g = 0; g < 4; ++g)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            d[4 * g + k] = make_float4(__uint_as_float(v[g][4 * k]) * sc, __uint_as_float(v[g][4 * k + 1]) * sc,
                                                       __uint_as_float(v[g][4 * k + 2]) * sc, __uint_as_float(v[g][4 * k + 3]) * sc);
                }
            }
        }
        tc_fence_before_sync();
        __syncthreads();  // accumulators read and the tile's shared memory free before the next tile
        tc_fence_after_sync();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------------------------
// out project: B = W_UV[h] as [128 v][512 c] (eight K blocks of 128 rows x 128 B = 128 KB: the rows'
// natural order); per 128-column scale block cb, A = the context tile's columns of that block as bf16
// hi + lo pieces (2 pieces x 2 K blocks x 16 KB), D[cb] = [128 rows][128 v] f32 at TMEM column 128 cb.
// ------------------------------------------------------------------------------------------------
struct OTcSmem {
    alignas(1024) uint8_t b[kKL / kKB][kVH * 128];  // W_UV, K block kb = columns 64kb..64kb+63
    alignas(1024) uint8_t a[2][2][kPT * 128];       // [piece][K block within the scale block]
    uint64_t mma_bar;
    uint32_t tmem_base;
};

__global__ void __launch_bounds__(kPThreads, 1) out_project_tc_kernel(const float *__restrict__ ctx, int S, int H,
                                                                      const uint8_t *__restrict__ w8,
                                                                      const float *__restrict__ w_scale,
                                                                      float *__restrict__ out, int *err_word) {
    extern __shared__ __align__(1024) uint8_t smem[];
    OTcSmem &sm = *reinterpret_cast<OTcSmem *>(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, h = blockIdx.x;
    if ((smem_u32(smem) & 1023u) != 0) {
        if (tid == 0 && err_word) atomicOr(err_word, (int)KV8_ERR_TIMEOUT);
        return;
    }
    if (tid == 0) {
        mbar_init(&sm.mma_bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem_base, 512);
        tmem_relinquish();
    }
    // a programmatic dependent: the weights (never written by the kernel before this one on the stream)
    // are decoded while that kernel finishes; the context rows are read only after it has completed
    grid_launch_dependents();
    // W_UV[h] (e4m3 [128 v][512 c]) -> b[c / 64][v][c % 64] as bf16: item (v, c8) = 8 consecutive c; each
    // thread's loads go out 16 at a time
    static_assert(kVH * (kKL / 8) % (16 * kPThreads) == 0, "weight items split evenly");
    for (int base = tid; base < kVH * (kKL / 8); base += 16 * kPThreads) {
        uint2 w[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int it = base + u * kPThreads, v = it / (kKL / 8), c8 = it - v * (kKL / 8);
            w[u] = __ldg(reinterpret_cast<const uint2 *>(w8 + ((int64_t)h * kKvbRows + kNope + v) * kKL) + c8);
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int it = base + u * kPThreads, v = it / (kKL / 8), c8 = it - v * (kKL / 8);
            const uint2 lo = e4m3x4_to_bf16x4(w[u].x), hi = e4m3x4_to_bf16x4(w[u].y);
            *reinterpret_cast<uint4 *>(&sm.b[0][0] + kmajor_off(v, 8 * c8, kVH)) = make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t idesc = idesc_bf16_f32(kPT, kVH);
    const int q = warp & 3, col_half = warp >> 2;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    const int n_tiles = (S + kPT - 1) / kPT;
    float sc[kNbc];
#pragma unroll
    for (int k = 0; k < kNbc; ++k) sc[k] = __ldg(w_scale + (int64_t)(2 * h + 1) * kNbc + k);
    // A stage is one scale block (128 columns) of a 128-row context tile: 128 rows x 16 items of 8 f32;
    // thread tid takes items tid + 256 u (u < 8).  The next stage's values are loaded into registers
    // while the current stage's MMAs (and, after a tile's last block, its epilogue) run.
    constexpr int kOItems = kPT * (kBlk / 8) / kPThreads;  // 8
    static_assert(kPT * (kBlk / 8) == kOItems * kPThreads, "context items split evenly");
    float4 raw[kOItems][2];
    auto load_stage = [&](int ti, int cb) {
#pragma unroll
        for (int u = 0; u < kOItems; ++u) {
            const int it = tid + u * kPThreads, r = it / (kBlk / 8), c8 = it - r * (kBlk / 8);
            const int srow = ti * kPT + r;
            raw[u][0] = raw[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ti < n_tiles && srow < S) {
                const float4 *src = reinterpret_cast<const float4 *>(ctx + ((int64_t)srow * H + h) * kKL + cb * kBlk + 8 * c8);
                raw[u][0] = __ldg(src);
                raw[u][1] = __ldg(src + 1);
            }
        }
    };
    grid_dependency_wait();
    load_stage(0, 0);
    bool ok = true;
    uint32_t phase = 0;
    for (int ti = 0; ti < n_tiles && ok; ++ti) {
        const int s0 = ti * kPT;
        for (int cb = 0; cb < kNbc && ok; ++cb) {
            // ---- context columns 128cb.. of the tile -> bf16 hi + lo: item (row, c8)
#pragma unroll
            for (int u = 0; u < kOItems; ++u) {
                const int it = tid + u * kPThreads, r = it / (kBlk / 8), c8 = it - r * (kBlk / 8);
                const float v[8] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w,
                                    raw[u][1].x, raw[u][1].y, raw[u][1].z, raw[u][1].w};
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t h0 = bf16_bits(v[2 * k]), h1 = bf16_bits(v[2 * k + 1]);
                    hi[k] = h0 | (h1 << 16);
                    const float r0 = v[2 * k] - __bfloat162float(__ushort_as_bfloat16((uint16_t)h0));
                    const float r1 = v[2 * k + 1] - __bfloat162float(__ushort_as_bfloat16((uint16_t)h1));
                    lo[k] = bf16_bits(r0) | (bf16_bits(r1) << 16);
                }
                const uint32_t off = kmajor_off(r, 8 * c8, kPT);
                *reinterpret_cast<uint4 *>(&sm.a[0][0][0] + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4 *>(&sm.a[1][0][0] + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            if (cb + 1 < kNbc)
                load_stage(ti, cb + 1);
            else
                load_stage(ti + 1, 0);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            __syncthreads();
            tc_fence_after_sync();
            if (tid == 0) {
                bool first = true;
                for (int pc = 0; pc < 2; ++pc)
                    for (int kb = 0; kb < 2; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = smem_desc(smem_u32(sm.a[pc][kb]) + kk * 32, 0, 1024, kSw128);
                            const uint64_t bd = smem_desc(smem_u32(sm.b[2 * cb + kb]) + kk * 32, 0, 1024, kSw128);
                            mma_bf16(tmem + (uint32_t)cb * 128u, ad, bd, idesc, first ? 0u : 1u);
                            first = false;
                        }
                mma_commit(&sm.mma_bar);
            }
            // one decision for the whole block (the barrier also frees the A tile for the next block)
            ok = __syncthreads_and(commit_wait(&sm.mma_bar, phase, err_word)) != 0;
            phase ^= 1u;
            tc_fence_after_sync();
        }
        // ---- epilogue: out[s][h][v] = sum_cb sc[cb] * D[cb][r][v]; thread (row r, half of the 128 v)
        const int r = q * 32 + lane, s = s0 + r;
        for (int v0 = col_half * 64; v0 < col_half * 64 + 64 && ok; v0 += 16) {
            float accv[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) accv[k] = 0.f;
            uint32_t d[kNbc][16];  // the four scale blocks' accumulators, one TMEM round trip
#pragma unroll
            for (int cb = 0; cb < kNbc; ++cb) tmem_ld_32x32b_x16(tmem + lane_addr + (uint32_t)(cb * 128 + v0), d[cb]);
            tmem_wait_ld();
#pragma unroll
            for (int cb = 0; cb < kNbc; ++cb)
#pragma unroll
                for (int k = 0; k < 16; ++k) accv[k] = fmaf(sc[cb], __uint_as_float(d[cb][k]), accv[k]);
            if (s < S) {
                float4 *dst = reinterpret_cast<float4 *>(out + ((int64_t)s * H + h) * kVH + v0);
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k] = make_float4(accv[4 * k], accv[4 * k + 1], accv[4 * k + 2], accv[4 * k + 3]);
            }
        }
        tc_fence_before_sync();
        __syncthreads();  // accumulators read before the next tile overwrites them
        tc_fence_after_sync();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_q_absorb_tc(const void *q_nope, int q_bf16, int S, int H, const uint8_t *w8, const float *w_scale,
                               void *q_lat, int out_bf16, int *err_word, cudaStream_t st) {
    const size_t smem = sizeof(QTcSmem);
    cudaError_t e = cudaFuncSetAttribute(q_absorb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)H);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, q_absorb_tc_kernel, q_nope, q_bf16, S, H, w8, w_scale, q_lat, out_bf16, err_word);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_out_project_tc(const float *ctx, int S, int H, const uint8_t *w8, const float *w_scale, float *out,
                                  int *err_word, cudaStream_t st) {
    const size_t smem = sizeof(OTcSmem);
    cudaError_t e = cudaFuncSetAttribute(out_project_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)H);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, out_project_tc_kernel, ctx, S, H, w8, w_scale, out, err_word);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kv8
