// attn_tc.cu -- absorbed MLA attention over e4m3 cache rows on the 5th-generation tensor cores
// (tcgen05, sm_103a), for bf16 queries.
//
// Page "KV8 long-context CUDA: fp8 device shadow, split-T kernels, DSA-aware gather":
//   first commit message  -- score = sm_scale * s_t * q.e4m3(row) (the row scale hoisted out of the dot);
//                            context = softmax-weighted sum of s_t * e4m3(Lc_t) (the latent is both key
//                            and value).
//   second commit message -- split-T: partial online-softmax blocks (cl[K], m, z) + log-sum-exp merge;
//                            the batch/prefill path streams tiles of rows.
//
// Every head reads the same latent rows, so the H x 576 by 576 x T score product and the H x T by
// T x 512 context product are dense contractions.  One CTA owns 64 heads and one partition of rows:
//
//   score   S^T[t][n]   = sum_k  K8[t][k] * Qs[n][k]        M = 128 rows, N = 128, K = 576 (e4m3 x e4m3)
//           Qs = [Q_hi ; Q_lo]: each bf16 query element q*2^e is split exactly into two e4m3 values
//           (8 significant bits = 4 + 4), so S[t][h] = S^T[t][h] + S^T[t][64+h] is the bf16-exact dot.
//           The cache bytes are the A operand as loaded (no dequantisation).
//   softmax one thread per tile row (TMEM lane); online max with a lazy rescale (only when a head's
//           max grows by more than kTau); weights w = 2^(s - m) * s_t / s_ref * 2^(8-kTau), split into
//           e4m3 hi + lo the same way.
//   context O^T[d][h]  += sum_t  V8[t][d] * W^T[t][h]        M = 128 dims (x4 chunks), N = 64, K = 128 rows
//           A = the same cache bytes read MN-major (V^T), B = the weights MN-major.
//
// Warps: 0 = TMA producer, 1 = MMA issuer (and TMEM owner), 2..9 = softmax / epilogue.
// Shared memory (231 KB): query image 72 KB, two 72 KB row stages (the weights' hi piece reuses the
// stage's rope block once the score has read it), weights' lo piece 8 KB, barriers and scratch.
// TMEM (512 columns): two 128-column score buffers, four 64-column context accumulators.
// Every wait is an mbarrier wait bounded in time; a timeout sets KV8_ERR_TIMEOUT and the CTA winds
// down without hanging.
#include "internal.h"
#include "sm100.cuh"

#include <cudaTypedefs.h>
#include <math.h>
#include <stddef.h>

#include <mutex>

namespace kv8 {
namespace {

using namespace sm100;

constexpr int kTile = 128;             // rows per tile
constexpr int kHeadsPerCta = 64;
constexpr int kThreads = 320;          // 10 warps
constexpr int kSoftmaxThreads = 256;   // warps 2..9
constexpr int kPrepThreads = 288;      // warps 1..9
constexpr uint32_t kImg = 73728;       // 4 x 16 KB (SW128, 128 B per row) + 8 KB (SW64, 64 B per row)
constexpr uint32_t kRcOff = 65536;     // rope block inside an image / stage
constexpr uint32_t OFF_Q = 0, OFF_ST0 = kImg, OFF_ST1 = 2 * kImg, OFF_PLO = 3 * kImg, OFF_MISC = 3 * kImg + 8192;
constexpr float kTau = 2.0f;           // lazy-rescale threshold (log2 units): p <= 2^kTau
constexpr float kWScale = 64.0f;       // 2^(8 - kTau): keeps w <= 256 < 448 (e4m3 max)

struct Misc {
    // per-head arrays first: m_run is read with 16-byte vector loads
    alignas(16) float m_run[kHeadsPerCta];
    alignas(16) float red[4][kHeadsPerCta];
    alignas(16) float alpha[kHeadsPerCta];
    alignas(16) float zsum[kHeadsPerCta];
    alignas(16) float wred[2][16];
    uint64_t kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full, pv_done, sync_bar, final_bar;
    uint32_t tmem_base;
    int abort_flag;
    int vote[2];
    float c_score;   // sm_scale * log2(e) * 2^-e
    float w_mul;     // kWScale / s_ref
    float out_mul;   // s_ref / kWScale
};
static_assert(OFF_MISC % 16 == 0 && offsetof(Misc, m_run) % 16 == 0, "vector loads of m_run need 16-byte alignment");
static_assert(offsetof(Misc, kv_full) % 8 == 0, "mbarriers need 8-byte alignment");
constexpr uint32_t kSmemBytes = OFF_MISC + sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct TcArgs {
    const __nv_bfloat16 *q_lat;  // [B][H][512]
    const __nv_bfloat16 *q_rope; // [B][H][64]
    int B, H, P, n_half;
    const float *kv_scale;
    int64_t T;
    int64_t pos0;                // causal: item b attends rows [0, pos0 + b]; -1: rows [0, T)
    float sm_scale_log2;
    float *ws;                   // partial sets, or nullptr
    float *out;                  // direct normalised output when ws == nullptr
    int *err_word;
};

__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// e4m3 pair encode (RNE, saturating): returns byte(a) | byte(b) << 8.
__device__ __forceinline__ uint32_t enc_pair(float a, float b) {
    uint16_t v;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(b), "f"(a));
    return v;
}

// decode an e4m3 pair (byte 0 -> .x) exactly
__device__ __forceinline__ float2 dec_pair(uint32_t v) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xFFFFu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<__half2 *>(&h));
}

// Split two values into e4m3 hi + lo pieces: x ~= dec(hi) + dec(lo).
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
    hi = enc_pair(a, b);
    const float2 h = dec_pair(hi);
    lo = enc_pair(a - h.x, b - h.y);
}

// Bounded barrier among the 256 softmax threads (an mbarrier, so a missing thread cannot hang it).
struct SoftSync {
    uint64_t *bar;
    volatile int *abort_flag;
    int *err;
    uint32_t n = 0;
    __device__ bool operator()() {
        mbar_arrive(bar);
        return mbar_wait(bar, (n++) & 1u, abort_flag, err);
    }
};

// 10 warps: a sub-partition holding 3 warps caps a thread at 168 registers (16K registers each).
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap map_lc, const __grid_constant__ CUtensorMap map_rc, TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc &ms = *reinterpret_cast<Misc *>(smem + OFF_MISC);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(smem) & 1023u) != 0) {  // swizzled operands need 1024-byte alignment
        if (tid == 0 && a.err_word) atomicOr(a.err_word, (int)KV8_ERR_TIMEOUT);
        return;
    }

    // ---- which item, partition and head half
    const int per_item = a.P * a.n_half;
    const int b = blockIdx.x / per_item, rem = blockIdx.x - b * per_item;
    const int part = rem / a.n_half, half = rem - part * a.n_half;
    const int64_t n_rows = a.pos0 >= 0 ? ((a.pos0 + b + 1 < a.T) ? a.pos0 + b + 1 : a.T) : a.T;
    const int64_t t0 = n_rows * part / a.P, t1 = n_rows * (part + 1) / a.P;
    const int n_tiles = (int)((t1 - t0 + kTile - 1) / kTile);

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&ms.kv_full[s], 1);
            mbar_init(&ms.kv_empty[s], 1);
            mbar_init(&ms.s_full[s], 1);
            mbar_init(&ms.s_free[s], kSoftmaxThreads);
            ms.vote[s] = 0;
        }
        mbar_init(&ms.p_full, kSoftmaxThreads);
        mbar_init(&ms.pv_done, 1);
        mbar_init(&ms.sync_bar, kSoftmaxThreads);
        mbar_init(&ms.final_bar, 1);
        ms.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&ms.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t sbase = smem_u32(smem);

    if (warp == 0) {
        // ================================ TMA producer ================================
        if (lane == 0 && n_tiles > 0) {
            prefetch_tensormap(&map_lc);
            prefetch_tensormap(&map_rc);
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i & 1;
                if (i >= 2 && !mbar_wait(&ms.kv_empty[s], ((i >> 1) - 1) & 1, &ms.abort_flag, a.err_word)) break;
                uint8_t *st = smem + (s ? OFF_ST1 : OFF_ST0);
                mbar_arrive_expect_tx(&ms.kv_full[s], kImg);
                const int y = (int)(t0 + (int64_t)i * kTile);
                for (int kb = 0; kb < 4; ++kb) tma_load_2d(st + kb * 16384, &map_lc, kb * 128, y, &ms.kv_full[s]);
                tma_load_2d(st + kRcOff, &map_rc, 512, y, &ms.kv_full[s]);
                issued = i + 1;
            }
            // every issued load must land before the CTA ends
            for (int i = (issued > 2 ? issued - 2 : 0); i < issued; ++i)
                mbar_wait(&ms.kv_full[i & 1], (i >> 1) & 1, nullptr, a.err_word, 200000000ull);
        }
        __syncwarp();
    } else {
        // ======================= prologue: query image, row-scale max =======================
        const int pt = tid - 32;  // 0..287
        float qmax = 0.f, smax = 0.f;
        for (int it = pt; it < kHeadsPerCta * 36; it += kPrepThreads) {
            const int h = it / 36, ch = it - h * 36;
            const int hg = half * kHeadsPerCta + h;
            if (hg < a.H) {
                const __nv_bfloat16 *src = ch < 32 ? a.q_lat + ((int64_t)b * a.H + hg) * kKL + ch * 16
                                                   : a.q_rope + ((int64_t)b * a.H + hg) * kKR + (ch - 32) * 16;
                const uint4 u0 = *reinterpret_cast<const uint4 *>(src), u1 = *reinterpret_cast<const uint4 *>(src + 8);
                const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[k]));
                    qmax = fmaxf(qmax, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
            }
        }
        for (int64_t t = t0 + pt; t < t1; t += kPrepThreads) smax = fmaxf(smax, fabsf(__ldg(a.kv_scale + t)));
        qmax = warp_max(qmax);
        smax = warp_max(smax);
        if (lane == 0) {
            ms.wred[0][warp - 1] = qmax;
            ms.wred[1][warp - 1] = smax;
        }
        named_sync(1, kPrepThreads);
        qmax = 0.f;
        smax = 0.f;
        for (int k = 0; k < 9; ++k) {
            qmax = fmaxf(qmax, ms.wred[0][k]);
            smax = fmaxf(smax, ms.wred[1][k]);
        }
        // q * 2^e lies in [128, 256): every bf16 value splits exactly into e4m3 hi + lo (down to the
        // e4m3 subnormal step); the score is rescaled by 2^-e.
        int E = 0;
        if (qmax > 0.f) frexpf(qmax, &E);
        const int e = qmax > 0.f ? 8 - E : 0;
        const float qmul = ldexpf(1.f, e);
        for (int it = pt; it < kHeadsPerCta * 36; it += kPrepThreads) {
            const int h = it / 36, ch = it - h * 36;
            const int hg = half * kHeadsPerCta + h;
            uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
            if (hg < a.H) {
                const __nv_bfloat16 *src = ch < 32 ? a.q_lat + ((int64_t)b * a.H + hg) * kKL + ch * 16
                                                   : a.q_rope + ((int64_t)b * a.H + hg) * kKR + (ch - 32) * 16;
                const uint4 u0 = *reinterpret_cast<const uint4 *>(src), u1 = *reinterpret_cast<const uint4 *>(src + 8);
                const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[k]));
                    uint32_t ph, pl;
                    split_pair(f.x * qmul, f.y * qmul, ph, pl);
                    hi[k >> 1] |= ph << ((k & 1) * 16);
                    lo[k >> 1] |= pl << ((k & 1) * 16);
                }
            }
            uint8_t *img = smem + OFF_Q;
            uint32_t off_hi, off_lo;
            if (ch < 32) {
                const uint32_t kb = ch >> 3, byte = (ch & 7) * 16;
                off_hi = kb * 16384 + sw128_offset(h, byte);
                off_lo = kb * 16384 + sw128_offset(h + 64, byte);
            } else {
                const uint32_t byte = (ch - 32) * 16;
                off_hi = kRcOff + sw64_offset(h, byte);
                off_lo = kRcOff + sw64_offset(h + 64, byte);
            }
            *reinterpret_cast<uint4 *>(img + off_hi) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(img + off_lo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
        if (pt < kHeadsPerCta) ms.m_run[pt] = -INFINITY;
        if (pt == 0) {
            const float s_ref = fmaxf(smax, 1e-30f);
            ms.c_score = a.sm_scale_log2 * ldexpf(1.f, -e);
            ms.w_mul = kWScale / s_ref;
            ms.out_mul = s_ref / kWScale;
        }
        fence_proxy_async_smem();
        named_sync(1, kPrepThreads);

        if (warp == 1) {
            // ================================ MMA issuer ================================
            if (lane == 0) {
                const uint32_t id_s = idesc_e4m3_f32(128, 128, false, false);
                const uint32_t id_pv = idesc_e4m3_f32(128, 64, true, true);
                const uint32_t qb = sbase + OFF_Q;
                for (int i = 0; i <= n_tiles; ++i) {
                    if (i < n_tiles) {
                        const int s = i & 1;
                        if (!mbar_wait(&ms.kv_full[s], (i >> 1) & 1, &ms.abort_flag, a.err_word)) break;
                        if (i >= 2 && !mbar_wait(&ms.s_free[s], ((i >> 1) - 1) & 1, &ms.abort_flag, a.err_word)) break;
                        tc_fence_after_sync();
                        const uint32_t st = sbase + (s ? OFF_ST1 : OFF_ST0);
                        const uint32_t d = tmem + (uint32_t)s * 128u;
#pragma unroll
                        for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_f8f6f4(d, smem_desc(st + kb * 16384 + kk * 32, 0, 1024, kSw128),
                                           smem_desc(qb + kb * 16384 + kk * 32, 0, 1024, kSw128), id_s,
                                           (kb | kk) != 0);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk)
                            mma_f8f6f4(d, smem_desc(st + kRcOff + kk * 32, 0, 512, kSw64),
                                       smem_desc(qb + kRcOff + kk * 32, 0, 512, kSw64), id_s, 1);
                        mma_commit(&ms.s_full[s]);
                    }
                    if (i >= 1) {
                        const int j = i - 1, s = j & 1;
                        if (!mbar_wait(&ms.p_full, j & 1, &ms.abort_flag, a.err_word)) break;
                        tc_fence_after_sync();
                        const uint32_t st = sbase + (s ? OFF_ST1 : OFF_ST0);
                        const uint32_t phi = st + kRcOff, plo = sbase + OFF_PLO;
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) {
                            const uint32_t d = tmem + 256u + (uint32_t)ch * 64u;
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk) {
                                const uint64_t ad = smem_desc(st + ch * 16384 + kk * 4096, 0, 1024, kSw128);
                                mma_f8f6f4(d, ad, smem_desc(phi + kk * 2048, 0, 512, kSw64), id_pv, (j | kk) != 0);
                                mma_f8f6f4(d, ad, smem_desc(plo + kk * 2048, 0, 512, kSw64), id_pv, 1);
                            }
                        }
                        mma_commit(&ms.kv_empty[s]);
                        mma_commit(&ms.pv_done);
                    }
                }
                // all issued MMAs complete before the CTA tears down
                mma_commit(&ms.final_bar);
                mbar_wait(&ms.final_bar, 0, nullptr, a.err_word, 200000000ull);
            }
            __syncwarp();
        } else {
            // ============================ softmax + epilogue ============================
            const int q = warp & 3;               // TMEM lane quadrant
            const int hh = (warp - 2) >> 2;       // which 32 of the CTA's 64 heads
            const int r = q * 32 + lane;          // row within the tile = TMEM lane
            const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
            SoftSync sync{&ms.sync_bar, &ms.abort_flag, a.err_word};
            const float c_score = ms.c_score, w_mul = ms.w_mul;
            float z[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] = 0.f;
            float sc_next = (n_tiles > 0 && t0 + r < t1) ? __ldg(a.kv_scale + t0 + r) : 0.f;
            bool ok = true;
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int bb = i & 1;
                const int64_t t = t0 + (int64_t)i * kTile + r;
                const bool valid = t < t1;
                const float sc_t = sc_next;
                sc_next = (i + 1 < n_tiles && t + kTile < t1) ? __ldg(a.kv_scale + t + kTile) : 0.f;

                if (!(ok = mbar_wait(&ms.s_full[bb], (i >> 1) & 1, &ms.abort_flag, a.err_word))) break;
                tc_fence_after_sync();
                const float f = sc_t * c_score;
                float s[32];
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2) {
                    uint32_t shi[16], slo[16];
                    tmem_ld_32x32b_x16(tmem + lane_addr + (uint32_t)bb * 128u + 32u * hh + 16u * k2, shi);
                    tmem_ld_32x32b_x16(tmem + lane_addr + (uint32_t)bb * 128u + 64u + 32u * hh + 16u * k2, slo);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        s[16 * k2 + j] = valid ? (__uint_as_float(shi[j]) + __uint_as_float(slo[j])) * f : -INFINITY;
                }
                tc_fence_before_sync();
                mbar_arrive(&ms.s_free[bb]);

                // lazy rescale check: does any score exceed its head's running max by more than kTau?
                bool need = false;
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(&ms.m_run[32 * hh + 4 * j4]);
                    need |= (s[4 * j4 + 0] > m4.x + kTau) | (s[4 * j4 + 1] > m4.y + kTau) |
                            (s[4 * j4 + 2] > m4.z + kTau) | (s[4 * j4 + 3] > m4.w + kTau);
                }
                if (need) ms.vote[bb] = i + 1;
                if (!(ok = sync())) break;
                if (ms.vote[bb] == i + 1) {
                    // tile max per head: warp reduce, then across the 4 quadrants
                    float mine = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float v = warp_max(s[j]);
                        if (lane == j) mine = v;
                    }
                    ms.red[q][32 * hh + lane] = mine;
                    if (!(ok = sync())) break;
                    if (q == 0) {
                        const int h = 32 * hh + lane;
                        const float tmax = fmaxf(fmaxf(ms.red[0][h], ms.red[1][h]), fmaxf(ms.red[2][h], ms.red[3][h]));
                        const float mo = ms.m_run[h];
                        const float mn = (tmax > mo + kTau) ? tmax : mo;
                        ms.alpha[h] = (mn == mo) ? 1.f : exp2f(mo - mn);
                        ms.m_run[h] = mn;
                    }
                    if (!(ok = sync())) break;
                    bool any = false;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float al = ms.alpha[32 * hh + j];
                        z[j] *= al;
                        any |= al != 1.f;
                    }
                    if (any && i >= 1) {
                        // rescale this warp's 32 head columns of the context accumulators (after PV(i-1))
                        if (!(ok = mbar_wait(&ms.pv_done, (i - 1) & 1, &ms.abort_flag, a.err_word))) break;
                        tc_fence_after_sync();
#pragma unroll 1
                        for (int ch = 0; ch < 8; ++ch) {
                            uint32_t o[16];
                            const uint32_t ta = tmem + lane_addr + 256u + 64u * (ch >> 1) + 32u * hh + 16u * (ch & 1);
                            tmem_ld_32x32b_x16(ta, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                o[j] = __float_as_uint(__uint_as_float(o[j]) * ms.alpha[32 * hh + 16 * (ch & 1) + j]);
                            tmem_st_32x32b_x16(ta, o);
                        }
                        tmem_wait_st();
                    }
                }
                // weights: p = 2^(s - m) (row sum z), w = p * s_t * kWScale / s_ref, split e4m3 hi + lo
                const float g = sc_t * w_mul;
                uint32_t whi[8], wlo[8];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(&ms.m_run[32 * hh + 4 * j4]);
                    const float p0 = exp2f(s[4 * j4 + 0] - m4.x), p1 = exp2f(s[4 * j4 + 1] - m4.y);
                    const float p2 = exp2f(s[4 * j4 + 2] - m4.z), p3 = exp2f(s[4 * j4 + 3] - m4.w);
                    z[4 * j4 + 0] += p0;
                    z[4 * j4 + 1] += p1;
                    z[4 * j4 + 2] += p2;
                    z[4 * j4 + 3] += p3;
                    uint32_t h01, l01, h23, l23;
                    split_pair(p0 * g, p1 * g, h01, l01);
                    split_pair(p2 * g, p3 * g, h23, l23);
                    whi[j4] = h01 | (h23 << 16);
                    wlo[j4] = l01 | (l23 << 16);
                }
                uint8_t *phi = smem + (bb ? OFF_ST1 : OFF_ST0) + kRcOff;  // the rope block, read by the score already
                *reinterpret_cast<uint4 *>(phi + sw64_offset(r, 32 * hh)) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
                *reinterpret_cast<uint4 *>(phi + sw64_offset(r, 32 * hh + 16)) =
                    make_uint4(whi[4], whi[5], whi[6], whi[7]);
                if (i >= 1 && !(ok = mbar_wait(&ms.pv_done, (i - 1) & 1, &ms.abort_flag, a.err_word))) break;
                uint8_t *plo = smem + OFF_PLO;
                *reinterpret_cast<uint4 *>(plo + sw64_offset(r, 32 * hh)) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
                *reinterpret_cast<uint4 *>(plo + sw64_offset(r, 32 * hh + 16)) =
                    make_uint4(wlo[4], wlo[5], wlo[6], wlo[7]);
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&ms.p_full);
            }

            // ================================ epilogue ================================
            if (ok && n_tiles > 0) ok = mbar_wait(&ms.pv_done, (n_tiles - 1) & 1, &ms.abort_flag, a.err_word);
            tc_fence_after_sync();
            // row sums: over the 32 lanes of the warp, then over the 4 quadrants
            float zmine = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const float v = warp_sum(z[j]);
                if (lane == j) zmine = v;
            }
            ms.red[q][32 * hh + lane] = zmine;
            if (ok) ok = sync();
            if (ok) {
                if (q == 0) {
                    const int h = 32 * hh + lane;
                    ms.zsum[h] = ms.red[0][h] + ms.red[1][h] + ms.red[2][h] + ms.red[3][h];
                }
                ok = sync();
            }
            if (ok) {
                const float out_mul = ms.out_mul;
                const int hbase = half * kHeadsPerCta + 32 * hh;
                PartialView pv(a.ws, a.B, a.P, a.H);
#pragma unroll 1
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t o[16];
                    if (n_tiles > 0) {
                        tmem_ld_32x32b_x16(tmem + lane_addr + 256u + 64u * (ch >> 1) + 32u * hh + 16u * (ch & 1), o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) o[j] = 0u;
                    }
                    const int d = 128 * (ch >> 1) + r;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int hl = 32 * hh + 16 * (ch & 1) + j;  // head within the CTA
                        const int hg = half * kHeadsPerCta + hl;
                        if (hg >= a.H) continue;
                        const float v = __uint_as_float(o[j]) * out_mul;
                        if (a.ws) {
                            pv.cl[(((int64_t)b * a.P + part) * a.H + hg) * kKL + d] = v;
                        } else {
                            const float zz = ms.zsum[hl];
                            a.out[((int64_t)b * a.H + hg) * kKL + d] = zz > 0.f ? v / zz : 0.f;
                        }
                    }
                }
                if (a.ws && q == 0) {
                    const int hg = hbase + lane;
                    if (hg < a.H) {
                        const int64_t idx = ((int64_t)b * a.P + part) * a.H + hg;
                        pv.m[idx] = n_tiles > 0 ? ms.m_run[32 * hh + lane] : -INFINITY;
                        pv.z[idx] = ms.zsum[32 * hh + lane];
                    }
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// Launch the tensor-core kernel over a cache of T rows.  The grid covers B items x P partitions x
// the head halves.  Returns cudaErrorNotSupported if the tensor-map encoder is unavailable.
cudaError_t launch_attn_tc(const AttnArgs &x, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    CUtensorMap m_lc, m_rc;
    const cuuint64_t dims[2] = {(cuuint64_t)kRow, (cuuint64_t)x.T};
    const cuuint64_t strides[1] = {(cuuint64_t)kRow};
    const cuuint32_t box_lc[2] = {128, kTile}, box_rc[2] = {64, kTile}, es[2] = {1, 1};
    void *base = const_cast<uint8_t *>(x.kv8);
    if (encode(&m_lc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box_lc, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS ||
        encode(&m_rc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box_rc, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    TcArgs a{};
    a.q_lat = static_cast<const __nv_bfloat16 *>(x.q_lat);
    a.q_rope = static_cast<const __nv_bfloat16 *>(x.q_rope);
    a.B = x.B;
    a.H = x.H;
    a.P = x.P;
    a.n_half = x.H > kHeadsPerCta ? 2 : 1;
    a.kv_scale = x.kv_scale;
    a.T = x.T;
    a.pos0 = x.pos0;
    a.sm_scale_log2 = x.sm_scale_log2;
    a.ws = x.ws;
    a.out = x.out;
    a.err_word = x.err_word;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)a.B * a.P * a.n_half;
    attn_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(m_lc, m_rc, a);
    return cudaGetLastError();
}

}  // namespace kv8
