// attn_mixed.cu -- decode over the mixed-precision cache on the 5th-generation tensor cores (tcgen05,
// sm_103a).
//
// Page "B1 Mixed FP8/BF16 FMHA first pass": each KV row keeps its no-position part (448 values) as e4m3
// bytes with a per-row f32 scale and its RoPE part (64 values) as bf16; the query's no-position part is
// quantized from bf16 to e4m3 right before the attention; the head width is 512 = 448 + 64 and the row
// is both key and value.  Per head h and row t:
//     score = sm_scale * ( q_scale[h] * k_scale[t] * sum_i e4m3(q8[h][i]) e4m3(k8[t][i]) + q_rope[h] . k_rope[t] )
//     value = [ k_scale[t] * e4m3(k8[t][0..447]) , k_rope[t][0..63] ]
// The output is split-T partial sets (cl[512], m, z) merged by the shared log-sum-exp merge.
//
// One CTA owns 64 heads and one partition of the rows, streamed as 128-row tiles:
//   score    S_n^T[t][h] = sum_i K8[t][i] Q8[h][i]    kind::f8f6f4 (e4m3 x e4m3), M = 128 rows, N = 64, K = 448
//            S_r^T[t][h] = sum_j KR[t][j] QR[h][j]    kind::f16 (bf16 x bf16), M = 128, N = 64, K = 64; an f32
//                                                     RoPE query enters as bf16 hi + lo (two passes)
//            s = sm_scale log2(e) (q_scale[h] k_scale[t] S_n + S_r)
//   softmax  one thread per tile row, online max with a lazy rescale (only when a head's max grows by
//            more than kTau); p = 2^(s - m); the no-position weights p k_scale[t] / s_ref are split into
//            e4m3 hi + lo, the RoPE weights are p as bf16
//   context  O_n^T[d][h] += sum_t K8[t][d] W8[t][h]     four M = 128 dim chunks read MN-major from the
//                                                      same tile bytes; N = 64, K = 128 rows
//            O_r^T[d][h] += sum_t KR[t][d] WB[t][h]     kind::f16, M = 128
//   The last no-position chunk (dims 384..447) and the RoPE chunk are 64 dims wide: their MMAs run at
//   M = 128 and lanes 64..127 of those accumulators take whatever bytes follow the 64-wide operand
//   (never read back).
//
// Shared memory (220 KB + barriers): two 73,728-byte row stages (no-position columns 0..383 as three
// 128-byte-swizzled blocks, 384..447 as one 64-byte-swizzled block, the RoPE values as one
// 128-byte-swizzled block), the query image (e4m3 rows, bf16 RoPE rows and their lo piece), the
// weights (e4m3 hi and lo, bf16).  TMEM (512 columns): one score buffer (S_n | S_r), five 64-column
// context accumulators.
// Warps: 0 = TMA producer, 1 = MMA issuer (and TMEM owner), 2..9 = softmax / epilogue.  The query image
// and the per-head score factors come from mixed_prep_kernel, run just before as the programmatic
// predecessor: the producer starts the first tile's loads before it waits for that grid; the prologue
// takes the largest row scale of the CTA's rows itself.  Every mbarrier wait is bounded in time; a timeout sets KV8_ERR_TIMEOUT, and the
// softmax warps then skip their remaining waits but pass every named barrier.
#include "internal.h"
#include "quant_row.cuh"
#include "sm100.cuh"

#include <math.h>
#include <stddef.h>

namespace kv8 {
namespace {

using namespace sm100;

constexpr int kMxNope = KV8_MX_NOPE;   // 448
constexpr int kMxRope = KV8_MX_ROPE;   // 64
constexpr int kTile = 128;             // rows per tile
constexpr int kHeads = 64;             // heads per CTA
constexpr int kThreads = 320;          // 10 warps
constexpr int kSoftmaxThreads = 256;   // warps 2..9
constexpr int kPrepThreads = 288;      // warps 1..9
// a row stage: no-position blocks 0..2 (16 KB each), block 3, the RoPE block
constexpr uint32_t kB3 = 49152;        // columns 384..447: 128 rows x 64 bytes, 64-byte swizzle
constexpr uint32_t kRope = 57344;      // 128 rows x 128 bytes (64 bf16), 128-byte swizzle
constexpr uint32_t kStage = 73728;
// the query image: e4m3 rows (blocks 0..2 of 64 x 128 bytes, block 3 of 64 x 64 bytes), bf16 RoPE rows
constexpr uint32_t kQB3 = 24576;
constexpr uint32_t kQR = 28672;        // hi piece (the bf16 query itself)
constexpr uint32_t kQRLo = 36864;      // lo piece (f32 queries)
constexpr uint32_t kQImg = 45056;
constexpr uint32_t OFF_ST0 = 0, OFF_ST1 = kStage, OFF_Q = 2 * kStage;
constexpr uint32_t OFF_WHI = OFF_Q + kQImg;   // e4m3 weights, hi piece: 128 rows x 64 heads, 64-byte swizzle
constexpr uint32_t OFF_WLO = OFF_WHI + 8192;  // lo piece
constexpr uint32_t OFF_WB = OFF_WLO + 8192;   // bf16 weights: 128 rows x 128 bytes, 128-byte swizzle
constexpr uint32_t OFF_MISC = OFF_WB + 16384;
// The 64-dim chunks' second M atom (lanes 64..127) lies this far past the first: block 3 -> the RoPE
// block; a RoPE block -> the next stage's block 0 or the query image.  Both stay inside the allocation.
constexpr uint32_t kB3Atom = kRope - kB3, kRopeAtom = 16384;
static_assert(OFF_ST1 + kRope + kRopeAtom + 16384 <= OFF_MISC, "second M atoms stay in shared memory");
// TMEM columns
constexpr uint32_t kColSn = 0, kColSr = 64, kColO = 128;  // context accumulator c at kColO + 64 c (c = 4: RoPE)
constexpr float kTau = 2.0f;           // lazy-rescale threshold (log2 units): p <= 2^kTau
constexpr float kWScale = 64.0f;       // 2^(8 - kTau): keeps the e4m3 weights <= 256 < 448

struct Misc {
    // per-head arrays first: they are read with 16-byte vector loads.  m_run / m_ref have two copies;
    // which one is current flips on a rescale.
    alignas(16) float m_run[2][kHeads];  // running max per head (log2 units), -inf before any valid row
    alignas(16) float m_ref[2][kHeads];  // the weights' reference: m_run, or 0 while that is -inf
    alignas(16) float c_head[kHeads];    // sm_scale * log2(e) * q_scale[h] (0 for padding heads)
    alignas(16) float red[4][kHeads];    // per-quadrant tile maxima / row sums
    union alignas(16) Phase {            // storage that is never live in two phases at once
        struct {
            float alpha[2][32];          // tile loop, per head half: rescale factors 2^(m_old - m_new)
            float delta[2][32];          // and the reference shifts m_ref_old - m_ref_new
        } tile;
        struct {
            float zsum[kHeads];          // epilogue: row sums per head
        } fin;
    } ph;
    uint64_t kv_full[2], kv_empty[2], s_full, s_free, p_full, pv_done, final_bar, q_full;
    uint64_t kv_blk[2][3];  // no-position block kb of a stage has been read by the context product
    uint32_t tmem_base;
    int abort_flag;
    float w_mul;     // kWScale / s_ref
    float out_mul;   // s_ref / kWScale
};
static_assert(OFF_MISC % 16 == 0 && offsetof(Misc, m_run) % 16 == 0 && offsetof(Misc, m_ref) % 16 == 0 &&
                  offsetof(Misc, red) % 16 == 0 && offsetof(Misc, ph) % 16 == 0 && offsetof(Misc, c_head) % 16 == 0,
              "vector accesses need 16-byte alignment");
static_assert(offsetof(Misc, kv_full) % 8 == 0, "mbarriers need 8-byte alignment");
constexpr uint32_t kSmemBytes = OFF_MISC + sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct MxArgs {
    const void *q_nope;          // [H][448]
    const void *q_rope;          // [H][64]
    int q_bf16, H, P, n_half;
    const float *k_scale;        // [T]
    int64_t T;
    float sm_scale_log2;
    float *ws;                   // partial sets [P][H]
    int *err_word;
    // written by mixed_prep_kernel: query images [n_half][kQImg], score factors [n_half * 64] (0 for a
    // padding head)
    const uint8_t *qimg;
    const float *c_head;
};

__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b) {  // a in the low half
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// four consecutive query values as f32 (bf16 or f32 storage; 8- or 16-byte aligned)
// 10 warps, one CTA per SM (220 KB of shared memory).
__global__ void __launch_bounds__(kThreads, 1)
    attn_mixed_tc_kernel(const __grid_constant__ CUtensorMap map_k8, const __grid_constant__ CUtensorMap map_k8b3,
                         const __grid_constant__ CUtensorMap map_kr, MxArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc &ms = *reinterpret_cast<Misc *>(smem + OFF_MISC);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if ((smem_u32(smem) & 1023u) != 0) {  // swizzled operands need 1024-byte alignment
        if (tid == 0 && a.err_word) atomicOr(a.err_word, (int)KV8_ERR_TIMEOUT);
        return;
    }
    const int part = blockIdx.x / a.n_half, half = blockIdx.x - part * a.n_half;
    const int64_t t0 = a.T * part / a.P, t1 = a.T * (part + 1) / a.P;
    const int n_tiles = (int)((t1 - t0 + kTile - 1) / kTile);

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&ms.kv_full[s], 1);
            mbar_init(&ms.kv_empty[s], 1);
            for (int kb = 0; kb < 3; ++kb) mbar_init(&ms.kv_blk[s][kb], 1);
        }
        mbar_init(&ms.s_full, 1);
        mbar_init(&ms.s_free, kSoftmaxThreads);
        mbar_init(&ms.p_full, kSoftmaxThreads);
        mbar_init(&ms.pv_done, 1);
        mbar_init(&ms.final_bar, 1);
        mbar_init(&ms.q_full, 1);
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
        // Each no-position block of a stage is refilled as soon as the context product of tile i-2 has
        // read it; block 3 and the RoPE block after the whole product.  The stage's full barrier is
        // re-armed only after the first release, which implies tile i-2's phase of it has completed.
        if (n_tiles > 0 && lane == 0) {
            prefetch_tensormap(&map_k8);
            prefetch_tensormap(&map_k8b3);
            prefetch_tensormap(&map_kr);
            int issued = 0, armed = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i & 1;
                uint8_t *st = smem + (s ? OFF_ST1 : OFF_ST0);
                const int y = (int)(t0 + (int64_t)i * kTile);
                const uint32_t ph = ((i >> 1) - 1) & 1;  // phase of tile i-2's release
                bool ok_p = true;
                for (int kb = 0; kb < 3 && ok_p; ++kb) {
                    if (i >= 2 && !(ok_p = mbar_wait(&ms.kv_blk[s][kb], ph, &ms.abort_flag, a.err_word))) break;
                    if (kb == 0) {
                        mbar_arrive_expect_tx(&ms.kv_full[s], kStage);
                        armed = i + 1;
                    }
                    tma_load_2d(st + kb * 16384, &map_k8, kb * 128, y, &ms.kv_full[s]);
                }
                if (ok_p && i >= 2) ok_p = mbar_wait(&ms.kv_empty[s], ph, &ms.abort_flag, a.err_word);
                if (!ok_p) break;
                tma_load_2d(st + kB3, &map_k8b3, 384, y, &ms.kv_full[s]);
                tma_load_2d(st + kRope, &map_kr, 0, y, &ms.kv_full[s]);
                issued = i + 1;
                if (i == 0) {
                    // the rows do not depend on the query prep; the query image does: it goes out after
                    // the first tile, so that the first score waits for one tile and the image only
                    grid_dependency_wait();
                    mbar_arrive_expect_tx(&ms.q_full, kQImg);
                    const uint8_t *src = a.qimg + (size_t)half * kQImg;
                    for (uint32_t o = 0; o < kQImg; o += 16384u)
                        bulk_load(smem + OFF_Q + o, src + o, kQImg - o < 16384u ? kQImg - o : 16384u, &ms.q_full);
                }
            }
            // every issued load lands before the CTA ends (a partly issued tile times out quickly, after
            // its issued blocks have landed)
            for (int i = (armed > 2 ? armed - 2 : 0); i < armed; ++i)
                mbar_wait(&ms.kv_full[i & 1], (i >> 1) & 1, nullptr, a.err_word,
                          i < issued ? 200000000ull : 20000000ull);
            if (issued >= 1) mbar_wait(&ms.q_full, 0, nullptr, a.err_word, 200000000ull);
        }
        __syncwarp();
    } else {
        // ============ prologue: the prep kernel's score factors, the rows' largest scale ============
        const int pt = tid - 32;  // 0..287
        grid_dependency_wait();
        // the largest row scale of this CTA's rows, read here (one round of loads beside the query image's
        // copy) rather than by the prep kernel, whose grid -- and with it the image -- then completes
        // sooner.  After the grid dependency: the step's append may just have written the last row.
        float mx = 0.f;
        for (int64_t t = t0 + pt; t < t1; t += 8 * kPrepThreads) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t tu = t + (int64_t)u * kPrepThreads;
                v[u] = tu < t1 ? __ldg(a.k_scale + tu) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) mx = fmaxf(mx, fabsf(v[u]));
        }
        mx = warp_max(mx);
        if (lane == 0) ms.red[0][warp - 1] = mx;  // scratch until the tile loop
        if (pt < kHeads) {
            ms.c_head[pt] = a.c_head[half * kHeads + pt];
            ms.m_run[0][pt] = ms.m_run[1][pt] = -INFINITY;
            ms.m_ref[0][pt] = ms.m_ref[1][pt] = 0.f;
        }
        named_sync(1, kPrepThreads);
        if (pt == 0) {
            float m = 0.f;
            for (int k = 0; k < kPrepThreads / 32; ++k) m = fmaxf(m, ms.red[0][k]);
            const float s_ref = fmaxf(m, 1e-30f);
            ms.w_mul = kWScale / s_ref;
            ms.out_mul = s_ref / kWScale;
        }
        named_sync(1, kPrepThreads);

        if (warp == 1) {
            // ================================ MMA issuer ================================
            if (lane == 0) {
                const uint32_t id_sn = idesc_e4m3_f32(128, 64, false, false);
                const uint32_t id_sr = idesc_bf16_f32(128, 64);
                const uint32_t id_pn = idesc_e4m3_f32(128, 64, true, true);
                const uint32_t id_pr = idesc_bf16_f32(128, 64, true, true);
                const uint32_t qb = sbase + OFF_Q;
                const bool rope_lo = !a.q_bf16;
                auto issue_score = [&](int i) {
                    const uint32_t st = sbase + ((i & 1) ? OFF_ST1 : OFF_ST0);
                    const uint32_t dn = tmem + kColSn, dr = tmem + kColSr;
#pragma unroll
                    for (int kb = 0; kb < 3; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f8f6f4(dn, smem_desc(st + kb * 16384 + kk * 32, 0, 1024, kSw128),
                                       smem_desc(qb + kb * 8192 + kk * 32, 0, 1024, kSw128), id_sn, (kb | kk) != 0);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        mma_f8f6f4(dn, smem_desc(st + kB3 + kk * 32, 0, 512, kSw64),
                                   smem_desc(qb + kQB3 + kk * 32, 0, 512, kSw64), id_sn, 1);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(dr, smem_desc(st + kRope + kk * 32, 0, 1024, kSw128),
                                 smem_desc(qb + kQR + kk * 32, 0, 1024, kSw128), id_sr, kk != 0);
                    if (rope_lo) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_bf16(dr, smem_desc(st + kRope + kk * 32, 0, 1024, kSw128),
                                     smem_desc(qb + kQRLo + kk * 32, 0, 1024, kSw128), id_sr, 1);
                    }
                    mma_commit(&ms.s_full);
                };
                auto issue_pv = [&](int j) {
                    const int s = j & 1;
                    const uint32_t st = sbase + (s ? OFF_ST1 : OFF_ST0);
                    const uint32_t whi = sbase + OFF_WHI, wlo = sbase + OFF_WLO, wb = sbase + OFF_WB;
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        const uint32_t d = tmem + kColO + 64u * ch;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // 32 rows per MMA; chunk 3 is the 64-byte-swizzled block with a second M atom
                            const uint64_t ad = ch < 3 ? smem_desc(st + ch * 16384 + kk * 4096, 0, 1024, kSw128)
                                                       : smem_desc(st + kB3 + kk * 2048, kB3Atom, 512, kSw64);
                            mma_f8f6f4(d, ad, smem_desc(whi + kk * 2048, 0, 512, kSw64), id_pn, (j | kk) != 0);
                            mma_f8f6f4(d, ad, smem_desc(wlo + kk * 2048, 0, 512, kSw64), id_pn, 1);
                        }
                        if (ch < 3) mma_commit(&ms.kv_blk[s][ch]);  // no-position block ch may be refilled
                    }
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // 16 rows per MMA
                        mma_bf16(tmem + kColO + 256u, smem_desc(st + kRope + kk * 2048, kRopeAtom, 1024, kSw128),
                                 smem_desc(wb + kk * 2048, 0, 1024, kSw128), id_pr, (j | kk) != 0);
                    mma_commit(&ms.kv_empty[s]);
                    mma_commit(&ms.pv_done);
                };
                // Issue whichever is ready, the context product first (it releases the row stage and the
                // weight buffers).  Score i needs tile i loaded and the score buffer read by the softmax of
                // tile i-1; PV j needs the weights of tile j.
                int ns = 0, np = 0;
                if (n_tiles > 0 && !mbar_wait(&ms.q_full, 0, &ms.abort_flag, a.err_word)) np = n_tiles;
                uint64_t t_last = globaltimer_ns();
                uint32_t spins = 0;
                while (np < n_tiles) {
                    if (np < ns && mbar_test_wait(&ms.p_full, np & 1)) {
                        tc_fence_after_sync();
                        issue_pv(np++);
                        spins = 0;
                        continue;
                    }
                    if (ns < n_tiles && mbar_test_wait(&ms.kv_full[ns & 1], (ns >> 1) & 1) &&
                        (ns == 0 || mbar_test_wait(&ms.s_free, (ns - 1) & 1))) {
                        tc_fence_after_sync();
                        issue_score(ns++);
                        spins = 0;
                        continue;
                    }
                    if ((++spins & 255u) == 0) {
                        const uint64_t now = globaltimer_ns();
                        if (ms.abort_flag) break;
                        if (spins > 256u && now - t_last > 2000000000ull) {  // no progress for 2 s
                            ms.abort_flag = 1;
                            if (a.err_word) atomicOr(a.err_word, (int)KV8_ERR_TIMEOUT);
                            break;
                        }
                    } else if (spins == 1) {
                        t_last = globaltimer_ns();
                    }
                }
                // all issued MMAs complete before the CTA tears down
                mma_commit(&ms.final_bar);
                mbar_wait(&ms.final_bar, 0, nullptr, a.err_word, 200000000ull);
            }
            __syncwarp();
        } else {
            // ============================ softmax + epilogue ============================
            // Each thread owns one tile row (TMEM lane) and the 32 heads of its head half.  The four
            // warps of a head half decide and rescale together through named barrier 2 + hh.  A wait
            // that gives up clears `ok`; the thread then skips its remaining waits but still reaches
            // every named barrier of every tile, so the other warps never wait for it.
            const int q = warp & 3;               // TMEM lane quadrant
            const int hh = (warp - 2) >> 2;       // which 32 of the CTA's 64 heads
            const int r = q * 32 + lane;          // row within the tile = TMEM lane
            const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
            const int bar_id = 2 + hh;
            const float w_mul = ms.w_mul;
            const float c_rope = a.sm_scale_log2;
            float z[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) z[j] = 0.f;
            float sc_next = n_tiles > 0 && t0 + r < t1 ? __ldg(a.k_scale + t0 + r) : -1.f;
            bool ok = true;
            bool seen = false;  // some valid row has been scored: every head's running max is finite
            int cur = 0;        // which copy of ms.m_run / ms.m_ref is current (uniform across the half)
            for (int i = 0; i < n_tiles; ++i) {
                const int64_t t = t0 + (int64_t)i * kTile + r;
                const float sc_t = sc_next;   // row scale, -1 for a row past the partition's end
                const bool valid = sc_t >= 0.f;
                sc_next = (i + 1 < n_tiles && t + kTile < t1) ? __ldg(a.k_scale + t + kTile) : -1.f;

                if (ok) ok = mbar_wait(&ms.s_full, i & 1, &ms.abort_flag, a.err_word);
                tc_fence_after_sync();
                uint32_t sn[32], sr[32];
                {
                    const uint32_t ta = tmem + lane_addr + 32u * hh;
                    tmem_ld_32x32b_x16(ta + kColSn, *reinterpret_cast<uint32_t(*)[16]>(sn));
                    tmem_ld_32x32b_x16(ta + kColSn + 16u, *reinterpret_cast<uint32_t(*)[16]>(sn + 16));
                    tmem_ld_32x32b_x16(ta + kColSr, *reinterpret_cast<uint32_t(*)[16]>(sr));
                    tmem_ld_32x32b_x16(ta + kColSr + 16u, *reinterpret_cast<uint32_t(*)[16]>(sr + 16));
                    tmem_wait_ld();
                }
                tc_fence_before_sync();
                mbar_arrive(&ms.s_free);

                // d = s - ref with s = sm_scale*log2(e) * (q_scale * k_scale * S_n + S_r); ref is the
                // running max, or 0 before any valid row
                float d[32];
                float dmax = -INFINITY;
                const float *mref = &ms.m_ref[cur][32 * hh];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float4 c4 = *reinterpret_cast<const float4 *>(&ms.c_head[32 * hh + 4 * j4]);
                    const float4 r4 = *reinterpret_cast<const float4 *>(mref + 4 * j4);
                    const float cj[4] = {c4.x, c4.y, c4.z, c4.w}, rj[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int j = 4 * j4 + u;
                        d[j] = fmaf(__uint_as_float(sn[j]), cj[u] * sc_t, fmaf(__uint_as_float(sr[j]), c_rope, -rj[u]));
                        dmax = fmaxf(dmax, d[j]);
                    }
                }
                if (!valid) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) d[j] = -INFINITY;
                    dmax = -INFINITY;
                }
                // lazy rescale: the half takes the slow path when some score exceeds its head's running
                // max by more than kTau, or while no valid row has been seen
                const bool slow = bar_red_or(bar_id, 128, dmax > kTau || !seen);
                bool any_alpha = false;
                if (slow) {
                    // tile max per head over this warp's 32 rows: butterfly transpose-reduction.  At
                    // step k each lane keeps the half of its heads selected by lane bit k and takes the
                    // max with the other half from lane ^ k; after 5 steps lane l holds head l's max.
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = d[j];
#pragma unroll
                    for (int k = 16; k >= 1; k >>= 1) {
                        const bool upper = (lane & k) != 0;
#pragma unroll
                        for (int j = 0; j < k; ++j) {
                            const float send = upper ? v[j] : v[j + k];
                            const float keep = upper ? v[j + k] : v[j];
                            v[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, k));
                        }
                    }
                    const int hj = 32 * hh + lane;  // lane l now speaks for head l of the half
                    ms.red[q][hj] = v[0];
                    named_sync(bar_id, 128);
                    const float ref_o = ms.m_ref[cur][hj], mo = ms.m_run[cur][hj];
                    const float tmax = fmaxf(fmaxf(ms.red[0][hj], ms.red[1][hj]), fmaxf(ms.red[2][hj], ms.red[3][hj])) + ref_o;
                    const float mn = mo == -INFINITY ? tmax : (tmax > mo + kTau ? tmax : mo);
                    const float al = (mo == -INFINITY || mn == mo) ? 1.f : ex2_approx(mo - mn);
                    const float ref_n = mn == -INFINITY ? 0.f : mn;
                    // the four quadrant warps write the same values
                    ms.m_run[cur ^ 1][hj] = mn;
                    ms.m_ref[cur ^ 1][hj] = ref_n;
                    ms.ph.tile.alpha[hh][lane] = al;
                    ms.ph.tile.delta[hh][lane] = ref_o - ref_n;
                    seen = __shfl_sync(0xffffffffu, mn, 0) != -INFINITY;  // the same for every head
                    any_alpha = __any_sync(0xffffffffu, al != 1.f);
                    __syncwarp();
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(&ms.ph.tile.alpha[hh][4 * j4]);
                        const float4 e4 = *reinterpret_cast<const float4 *>(&ms.ph.tile.delta[hh][4 * j4]);
                        d[4 * j4 + 0] += e4.x;
                        d[4 * j4 + 1] += e4.y;
                        d[4 * j4 + 2] += e4.z;
                        d[4 * j4 + 3] += e4.w;
                        z[4 * j4 + 0] *= a4.x;
                        z[4 * j4 + 1] *= a4.y;
                        z[4 * j4 + 2] *= a4.z;
                        z[4 * j4 + 3] *= a4.w;
                    }
                    cur ^= 1;
                }
                // weights: p = 2^d (row sum z); no-position w = p * k_scale * kWScale / s_ref as e4m3
                // hi + lo; RoPE w = p as bf16
                const float g = valid ? sc_t * w_mul : 0.f;
                uint32_t whi[8], wlo[8], wbf[16];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const float p0 = ex2_approx(d[4 * j4 + 0]), p1 = ex2_approx(d[4 * j4 + 1]);
                    const float p2 = ex2_approx(d[4 * j4 + 2]), p3 = ex2_approx(d[4 * j4 + 3]);
                    z[4 * j4 + 0] += p0;
                    z[4 * j4 + 1] += p1;
                    z[4 * j4 + 2] += p2;
                    z[4 * j4 + 3] += p3;
                    uint32_t h01, l01, h23, l23;
                    split_pair_h(p0 * g, p1 * g, h01, l01);
                    split_pair_h(p2 * g, p3 * g, h23, l23);
                    whi[j4] = h01 | (h23 << 16);
                    wlo[j4] = l01 | (l23 << 16);
                    wbf[2 * j4] = bf16x2_bits(p0, p1);
                    wbf[2 * j4 + 1] = bf16x2_bits(p2, p3);
                }
                if (i >= 1) {
                    // the previous context product must be done before the weight buffers are reused and
                    // before its accumulators are rescaled
                    if (ok) ok = mbar_wait(&ms.pv_done, (i - 1) & 1, &ms.abort_flag, a.err_word);
                    if (any_alpha) {
                        // rescale this half's columns of the context accumulators (lanes 64..127 of the
                        // two 64-dim accumulators hold nothing)
                        tc_fence_after_sync();
                        const int n_acc = q < 2 ? 5 : 3;
#pragma unroll 1
                        for (int c = 0; c < n_acc; ++c) {
                            const uint32_t ta = tmem + lane_addr + kColO + 64u * c + 32u * hh;
                            uint32_t o[32];
                            tmem_ld_32x32b_x16(ta, *reinterpret_cast<uint32_t(*)[16]>(o));
                            tmem_ld_32x32b_x16(ta + 16u, *reinterpret_cast<uint32_t(*)[16]>(o + 16));
                            tmem_wait_ld();
                            const float *al = ms.ph.tile.alpha[hh];
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {
                                const float4 a4 = *reinterpret_cast<const float4 *>(al + 4 * j4);
                                o[4 * j4 + 0] = __float_as_uint(__uint_as_float(o[4 * j4 + 0]) * a4.x);
                                o[4 * j4 + 1] = __float_as_uint(__uint_as_float(o[4 * j4 + 1]) * a4.y);
                                o[4 * j4 + 2] = __float_as_uint(__uint_as_float(o[4 * j4 + 2]) * a4.z);
                                o[4 * j4 + 3] = __float_as_uint(__uint_as_float(o[4 * j4 + 3]) * a4.w);
                            }
                            tmem_st_32x32b_x16(ta, *reinterpret_cast<const uint32_t(*)[16]>(o));
                            tmem_st_32x32b_x16(ta + 16u, *reinterpret_cast<const uint32_t(*)[16]>(o + 16));
                        }
                        tmem_wait_st();
                    }
                }
                *reinterpret_cast<uint4 *>(smem + OFF_WHI + sw64_offset(r, 32 * hh)) = make_uint4(whi[0], whi[1], whi[2], whi[3]);
                *reinterpret_cast<uint4 *>(smem + OFF_WHI + sw64_offset(r, 32 * hh + 16)) = make_uint4(whi[4], whi[5], whi[6], whi[7]);
                *reinterpret_cast<uint4 *>(smem + OFF_WLO + sw64_offset(r, 32 * hh)) = make_uint4(wlo[0], wlo[1], wlo[2], wlo[3]);
                *reinterpret_cast<uint4 *>(smem + OFF_WLO + sw64_offset(r, 32 * hh + 16)) = make_uint4(wlo[4], wlo[5], wlo[6], wlo[7]);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(smem + OFF_WB + sw128_offset(r, 64 * hh + 16 * c)) =
                        make_uint4(wbf[4 * c], wbf[4 * c + 1], wbf[4 * c + 2], wbf[4 * c + 3]);
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&ms.p_full);
            }

            // ================================ epilogue ================================
            grid_launch_dependents();  // the merge may start launching
            if (ok && n_tiles > 0) ok = mbar_wait(&ms.pv_done, (n_tiles - 1) & 1, &ms.abort_flag, a.err_word);
            tc_fence_after_sync();
            // row sums per head over the warp's 32 rows: butterfly transpose-reduction (lane l ends with
            // head l's sum), then over the 4 quadrants
#pragma unroll
            for (int k = 16; k >= 1; k >>= 1) {
                const bool upper = (lane & k) != 0;
#pragma unroll
                for (int j = 0; j < k; ++j) {
                    const float send = upper ? z[j] : z[j + k];
                    const float keep = upper ? z[j + k] : z[j];
                    z[j] = keep + __shfl_xor_sync(0xffffffffu, send, k);
                }
            }
            ms.red[q][32 * hh + lane] = z[0];
            named_sync(bar_id, 128);
            if (q == 0) {
                const int h = 32 * hh + lane;
                ms.ph.fin.zsum[h] = ms.red[0][h] + ms.red[1][h] + ms.red[2][h] + ms.red[3][h];
            }
            named_sync(bar_id, 128);
            if (ok) {
                const float out_mul = ms.out_mul;
                PartialView pv(a.ws, 1, a.P, a.H);
                // accumulators 0..3: no-position dims 128c + lane (the last only lanes 0..63); 4: RoPE
                // dims 448 + lane (lanes 0..63)
                const int n_acc = q < 2 ? 5 : 3;
#pragma unroll 1
                for (int c = 0; c < n_acc; ++c) {
                    const float mul = c < 4 ? out_mul : 1.f;
                    const int dd = c < 4 ? 128 * c + r : kMxNope + r;
                    uint32_t o[32];  // this half's 32 heads of accumulator c, one TMEM round trip
                    if (n_tiles > 0) {
                        tmem_ld_32x32b_x16(tmem + lane_addr + kColO + 64u * c + 32u * hh, *reinterpret_cast<uint32_t(*)[16]>(o));
                        tmem_ld_32x32b_x16(tmem + lane_addr + kColO + 64u * c + 32u * hh + 16u,
                                           *reinterpret_cast<uint32_t(*)[16]>(o + 16));
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = 0u;
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int hg = half * kHeads + 32 * hh + j;
                        if (hg < a.H) pv.cl[((int64_t)part * a.H + hg) * kKL + dd] = __uint_as_float(o[j]) * mul;
                    }
                }
                if (q == 0) {
                    const int hg = half * kHeads + 32 * hh + lane;
                    if (hg < a.H) {
                        const int64_t pidx = (int64_t)part * a.H + hg;
                        pv.m[pidx] = n_tiles > 0 ? ms.m_run[cur][32 * hh + lane] : -INFINITY;  // -inf: no row
                        pv.z[pidx] = ms.ph.fin.zsum[32 * hh + lane];
                    }
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// Query prep, the decode kernel's programmatic predecessor.  Warp w of block g (g < n_groups) takes head
// 8g + w: its no-position part goes through the row quantizer's f32 steps (the bytes the cache quantizer
// would give) into K-major e4m3 rows of its head half's image, its RoPE part into bf16 rows (an f32 query
// also gets the lo piece x - bf16(x)), and its score factor sm_scale*log2(e)*q_scale (a padding head gets
// zeros).
struct MxPrepArgs {
    const void *q_nope, *q_rope;
    int q_bf16, H, n_groups, P;
    float sm_scale_log2;
    const float *k_scale;
    int64_t T;
    uint8_t *img;     // [n_half][kQImg]
    float *c_head;    // [n_half * 64]
};
constexpr int kMxPrepThreads = 256;  // 8 warps, one head each

__global__ void __launch_bounds__(kMxPrepThreads) mixed_prep_kernel(MxPrepArgs a) {
    // launched as a programmatic dependent of whatever came before on the stream: nothing is read until
    // that grid has completed; then the decode kernel may start its row loads while this runs
    grid_dependency_wait();
    grid_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    {
        const int hg = (int)blockIdx.x * (kMxPrepThreads / 32) + warp;
        const int half = hg / kHeads, h = hg - half * kHeads;
        uint8_t *img = a.img + (size_t)half * kQImg;
        constexpr int kF4 = kMxNope / 4;  // 112 groups of four, up to 4 per lane
        // every load is issued before any is converted (raw bits: f32 16 bytes, bf16 8 bytes in .x and
        // .y), so the five loads share one memory round trip
        uint4 raw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int f = j * 32 + lane;
            raw[j] = make_uint4(0u, 0u, 0u, 0u);
            if (hg < a.H && f < kF4) {
                const int64_t i = (int64_t)hg * kMxNope + 4 * f;
                if (a.q_bf16) {
                    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(a.q_nope) + i));
                    raw[j] = make_uint4(u.x, u.y, 0u, 0u);
                } else {
                    raw[j] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const float *>(a.q_nope) + i));
                }
            }
        }
        uint2 rraw = make_uint2(0u, 0u);  // RoPE values 2*lane, 2*lane + 1
        if (hg < a.H) {
            const int64_t e = (int64_t)hg * kMxRope + 2 * lane;
            if (a.q_bf16)
                rraw.x = __ldg(reinterpret_cast<const uint32_t *>(static_cast<const __nv_bfloat16 *>(a.q_rope) + e));
            else
                rraw = __ldg(reinterpret_cast<const uint2 *>(static_cast<const float *>(a.q_rope) + e));
        }
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (a.q_bf16) {
                const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw[j].x));
                const float2 hi2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw[j].y));
                v[j] = make_float4(lo.x, lo.y, hi2.x, hi2.y);
            } else {
                v[j] = make_float4(__uint_as_float(raw[j].x), __uint_as_float(raw[j].y), __uint_as_float(raw[j].z),
                                   __uint_as_float(raw[j].w));
            }
        }
        const float2 rp = a.q_bf16 ? __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&rraw.x))
                                   : make_float2(__uint_as_float(rraw.x), __uint_as_float(rraw.y));
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            amax = finite_abs_max(amax, v[j].x);
            amax = finite_abs_max(amax, v[j].y);
            amax = finite_abs_max(amax, v[j].z);
            amax = finite_abs_max(amax, v[j].w);
        }
        amax = warp_max(amax);
        float pre, mul, qs;
        row_quant_factors(amax, pre, mul, qs);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int f = j * 32 + lane;
            if (f < kF4) {
                const uint32_t byte = 4u * (uint32_t)f;
                const uint32_t off = byte < 384u ? (byte >> 7) * 8192u + sw128_offset(h, byte & 127u)
                                                 : kQB3 + sw64_offset(h, byte - 384u);
                *reinterpret_cast<uint32_t *>(img + off) = enc4(scale4(v[j], pre, mul));
            }
        }
        const uint32_t hi = bf16x2_bits(rp.x, rp.y);
        const float2 back = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hi));
        *reinterpret_cast<uint32_t *>(img + kQR + sw128_offset(h, 4u * lane)) = hi;
        if (!a.q_bf16) *reinterpret_cast<uint32_t *>(img + kQRLo + sw128_offset(h, 4u * lane)) = bf16x2_bits(rp.x - back.x, rp.y - back.y);
        if (lane == 0) a.c_head[hg] = hg < a.H ? a.sm_scale_log2 * qs : 0.f;
    }
}

}  // namespace

int mixed_partitions(int H, int64_t T) {
    // one wave of tensor-core CTAs on the current device (one per SM: a CTA per partition and 64-head
    // half), at least 128 rows per partition
    const int64_t sms = device_sm_count();
    const int64_t cap = H > kHeads ? sms / 2 : sms;
    const int64_t p = (T + kTile - 1) / kTile;
    return (int)(p < cap ? p : (cap < 1 ? 1 : cap));
}

size_t mixed_scratch_bytes(int H, int P) {
    // query images and score factors (each 256-byte aligned), then P floats that nothing writes any more
    // (kept so that the workspace size stays what earlier callers sized)
    const size_t n_half = H > kHeads ? 2 : 1;
    return n_half * kQImg + ((n_half * kHeads * sizeof(float) + 255) & ~(size_t)255) +
           (((size_t)P * sizeof(float) + 255) & ~(size_t)255);
}

// Tensor maps over the cache: the no-position bytes [T][448] (128-column boxes with the 128-byte swizzle,
// and a 64-column box at column 384 with the 64-byte swizzle) and the RoPE rows [T][128 bytes] (128-byte
// swizzle); rows past T read as zeros.  Returns cudaErrorNotSupported if the tensor-map encoder is
// unavailable.
cudaError_t launch_attn_mixed(const void *q_nope, const void *q_rope, int q_bf16, int H, const uint8_t *k8,
                              const float *k_scale, const void *k_rope, int64_t T, float sm_scale_log2, int P,
                              float *ws, void *scratch, int *err_word, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    if (T < 1 || T > 0x7fffffffLL || P < 1) return cudaErrorInvalidValue;  // row coordinates are 32-bit
    CUtensorMap m8, m8b3, mr;
    const cuuint64_t dims8[2] = {(cuuint64_t)kMxNope, (cuuint64_t)T}, str8[1] = {(cuuint64_t)kMxNope};
    const cuuint64_t dimsr[2] = {(cuuint64_t)(2 * kMxRope), (cuuint64_t)T}, strr[1] = {(cuuint64_t)(2 * kMxRope)};
    const cuuint32_t box8[2] = {128, kTile}, box3[2] = {64, kTile}, boxr[2] = {128, kTile}, es[2] = {1, 1};
    void *b8 = const_cast<uint8_t *>(k8);
    void *br = const_cast<void *>(k_rope);
    if (encode(&m8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, b8, dims8, str8, box8, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS ||
        encode(&m8b3, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, b8, dims8, str8, box3, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS ||
        encode(&mr, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, br, dimsr, strr, boxr, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    MxArgs a{};
    a.q_nope = q_nope;
    a.q_rope = q_rope;
    a.q_bf16 = q_bf16;
    a.H = H;
    a.P = P;
    a.n_half = H > kHeads ? 2 : 1;
    a.k_scale = k_scale;
    a.T = T;
    a.sm_scale_log2 = sm_scale_log2;
    a.ws = ws;
    a.err_word = err_word;
    MxPrepArgs pa{};
    pa.q_nope = q_nope;
    pa.q_rope = q_rope;
    pa.q_bf16 = q_bf16;
    pa.H = H;
    pa.n_groups = a.n_half * kHeads / (kMxPrepThreads / 32);
    pa.P = P;
    pa.sm_scale_log2 = sm_scale_log2;
    pa.k_scale = k_scale;
    pa.T = T;
    pa.img = static_cast<uint8_t *>(scratch);
    pa.c_head = reinterpret_cast<float *>(pa.img + (size_t)a.n_half * kQImg);
    a.qimg = pa.img;
    a.c_head = pa.c_head;
    cudaError_t e =
        cudaFuncSetAttribute(attn_mixed_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t pcfg = {};
    pcfg.gridDim = dim3((unsigned)pa.n_groups);
    pcfg.blockDim = dim3(kMxPrepThreads);
    pcfg.stream = st;
    cudaLaunchAttribute pattr[1];
    pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pattr[0].val.programmaticStreamSerializationAllowed = 1;
    pcfg.attrs = pattr;
    pcfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&pcfg, mixed_prep_kernel, pa)) != cudaSuccess) return e;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(P * a.n_half));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((e = cudaLaunchKernelEx(&cfg, attn_mixed_tc_kernel, m8, m8b3, mr, a)) != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kv8
