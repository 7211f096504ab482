// attn_tc.cu -- absorbed MLA attention over e4m3 cache rows on the 5th-generation tensor cores
// (tcgen05, sm_103a), for bf16 queries.
//
// Page "KV8 long-context CUDA: fp8 device shadow, split-T kernels, DSA-aware gather":
//   first commit message  -- score = sm_scale * s_t * q.e4m3(row) (the row scale hoisted out of the dot);
//                            context = softmax-weighted sum of s_t * e4m3(Lc_t) (the latent row serves
//                            as the key and as the value).
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
//   context O^T[d][n]  += sum_t  V8[t][d] * W^T[t][n]        M = 128 dims (x4 chunks), K = 128 rows
//           A = the same cache bytes read MN-major (V^T), B = the weights MN-major.  Dims 0..255 take
//           the hi and lo weights side by side (N = 128, one accumulator column per head and piece,
//           summed at the end); dims 256..511 add both pieces into one accumulator (two N = 64 passes).
//           An MMA reading A MN-major costs about the same at N = 64 as at N = 128, so the wide passes
//           halve the first two chunks' tensor time; TMEM has room for two of them.
//
// Rows reach shared memory by TMA as 128-row tiles (dense and causal ranges); selected rows (DSA) by
// cp.async, one row per warp instruction (32 lanes x 16 bytes), written into the same swizzled image
// (as fast as four-row TMA gathers, and it leaves the copy engine to the query image).
//
// Warps: 0 = TMA producer, 1 = MMA issuer (and TMEM owner), 2..17 = softmax / epilogue in four groups of
// four warps (one per TMEM lane quadrant), each group owning 16 of the CTA's 64 heads.
// Shared memory (231 KB): query image 72 KB, two 72 KB row stages (the weights' hi piece reuses the
// stage's rope block once the score has read it), weights' lo piece 8 KB, barriers and scratch.
// TMEM (512 columns): one 128-column score buffer (hi / lo query pieces side by side), then six 64-column
// context accumulators: dims 0..127 hi, lo; dims 128..255 hi, lo; dims 256..383; dims 384..511.
// Every mbarrier wait is bounded in time; a timeout sets KV8_ERR_TIMEOUT.  The softmax warps then skip
// their remaining waits but still pass every named barrier of every tile, so the CTA winds down without
// hanging.
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
constexpr int kHG = 16;                // heads per softmax group (four warps, one per TMEM lane quadrant)
constexpr int kNG = kHeadsPerCta / kHG;  // softmax groups
constexpr int kThreads = 64 + 128 * kNG; // warp 0 TMA, warp 1 MMA, then the softmax groups
constexpr int kSoftmaxThreads = 128 * kNG;
constexpr int kPrepThreads = 288;      // warps 1..9: the in-kernel query prep's workers
constexpr int kPrepAll = kThreads - 32;  // warps 1..: every thread that waits for the prologue
static_assert(kPrepAll / 32 <= 32, "one prologue maximum slot per warp");
static_assert(kHG == 16 || kHG == 32, "a softmax thread's heads: one or two 16-column TMEM loads");
constexpr uint32_t kImg = 73728;       // 4 x 16 KB (SW128, 128 B per row) + 8 KB (SW64, 64 B per row)
constexpr uint32_t kRcOff = 65536;     // rope block inside an image / stage
constexpr uint32_t OFF_Q = 0, OFF_ST0 = kImg, OFF_ST1 = 2 * kImg, OFF_PLO = 3 * kImg, OFF_MISC = 3 * kImg + 8192;
constexpr float kTau = 2.0f;           // lazy-rescale threshold (log2 units): p <= 2^kTau
constexpr float kWScale = 64.0f;       // 2^(8 - kTau): keeps w <= 256 < 448 (e4m3 max)
constexpr uint32_t TM_S = 0;           // score: columns 0..63 hi piece, 64..127 lo piece
constexpr uint32_t TM_O = 128;         // context piece k (0..5) at TM_O + 64k, see the header
constexpr int kOPieces = 6;

struct Misc {
    // per-head arrays first: they are read with 16-byte vector loads.  m_run / m_ref have two copies;
    // which one is current flips on a rescale.
    alignas(16) float m_run[2][kHeadsPerCta];  // running max per head (log2 units), -inf before any valid row
    alignas(16) float m_ref[2][kHeadsPerCta];  // the weights' reference: m_run, or 0 while that is -inf
    alignas(16) float c_head[kHeadsPerCta];    // sm_scale * log2(e) * 2^-e_h per head (0 for padding heads)
    alignas(16) float red[4][kHeadsPerCta];    // per-quadrant tile maxima / row sums
    union alignas(16) Phase {                  // storage that is never live in two phases at once
        struct {
            int qmax_bits[kHeadsPerCta];       // prologue: per-head max |q| (bits of a non-negative float)
            float wred[2][16];                 // prologue: per-warp maxima (flat: one slot per warp 1..17)
        } pro;
        struct {
            float alpha[kNG][kHG];             // tile loop, per softmax group: rescale factors 2^(m_old - m_new)
            float delta[kNG][kHG];             // and the reference shifts m_ref_old - m_ref_new
        } tile;
        struct {
            float zsum[kHeadsPerCta];          // epilogue: row sums per head
            float zinv[kHeadsPerCta];          // and the direct output's factors s_ref / kWScale / zsum
        } fin;
    } ph;
    uint64_t kv_full[2], kv_empty[2], s_full, s_free, p_full, lo_free, final_bar, q_full;
    uint64_t pv_done[2];    // context product of a tile of that parity done (one phase per two tiles)
    uint64_t kv_blk[2][4];  // latent block kb of a stage has been read by the context product
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

struct TcArgs {
    const __nv_bfloat16 *q_lat;  // [B][H][512]
    const __nv_bfloat16 *q_rope; // [B][H][64]
    int B, H, P, n_half;
    const uint8_t *kv8;          // cache rows [..][576] (selected rows are copied from here directly)
    const float *kv_scale;
    int64_t T;
    int64_t pos0;                // causal: item b attends rows [0, pos0 + b]; -1: rows [0, T)
    const int32_t *lens;         // batched dense decode: item b attends its rows [0, lens[b]) (clamped to T)
    const int32_t *idx;          // selection: item b attends rows idx[b][0..NS) of its own cache (else null)
    int NS;
    int64_t seq_stride_rows;     // selection: rows between consecutive items' caches
    float sm_scale_log2;
    float *ws;                   // partial sets, or nullptr
    float *out;                  // direct normalised output when ws == nullptr
    int *err_word;
    // written by tc_prep_kernel (decode): query images [n_half][kImg], per-head factors [n_half*64],
    // per-partition row-scale maxima [P].  Null: the kernel prepares its own queries (prefill).
    const uint8_t *qimg;
    const float *c_head;
    const float *smax;
};

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

// 18 warps: a sub-partition holding 5 warps caps a thread at 96 registers (16K registers each).
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
    // the list this CTA walks: positions [t0, t1) of rows 0..n_rows-1 (dense / causal) or of idx[b] (selection)
    const int64_t n_rows = a.idx           ? (int64_t)a.NS
                           : a.pos0 >= 0   ? ((a.pos0 + b + 1 < a.T) ? a.pos0 + b + 1 : a.T)
                           : a.lens        ? min((int64_t)max(__ldg(a.lens + b), 0), a.T)
                                           : a.T;
    const int32_t *idx_b = a.idx ? a.idx + (int64_t)b * a.NS : nullptr;
    // each item's cache starts seq_stride_rows after the previous one (0 for one cache shared by all items)
    const int64_t seq_base = (int64_t)b * a.seq_stride_rows;
    const int64_t t0 = n_rows * part / a.P, t1 = n_rows * (part + 1) / a.P;
    const int n_tiles = (int)((t1 - t0 + kTile - 1) / kTile);

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&ms.kv_full[s], idx_b ? 32 : 1);  // selected rows: one cp.async arrival per producer lane
            mbar_init(&ms.kv_empty[s], 1);
            for (int kb = 0; kb < 4; ++kb) mbar_init(&ms.kv_blk[s][kb], 1);
            mbar_init(&ms.pv_done[s], 1);
        }
        mbar_init(&ms.s_full, 1);
        mbar_init(&ms.s_free, kSoftmaxThreads);
        mbar_init(&ms.p_full, kSoftmaxThreads);
        mbar_init(&ms.lo_free, 1);
        mbar_init(&ms.final_bar, 1);
        mbar_init(&ms.q_full, 1);
        ms.abort_flag = 0;
        fence_barrier_init();
        if (!idx_b && n_tiles > 0) {
            // dense rows: tile 0's copies go out now (this is the producer lane), before the CTA-wide
            // barrier -- they depend on nothing the other warps set up
            const int y = (int)(seq_base + t0);
            mbar_arrive_expect_tx(&ms.kv_full[0], kImg);
            for (int kb = 0; kb < 4; ++kb) tma_load_2d(smem + OFF_ST0 + kb * 16384, &map_lc, kb * 128, y, &ms.kv_full[0]);
            tma_load_2d(smem + OFF_ST0 + kRcOff, &map_rc, 512, y, &ms.kv_full[0]);
        }
    }
    if (warp == 1) {
        tmem_alloc(&ms.tmem_base, 512);
        tmem_relinquish();
    }
    if (tid < kHeadsPerCta) ms.ph.pro.qmax_bits[tid] = 0;
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t sbase = smem_u32(smem);

    if (warp == 0) {
        // ================================ TMA producer ================================
        // Dense rows: lane 0 issues the tile copies and does the waits.  Selection: the whole warp reads
        // the tile's 128 row indices (4 per lane) and copies the rows, one row per instruction.
        if (n_tiles > 0) {
            if (lane == 0) {
                prefetch_tensormap(&map_lc);
                prefetch_tensormap(&map_rc);
            }
            int issued = 0, armed = (!idx_b && n_tiles > 0) ? 1 : 0;  // dense tile 0: issued at the start
            // the query image (which depends on the query prep) goes out after the first tile's rows (which
            // do not), so that the first score waits for one tile and the image only
            const int q_at = n_tiles > 1 ? 1 : 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i & 1;
                if (lane == 0 && i == q_at && a.qimg) {
                    grid_dependency_wait();
                    mbar_arrive_expect_tx(&ms.q_full, kImg);
                    const uint8_t *src = a.qimg + ((size_t)b * a.n_half + half) * kImg;
                    for (int kb = 0; kb < 4; ++kb) bulk_load(smem + OFF_Q + kb * 16384, src + kb * 16384, 16384, &ms.q_full);
                    bulk_load(smem + OFF_Q + kRcOff, src + kRcOff, 8192, &ms.q_full);
                }
                uint8_t *st = smem + (s ? OFF_ST1 : OFF_ST0);
                const int64_t p0 = t0 + (int64_t)i * kTile;
                const uint32_t ph = ((i >> 1) - 1) & 1;  // phase of tile i-2's release
                bool ok_p = true;
                if (!idx_b) {
                    // each latent block is refilled as soon as the context product of tile i-2 has read
                    // it; the rope block also holds tile i-2's weights and is refilled after the whole
                    // product.  The stage's full barrier is re-armed only after the first release: that
                    // implies tile i-2's phase of it has completed (one arrival per phase).
                    if (lane == 0 && i > 0) {
                        const int y = (int)(seq_base + p0);
                        for (int kb = 0; kb < 4 && ok_p; ++kb) {
                            if (i >= 2 && !(ok_p = mbar_wait(&ms.kv_blk[s][kb], ph, &ms.abort_flag, a.err_word))) break;
                            if (kb == 0) {
                                mbar_arrive_expect_tx(&ms.kv_full[s], kImg);
                                armed = i + 1;
                            }
                            tma_load_2d(st + kb * 16384, &map_lc, kb * 128, y, &ms.kv_full[s]);
                        }
                        if (ok_p && i >= 2) ok_p = mbar_wait(&ms.kv_empty[s], ph, &ms.abort_flag, a.err_word);
                        if (ok_p) tma_load_2d(st + kRcOff, &map_rc, 512, y, &ms.kv_full[s]);
                    }
                } else {
                    // rows of this tile: invalid or past-the-end entries fetch row 0 of the item's cache
                    // (the softmax masks them).  The stage is refilled once tile i-2's context product is done.
                    int rows[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int64_t pos = p0 + 4 * lane + k;
                        int r = pos < t1 ? __ldg(idx_b + pos) : 0;
                        if (r < 0 || (int64_t)r >= a.T) r = 0;
                        rows[k] = (int)(seq_base + r);
                    }
                    if (lane == 0 && i >= 2) ok_p = mbar_wait(&ms.kv_empty[s], ph, &ms.abort_flag, a.err_word);
                    ok_p = __shfl_sync(0xffffffffu, ok_p, 0);
                    if (ok_p) {
                        // the context product's reads of this stage are complete; order them before the
                        // copies' writes (another proxy)
                        fence_proxy_async_smem();
                        armed = i + 1;
                        // latent rows one per instruction: lane l copies bytes 16l..16l+15 (latent block l/8)
                        // into the 128-byte-swizzled image the tile copies would make
                        const uint8_t *kv = a.kv8;
#pragma unroll 1
                        for (int r4 = 0; r4 < 32; ++r4) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const int r = 4 * r4 + k;
                                const int row = __shfl_sync(0xffffffffu, rows[k], r4);
                                cp_async_16(st + (lane >> 3) * 16384 + sw128_offset((uint32_t)r, (uint32_t)(lane & 7) * 16u),
                                            kv + (int64_t)row * kRow + lane * 16);
                            }
                        }
                        // rope bytes: 64 per row, eight rows per instruction (lane l: row r0 + l/4, chunk l%4)
#pragma unroll 1
                        for (int r0 = 0; r0 < kTile; r0 += 8) {
                            const int r = r0 + (lane >> 2), src_lane = r >> 2, k = r & 3;
                            const int c0 = __shfl_sync(0xffffffffu, rows[0], src_lane);
                            const int c1 = __shfl_sync(0xffffffffu, rows[1], src_lane);
                            const int c2 = __shfl_sync(0xffffffffu, rows[2], src_lane);
                            const int c3 = __shfl_sync(0xffffffffu, rows[3], src_lane);
                            const int row = k == 0 ? c0 : k == 1 ? c1 : k == 2 ? c2 : c3;
                            cp_async_16(st + kRcOff + sw64_offset((uint32_t)r, (uint32_t)(lane & 3) * 16u),
                                        kv + (int64_t)row * kRow + kKL + (lane & 3) * 16);
                        }
                        // one arrival per lane (the barrier expects 32 for selected rows) when its copies land
                        cp_async_mbar_arrive(&ms.kv_full[s]);
                    }
                }
                ok_p = __shfl_sync(0xffffffffu, ok_p, 0);
                if (!ok_p) break;
                issued = i + 1;
            }
            if (lane == 0) {
                // every issued load must land before the CTA ends (a partly issued tile times out
                // quickly, after its issued blocks have landed)
                for (int i = (armed > 2 ? armed - 2 : 0); i < armed; ++i)
                    mbar_wait(&ms.kv_full[i & 1], (i >> 1) & 1, nullptr, a.err_word,
                              i < issued ? 200000000ull : 20000000ull);
                if (a.qimg && issued > 0) mbar_wait(&ms.q_full, 0, nullptr, a.err_word, 200000000ull);
            }
        }
        __syncwarp();
    } else {
        // ======================= prologue: query image, row-scale max =======================
        const int pt = tid - 32;  // 0..kPrepAll-1; the query-prep workers are pt < kPrepThreads
        float smax = 0.f;
        if (a.qimg) {
            // decode: the prep kernel wrote the query image (loaded by the producer) and the factors
            grid_dependency_wait();
            if (pt < kHeadsPerCta) ms.c_head[pt] = a.c_head[(b * a.n_half + half) * kHeadsPerCta + pt];
            if (idx_b) {
                smax = a.smax[b * a.P + part];
            } else {
                // dense rows: the largest row scale of this CTA's rows, read here (one round of loads,
                // beside the query image's copy) rather than by the prep kernel, whose grid -- and with it
                // the query image -- then completes sooner.  After the grid dependency: the step's append
                // may just have written the last row's scale.
                const float *sc = a.kv_scale + seq_base;
                for (int64_t t = t0 + pt; t < t1; t += 8 * kPrepAll) {
                    float v[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int64_t tu = t + (int64_t)u * kPrepAll;
                        v[u] = tu < t1 ? __ldg(sc + tu) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < 8; ++u) smax = fmaxf(smax, fabsf(v[u]));
                }
                smax = warp_max(smax);
                float *wr = &ms.ph.pro.wred[0][0];  // 32 slots for the prologue's 17 warps
                if (lane == 0) wr[warp - 1] = smax;
                named_sync(1, kPrepAll);
                smax = 0.f;
                for (int k = 0; k < kPrepAll / 32; ++k) smax = fmaxf(smax, wr[k]);
            }
        } else {
            // prefill: each CTA prepares its own 64 heads (the image is reused for all its tiles)
            constexpr int kItems = kHeadsPerCta * 36 / kPrepThreads;  // 8 chunks of 16 query elements
            static_assert(kHeadsPerCta * 36 == kItems * kPrepThreads, "query chunks split evenly");
            const bool worker = pt < kPrepThreads;
            // query chunk k of this thread (16 bf16 values as two uint4), zeros for a padding head; loaded
            // before the barrier for the maxima and again after it for the split (not held across it)
            auto load_chunk = [&](int k, uint4 &u0, uint4 &u1) {
                const int it = pt + k * kPrepThreads, h = it / 36, ch = it - h * 36;
                const int hg = half * kHeadsPerCta + h;
                u0 = u1 = make_uint4(0u, 0u, 0u, 0u);
                if (worker && hg < a.H) {
                    const __nv_bfloat16 *src = ch < 32 ? a.q_lat + ((int64_t)b * a.H + hg) * kKL + ch * 16
                                                       : a.q_rope + ((int64_t)b * a.H + hg) * kKR + (ch - 32) * 16;
                    u0 = __ldg(reinterpret_cast<const uint4 *>(src));
                    u1 = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
                }
            };
            static_assert(kItems % 4 == 0, "query chunks in rounds of four");
#pragma unroll 1
            for (int k0 = 0; k0 < kItems; k0 += 4) {
                uint4 qv[4][2];
#pragma unroll
                for (int u = 0; u < 4; ++u) load_chunk(k0 + u, qv[u][0], qv[u][1]);
#pragma unroll
                for (int u = 0; u < 4 && worker; ++u) {
                    const int k = u;
                    const int it = pt + (k0 + u) * kPrepThreads, h = it / 36;
                    const uint32_t w[8] = {qv[k][0].x, qv[k][0].y, qv[k][0].z, qv[k][0].w,
                                           qv[k][1].x, qv[k][1].y, qv[k][1].z, qv[k][1].w};
                    float mx = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
                        mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
                    }
                    atomicMax(&ms.ph.pro.qmax_bits[h], __float_as_int(mx));  // non-negative floats order like ints
                }
            }
            for (int64_t t = t0 + pt; worker && t < t1; t += 8 * kPrepThreads) {
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t tu = t + (int64_t)u * kPrepThreads;
                    v[u] = tu < t1 ? __ldg(a.kv_scale + tu) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) smax = fmaxf(smax, fabsf(v[u]));
            }
            smax = warp_max(smax);
            if (lane == 0 && pt < kPrepThreads) ms.ph.pro.wred[1][warp - 1] = smax;
            named_sync(1, kPrepAll);
            smax = 0.f;
            for (int k = 0; k < 9; ++k) smax = fmaxf(smax, ms.ph.pro.wred[1][k]);
            // q_h * 2^e_h lies in [128, 256): every bf16 value splits exactly into e4m3 hi + lo (down to
            // the e4m3 subnormal step); the score is rescaled by 2^-e_h.
#pragma unroll 2
            for (int k = 0; k < kItems && worker; ++k) {
                const int it = pt + k * kPrepThreads, h = it / 36, ch = it - h * 36;
                uint4 u0, u1;
                load_chunk(k, u0, u1);
                const float qmax = __int_as_float(ms.ph.pro.qmax_bits[h]);
                int E = 0;
                if (qmax > 0.f) frexpf(qmax, &E);
                const int sh = qmax > 0.f ? 8 - E : 0;  // values are scaled, not a 2^sh factor: it may overflow
                const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int e2 = 0; e2 < 8; ++e2) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e2]));
                    uint32_t ph, pl;
                    split_pair(ldexpf(f.x, sh), ldexpf(f.y, sh), ph, pl);
                    hi[e2 >> 1] |= ph << ((e2 & 1) * 16);
                    lo[e2 >> 1] |= pl << ((e2 & 1) * 16);
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
            if (pt < kHeadsPerCta) {
                const int hg = half * kHeadsPerCta + pt;
                const float qmax = __int_as_float(ms.ph.pro.qmax_bits[pt]);
                int E = 0;
                if (qmax > 0.f) frexpf(qmax, &E);
                ms.c_head[pt] = hg < a.H ? (qmax > 0.f ? ldexpf(a.sm_scale_log2, E - 8) : a.sm_scale_log2) : 0.f;
            }
        }
        if (pt < kHeadsPerCta) {
            ms.m_run[0][pt] = ms.m_run[1][pt] = -INFINITY;
            ms.m_ref[0][pt] = ms.m_ref[1][pt] = 0.f;
        }
        if (pt == 0) {
            const float s_ref = fmaxf(smax, 1e-30f);
            ms.w_mul = kWScale / s_ref;
            ms.out_mul = s_ref / kWScale;
        }
        fence_proxy_async_smem();
        named_sync(1, kPrepAll);

        if (warp == 1) {
            // ================================ MMA issuer ================================
            if (lane == 0) {
                const uint32_t id_s = idesc_e4m3_f32(128, 128, false, false);
                const uint32_t id_pv = idesc_e4m3_f32(128, 64, true, true);
                const uint32_t id_pw = idesc_e4m3_f32(128, 128, true, true);
                const uint32_t qb = sbase + OFF_Q;
                auto issue_score = [&](int i) {
                    const int s = i & 1;
                    const uint32_t st = sbase + (s ? OFF_ST1 : OFF_ST0);
                    // S^T = K8 [Q_hi; Q_lo]^T in one N = 128 pass: columns 0..63 hold the hi piece's
                    // scores, 64..127 the lo piece's (one pass reads the rows once; two N = 64 passes
                    // into one accumulator take about 60% longer on the tensor cores)
                    const uint32_t d = tmem + TM_S;
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f8f6f4(d, smem_desc(st + kb * 16384 + kk * 32, 0, 1024, kSw128),
                                       smem_desc(qb + kb * 16384 + kk * 32, 0, 1024, kSw128), id_s, (kb | kk) != 0);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        mma_f8f6f4(d, smem_desc(st + kRcOff + kk * 32, 0, 512, kSw64),
                                   smem_desc(qb + kRcOff + kk * 32, 0, 512, kSw64), id_s, 1);
                    mma_commit(&ms.s_full);
                };
                auto issue_pv = [&](int j) {
                    const int s = j & 1;
                    const uint32_t st = sbase + (s ? OFF_ST1 : OFF_ST0);
                    const uint32_t phi = st + kRcOff, plo = sbase + OFF_PLO;
                    // dims 0..255: B = 128 columns, the hi piece's 64 heads then the lo piece's (MN-major,
                    // 64-byte swizzle atoms; the second atom along N sits at the leading-byte offset)
                    const uint32_t lbo = plo - phi;
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        const uint32_t d = tmem + TM_O + 128u * (uint32_t)ch;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f8f6f4(d, smem_desc(st + ch * 16384 + kk * 4096, 0, 1024, kSw128),
                                       smem_desc(phi + kk * 2048, lbo, 512, kSw64), id_pw, (j | kk) != 0);
                        mma_commit(&ms.kv_blk[s][ch]);  // latent block ch may be refilled
                    }
                    // dims 256..511: the lo piece's passes first, so that the next tile's softmax may
                    // overwrite the lo buffer while the hi passes run
#pragma unroll
                    for (int ch = 2; ch < 4; ++ch)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f8f6f4(tmem + TM_O + 64u * (uint32_t)(ch + 2),
                                       smem_desc(st + ch * 16384 + kk * 4096, 0, 1024, kSw128),
                                       smem_desc(plo + kk * 2048, 0, 512, kSw64), id_pv, (j | kk) != 0);
                    mma_commit(&ms.lo_free);
#pragma unroll
                    for (int ch = 2; ch < 4; ++ch) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_f8f6f4(tmem + TM_O + 64u * (uint32_t)(ch + 2),
                                       smem_desc(st + ch * 16384 + kk * 4096, 0, 1024, kSw128),
                                       smem_desc(phi + kk * 2048, 0, 512, kSw64), id_pv, 1);
                        mma_commit(&ms.kv_blk[s][ch]);
                    }
                    mma_commit(&ms.kv_empty[s]);
                    mma_commit(&ms.pv_done[s]);
                };
                // Issue whichever is ready, the context product first: it releases the row stage for
                // the next load.  Score i needs tile i loaded and the score buffer read by the softmax
                // of tile i-1; PV j needs the weights of tile j.
                int ns = 0, np = 0;
                if (a.qimg && n_tiles > 0 && !mbar_wait(&ms.q_full, 0, &ms.abort_flag, a.err_word)) np = n_tiles;
                const uint64_t t_start = globaltimer_ns();
                uint64_t t_last = t_start;
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
                        // selected rows arrive by cp.async (generic proxy): make them visible to the MMAs
                        if (idx_b) fence_proxy_async_smem();
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
                (void)t_start;
                // all issued MMAs complete before the CTA tears down
                mma_commit(&ms.final_bar);
                mbar_wait(&ms.final_bar, 0, nullptr, a.err_word, 200000000ull);
            }
            __syncwarp();
        } else {
            // ============================ softmax + epilogue ============================
            // Each thread owns one tile row (TMEM lane) and the kHG heads of its softmax group.  The four
            // warps of a group decide and rescale together through named barrier 2 + grp.  A wait that
            // gives up clears `ok`; the thread then skips its remaining waits but still reaches every named
            // barrier of every tile, so the other warps never wait for it.
            constexpr int kV4 = kHG / 4, kLd = kHG / 16;  // float4s / 16-column TMEM loads per head set
            const int q = warp & 3;               // TMEM lane quadrant
            const int grp = (warp - 2) >> 2;      // which kHG of the CTA's 64 heads
            const int h0 = kHG * grp;             // the group's first head (within the CTA)
            const int r = q * 32 + lane;          // row within the tile = TMEM lane
            const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
            const int bar_id = 2 + grp;
            const float w_mul = ms.w_mul;
            constexpr int kP = kHG / 2;  // head pairs (f32x2 lanes)
            uint64_t z2[kP];             // row sums per head pair, relative to the heads' references
#pragma unroll
            for (int j = 0; j < kP; ++j) z2[j] = f2_pack(0.f, 0.f);
            // scale of the row at list position pos, or -1 if that row is masked (past the end, or an
            // index outside [0, T), which is also reported)
            bool bad_index = false;
            auto row_scale = [&](int64_t pos) -> float {
                if (pos >= t1) return -1.f;
                if (!idx_b) return __ldg(a.kv_scale + seq_base + pos);
                const int ri = __ldg(idx_b + pos);
                if (ri < 0 || (int64_t)ri >= a.T) {
                    bad_index = true;
                    return -1.f;
                }
                return __ldg(a.kv_scale + seq_base + ri);
            };
            // butterfly transpose-reduction of kHG values over the warp: at step k each lane keeps the half
            // of its heads selected by lane bit k and combines the other half from lane ^ k; after log2(kHG)
            // steps lane l holds head (l % kHG) over the lanes that differ in the low bits, and the last
            // steps combine the lanes that differ in the high bits
            auto warp_reduce_heads = [&](float (&v)[kHG], bool take_max) -> float {
#pragma unroll
                for (int k = kHG / 2; k >= 1; k >>= 1) {
                    const bool upper = (lane & k) != 0;
#pragma unroll
                    for (int j = 0; j < k; ++j) {
                        const float send = upper ? v[j] : v[j + k];
                        const float keep = upper ? v[j + k] : v[j];
                        const float other = __shfl_xor_sync(0xffffffffu, send, k);
                        v[j] = take_max ? fmaxf(keep, other) : keep + other;
                    }
                }
                float x = v[0];
#pragma unroll
                for (int o = kHG; o < 32; o <<= 1) {
                    const float other = __shfl_xor_sync(0xffffffffu, x, o);
                    x = take_max ? fmaxf(x, other) : x + other;
                }
                return x;
            };
            float sc_next = n_tiles > 0 ? row_scale(t0 + r) : -1.f;
            bool ok = true;
            bool seen = false;  // some valid row has been scored: every head's running max is finite
            int cur = 0;        // which copy of ms.m_run / ms.m_ref is current (uniform across the group)
            for (int i = 0; i < n_tiles; ++i) {
                const int bb = i & 1;
                const int64_t t = t0 + (int64_t)i * kTile + r;
                const float sc_t = sc_next;
                const bool valid = sc_t >= 0.f;
                sc_next = i + 1 < n_tiles ? row_scale(t + kTile) : -1.f;

                if (ok) ok = mbar_wait(&ms.s_full, i & 1, &ms.abort_flag, a.err_word);
                tc_fence_after_sync();
                uint64_t s2[kP];  // S = hi piece + lo piece (one TMEM round trip), head pairs packed
                {
                    uint32_t shi[kLd][16], slo[kLd][16];
                    const uint32_t ta = tmem + lane_addr + TM_S + (uint32_t)h0;
#pragma unroll
                    for (int u = 0; u < kLd; ++u) {
                        tmem_ld_32x32b_x16(ta + 16u * u, shi[u]);
                        tmem_ld_32x32b_x16(ta + 64u + 16u * u, slo[u]);
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < kP; ++j) {
                        const int a0 = 2 * j, a1 = 2 * j + 1;
                        s2[j] = f2_add(f2_pack(__uint_as_float(shi[a0 >> 4][a0 & 15]), __uint_as_float(shi[a1 >> 4][a1 & 15])),
                                       f2_pack(__uint_as_float(slo[a0 >> 4][a0 & 15]), __uint_as_float(slo[a1 >> 4][a1 & 15])));
                    }
                }
                tc_fence_before_sync();
                mbar_arrive(&ms.s_free);

                // d = s - ref with s = S * sm_scale*log2(e)*2^-e_h * s_t (the factor is rounded once, then
                // one fused multiply-add per score); ref is the running max, or 0 before any valid row
                uint64_t d2[kP];
                float dmax = -INFINITY;
                {
                    const float *mref = &ms.m_ref[cur][h0];
                    const uint64_t st2 = f2_pack(sc_t, sc_t);
#pragma unroll
                    for (int j4 = 0; j4 < kV4; ++j4) {
                        const float4 c4 = *reinterpret_cast<const float4 *>(&ms.c_head[h0 + 4 * j4]);
                        const float4 r4 = *reinterpret_cast<const float4 *>(mref + 4 * j4);
                        d2[2 * j4] = f2_fma(s2[2 * j4], f2_mul(f2_pack(c4.x, c4.y), st2), f2_pack(-r4.x, -r4.y));
                        d2[2 * j4 + 1] = f2_fma(s2[2 * j4 + 1], f2_mul(f2_pack(c4.z, c4.w), st2), f2_pack(-r4.z, -r4.w));
                        float a, b, c, e;
                        f2_unpack(d2[2 * j4], a, b);
                        f2_unpack(d2[2 * j4 + 1], c, e);
                        dmax = fmaxf(dmax, fmaxf(fmaxf(a, b), fmaxf(c, e)));
                    }
                }
                if (!valid) {
#pragma unroll
                    for (int j = 0; j < kP; ++j) d2[j] = f2_pack(-INFINITY, -INFINITY);
                    dmax = -INFINITY;
                }
                // lazy rescale: the group takes the slow path when some score exceeds its head's running
                // max by more than kTau, or while no valid row has been seen
                const bool slow = bar_red_or(bar_id, 128, dmax > kTau || !seen);
                bool any_alpha = false;
                if (slow) {
                    // per-head maxima over this warp's 32 rows (one warp reduction per head), then over the
                    // group's four lane quadrants through shared memory
                    float hm[kHG];
#pragma unroll
                    for (int j = 0; j < kP; ++j) {
                        float a, b;
                        f2_unpack(d2[j], a, b);
                        hm[2 * j] = warp_redux_max(a);
                        hm[2 * j + 1] = warp_redux_max(b);
                    }
                    if (lane == 0) {
#pragma unroll
                        for (int j4 = 0; j4 < kV4; ++j4)
                            *reinterpret_cast<float4 *>(&ms.red[q][h0 + 4 * j4]) =
                                make_float4(hm[4 * j4], hm[4 * j4 + 1], hm[4 * j4 + 2], hm[4 * j4 + 3]);
                    }
                    const int hl = lane & (kHG - 1);
                    const int hj = h0 + hl;
                    named_sync(bar_id, 128);
                    const float ref_o = ms.m_ref[cur][hj], mo = ms.m_run[cur][hj];
                    const float tmax = fmaxf(fmaxf(ms.red[0][hj], ms.red[1][hj]), fmaxf(ms.red[2][hj], ms.red[3][hj])) + ref_o;
                    const float mn = mo == -INFINITY ? tmax : (tmax > mo + kTau ? tmax : mo);
                    const float al = (mo == -INFINITY || mn == mo) ? 1.f : ex2_approx(mo - mn);
                    const float ref_n = mn == -INFINITY ? 0.f : mn;
                    // the four quadrant warps write the same values
                    if (lane < kHG) {
                        ms.m_run[cur ^ 1][hj] = mn;
                        ms.m_ref[cur ^ 1][hj] = ref_n;
                        ms.ph.tile.alpha[grp][hl] = al;
                        ms.ph.tile.delta[grp][hl] = ref_o - ref_n;
                    }
                    seen = __shfl_sync(0xffffffffu, mn, 0) != -INFINITY;  // the same for every head
                    any_alpha = __any_sync(0xffffffffu, al != 1.f);
                    __syncwarp();
#pragma unroll
                    for (int j4 = 0; j4 < kV4; ++j4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(&ms.ph.tile.alpha[grp][4 * j4]);
                        const float4 e4 = *reinterpret_cast<const float4 *>(&ms.ph.tile.delta[grp][4 * j4]);
                        d2[2 * j4] = f2_add(d2[2 * j4], f2_pack(e4.x, e4.y));
                        d2[2 * j4 + 1] = f2_add(d2[2 * j4 + 1], f2_pack(e4.z, e4.w));
                        z2[2 * j4] = f2_mul(z2[2 * j4], f2_pack(a4.x, a4.y));
                        z2[2 * j4 + 1] = f2_mul(z2[2 * j4 + 1], f2_pack(a4.z, a4.w));
                    }
                    cur ^= 1;
                }
                // weights: p = 2^d (row sum z), w = p * s_t * kWScale / s_ref, split e4m3 hi + lo
                const float g = valid ? sc_t * w_mul : 0.f;
                const uint64_t g2 = f2_pack(g, g);
                uint32_t whi[kV4], wlo[kV4];
#pragma unroll
                for (int j4 = 0; j4 < kV4; ++j4) {
                    float d0, d1, e0, e1;
                    f2_unpack(d2[2 * j4], d0, d1);
                    f2_unpack(d2[2 * j4 + 1], e0, e1);
                    const uint64_t p01 = f2_pack(ex2_approx(d0), ex2_approx(d1));
                    const uint64_t p23 = f2_pack(ex2_approx(e0), ex2_approx(e1));
                    z2[2 * j4] = f2_add(z2[2 * j4], p01);
                    z2[2 * j4 + 1] = f2_add(z2[2 * j4 + 1], p23);
                    float w0, w1, w2, w3;
                    f2_unpack(f2_mul(p01, g2), w0, w1);
                    f2_unpack(f2_mul(p23, g2), w2, w3);
                    uint32_t h01, l01, h23, l23;
                    split_pair_h(w0, w1, h01, l01);
                    split_pair_h(w2, w3, h23, l23);
                    whi[j4] = h01 | (h23 << 16);
                    wlo[j4] = l01 | (l23 << 16);
                }
                uint8_t *phi = smem + (bb ? OFF_ST1 : OFF_ST0) + kRcOff;  // the rope block, read by the score already
#pragma unroll
                for (int u = 0; u < kV4 / 4; ++u)
                    *reinterpret_cast<uint4 *>(phi + sw64_offset(r, h0 + 16 * u)) =
                        make_uint4(whi[4 * u], whi[4 * u + 1], whi[4 * u + 2], whi[4 * u + 3]);
                if (i >= 1) {
                    // the previous context product must have read its weights' lo buffer before it is
                    // reused, and be done before its accumulators are rescaled.  lo_free is waited on every
                    // tile; pv_done only on a rescale, so it has one barrier per tile parity: the phase
                    // before the awaited one (tile i-3) is complete, which keeps the parity unambiguous.
                    // lo_free also covers every MMA issued before the lo passes (the dims 0..255 passes):
                    // pieces 0..3 are rescaled right away, pieces 4, 5 once the hi passes are done too.
                    if (ok) ok = mbar_wait(&ms.lo_free, (i - 1) & 1, &ms.abort_flag, a.err_word);
                    if (any_alpha) {
                        // rescale this group's columns of the six context accumulators, 32 columns per
                        // TMEM round trip
                        constexpr int kPerTrip = 32 / kHG;  // accumulators per round trip
                        static_assert(4 % kPerTrip == 0, "pieces 0..3 and 4..5 in whole round trips");
                        auto rescale_trip = [&](int c0) {
                            uint32_t o[kPerTrip][kHG];
#pragma unroll
                            for (int c = 0; c < kPerTrip; ++c)
#pragma unroll
                                for (int u = 0; u < kLd; ++u)
                                    tmem_ld_32x32b_x16(tmem + lane_addr + TM_O + 64u * (c0 + c) + (uint32_t)h0 + 16u * u,
                                                       *reinterpret_cast<uint32_t(*)[16]>(&o[c][16 * u]));
                            tmem_wait_ld();
                            const float *al = ms.ph.tile.alpha[grp];
#pragma unroll
                            for (int j4 = 0; j4 < kV4; ++j4) {
                                const float4 a4 = *reinterpret_cast<const float4 *>(al + 4 * j4);
                                const uint64_t a01 = f2_pack(a4.x, a4.y), a23 = f2_pack(a4.z, a4.w);
#pragma unroll
                                for (int c = 0; c < kPerTrip; ++c) {
                                    uint32_t *oc = &o[c][4 * j4];
                                    float x0, x1, x2, x3;
                                    f2_unpack(f2_mul(f2_pack(__uint_as_float(oc[0]), __uint_as_float(oc[1])), a01), x0, x1);
                                    f2_unpack(f2_mul(f2_pack(__uint_as_float(oc[2]), __uint_as_float(oc[3])), a23), x2, x3);
                                    oc[0] = __float_as_uint(x0);
                                    oc[1] = __float_as_uint(x1);
                                    oc[2] = __float_as_uint(x2);
                                    oc[3] = __float_as_uint(x3);
                                }
                            }
#pragma unroll
                            for (int c = 0; c < kPerTrip; ++c)
#pragma unroll
                                for (int u = 0; u < kLd; ++u)
                                    tmem_st_32x32b_x16(tmem + lane_addr + TM_O + 64u * (c0 + c) + (uint32_t)h0 + 16u * u,
                                                       *reinterpret_cast<const uint32_t(*)[16]>(&o[c][16 * u]));
                        };
                        tc_fence_after_sync();
#pragma unroll 1
                        for (int c0 = 0; c0 < 4; c0 += kPerTrip) rescale_trip(c0);
                        if (ok) ok = mbar_wait(&ms.pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, &ms.abort_flag, a.err_word);
                        tc_fence_after_sync();
#pragma unroll 1
                        for (int c0 = 4; c0 < kOPieces; c0 += kPerTrip) rescale_trip(c0);
                        tmem_wait_st();
                    }
                }
                uint8_t *plo = smem + OFF_PLO;
#pragma unroll
                for (int u = 0; u < kV4 / 4; ++u)
                    *reinterpret_cast<uint4 *>(plo + sw64_offset(r, h0 + 16 * u)) =
                        make_uint4(wlo[4 * u], wlo[4 * u + 1], wlo[4 * u + 2], wlo[4 * u + 3]);
                fence_proxy_async_smem();
                tc_fence_before_sync();
                mbar_arrive(&ms.p_full);
            }

            // ================================ epilogue ================================
            grid_launch_dependents();
            if (grp == 0 && __any_sync(0xffffffffu, bad_index) && lane == 0 && a.err_word)
                atomicOr(a.err_word, (int)KV8_ERR_INDEX);
            if (ok && n_tiles > 0)
                ok = mbar_wait(&ms.pv_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1, &ms.abort_flag, a.err_word);
            tc_fence_after_sync();
            // row sums per head: over the warp's 32 rows (the butterfly), then over the 4 quadrants
            {
                float z[kHG];
#pragma unroll
                for (int j = 0; j < kP; ++j) f2_unpack(z2[j], z[2 * j], z[2 * j + 1]);
                const float zw = warp_reduce_heads(z, false);
                if (lane < kHG) ms.red[q][h0 + lane] = zw;
            }
            named_sync(bar_id, 128);
            if (q == 0 && lane < kHG) {
                const int h = h0 + lane;
                const float zz = ms.red[0][h] + ms.red[1][h] + ms.red[2][h] + ms.red[3][h];
                ms.ph.fin.zsum[h] = zz;
                ms.ph.fin.zinv[h] = zz > 0.f ? ms.out_mul / zz : 0.f;
            }
            named_sync(bar_id, 128);
            if (ok) {
                const float out_mul = ms.out_mul;
                PartialView pv(a.ws, a.B, a.P, a.H);
                // this thread's row (dims 128c + r) of the accumulators (dims 0..255: the hi and lo
                // pieces' accumulators, summed); partial sets (relative to the running max) or the
                // normalised output
                float *const dst = a.ws ? pv.cl + ((int64_t)b * a.P + part) * a.H * kKL : a.out + (int64_t)b * a.H * kKL;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    // chunk c: pieces 2c and 2c+1 for dims 0..255, piece c+2 for the rest
                    uint32_t o[kHG];
                    if (n_tiles > 0) {
                        if (c < 2) {
                            uint32_t e[kHG];
#pragma unroll
                            for (int u = 0; u < kLd; ++u) {
                                tmem_ld_32x32b_x16(tmem + lane_addr + TM_O + 128u * c + (uint32_t)h0 + 16u * u,
                                                   *reinterpret_cast<uint32_t(*)[16]>(&o[16 * u]));
                                tmem_ld_32x32b_x16(tmem + lane_addr + TM_O + 128u * c + 64u + (uint32_t)h0 + 16u * u,
                                                   *reinterpret_cast<uint32_t(*)[16]>(&e[16 * u]));
                            }
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < kHG; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) + __uint_as_float(e[j]));
                        } else {
#pragma unroll
                            for (int u = 0; u < kLd; ++u)
                                tmem_ld_32x32b_x16(tmem + lane_addr + TM_O + 64u * (c + 2) + (uint32_t)h0 + 16u * u,
                                                   *reinterpret_cast<uint32_t(*)[16]>(&o[16 * u]));
                            tmem_wait_ld();
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < kHG; ++j) o[j] = 0u;
                    }
                    float *const col = dst + 128 * c + r;
#pragma unroll
                    for (int j = 0; j < kHG; ++j) {
                        const int hl = h0 + j;  // head within the CTA
                        const int hg = half * kHeadsPerCta + hl;
                        if (hg < a.H) col[(int64_t)hg * kKL] = __uint_as_float(o[j]) * (a.ws ? out_mul : ms.ph.fin.zinv[hl]);
                    }
                }
                if (a.ws && q == 0 && lane < kHG) {
                    const int hg = half * kHeadsPerCta + h0 + lane;
                    if (hg < a.H) {
                        const int64_t pidx = ((int64_t)b * a.P + part) * a.H + hg;
                        pv.m[pidx] = n_tiles > 0 ? ms.m_run[cur][h0 + lane] : -INFINITY;  // -inf: no valid row
                        pv.z[pidx] = ms.ph.fin.zsum[h0 + lane];
                    }
                }
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// Query prep, run once before the partial kernel (decode and selection).  Block b * n_heads_pad/8 + g
// splits heads 8g..8g+7 of item b (each scaled by 2^e_h so that max|q| * 2^e_h lies in [128, 256)) into
// e4m3 hi + lo rows of that item's head-group image and writes their score factors
// sm_scale*log2(e)*2^-e_h (0 for a padding head); for selected rows, block B * n_heads_pad/8 + b * P + p
// takes the largest scale among the rows that partition p of item b attends (dense rows: the partial
// kernel takes it itself).
struct PrepArgs {
    const __nv_bfloat16 *q_lat, *q_rope;
    int B, H, n_heads_pad, P;
    float sm_scale_log2;
    const float *kv_scale;
    int64_t T;
    const int32_t *idx;  // selection lists [B][NS], or null (rows 0..T-1 of one item)
    int NS;
    int64_t seq_stride_rows;
    const int32_t *lens; // batched dense decode: rows per item, or null
    uint8_t *img;        // [B][n_half][kImg]
    float *c_head;       // [B][n_heads_pad]
    float *smax;         // [B][P]
};

constexpr int kPrepHeads = 8;                   // heads per query-prep block
constexpr int kPrepBlock = kPrepHeads * 36;     // one thread per (head, 16-element chunk)

__global__ void __launch_bounds__(kPrepBlock) tc_prep_kernel(PrepArgs a) {
    // launched as a programmatic dependent of whatever came before on the stream: nothing is read until
    // that grid has completed; then the partial kernel may start its row loads while this runs
    grid_dependency_wait();
    grid_launch_dependents();
    __shared__ float red[kPrepBlock / 32];
    __shared__ int qmax_bits[kPrepHeads];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, bid = blockIdx.x;
    const int n_groups = a.n_heads_pad / kPrepHeads;
    if (bid < a.B * n_groups) {
        const int b = bid / n_groups, g = bid - b * n_groups;
        const int hl = tid / 36, ch = tid - hl * 36, h = g * kPrepHeads + hl;
        const int half = h / kHeadsPerCta, row = h - half * kHeadsPerCta;
        if (tid < kPrepHeads) qmax_bits[tid] = 0;
        __syncthreads();
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (h < a.H) {
            const int64_t qh = (int64_t)b * a.H + h;
            const __nv_bfloat16 *src = ch < 32 ? a.q_lat + qh * kKL + ch * 16 : a.q_rope + qh * kKR + (ch - 32) * 16;
            const uint4 u0 = __ldg(reinterpret_cast<const uint4 *>(src)), u1 = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
            w[0] = u0.x; w[1] = u0.y; w[2] = u0.z; w[3] = u0.w;
            w[4] = u1.x; w[5] = u1.y; w[6] = u1.z; w[7] = u1.w;
            float mx = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
                mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
            atomicMax(&qmax_bits[hl], __float_as_int(mx));  // non-negative floats order like ints
        }
        __syncthreads();
        const float mx = __int_as_float(qmax_bits[hl]);
        int E = 0;
        if (mx > 0.f) frexpf(mx, &E);
        const int sh = mx > 0.f ? 8 - E : 0;  // values are scaled, not a 2^sh factor: it may overflow
        uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
            uint32_t ph, pl;
            split_pair(ldexpf(f.x, sh), ldexpf(f.y, sh), ph, pl);
            hi[e >> 1] |= ph << ((e & 1) * 16);
            lo[e >> 1] |= pl << ((e & 1) * 16);
        }
        uint8_t *dst = a.img + ((size_t)b * (a.n_heads_pad / kHeadsPerCta) + half) * kImg;
        uint32_t off_hi, off_lo;
        if (ch < 32) {
            const uint32_t kb = ch >> 3, byte = (ch & 7) * 16;
            off_hi = kb * 16384 + sw128_offset(row, byte);
            off_lo = kb * 16384 + sw128_offset(row + 64, byte);
        } else {
            const uint32_t byte = (ch - 32) * 16;
            off_hi = kRcOff + sw64_offset(row, byte);
            off_lo = kRcOff + sw64_offset(row + 64, byte);
        }
        *reinterpret_cast<uint4 *>(dst + off_hi) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(dst + off_lo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if (ch == 0)
            a.c_head[(int64_t)b * a.n_heads_pad + h] =
                h < a.H ? (mx > 0.f ? ldexpf(a.sm_scale_log2, E - 8) : a.sm_scale_log2) : 0.f;
    } else {
        const int bp = bid - a.B * n_groups, b = bp / a.P, p = bp - b * a.P;
        const int64_t n_list = a.idx ? (int64_t)a.NS : a.lens ? min((int64_t)max(__ldg(a.lens + b), 0), a.T) : a.T;
        const int64_t t0 = n_list * p / a.P, t1 = n_list * (p + 1) / a.P;
        const int32_t *idx_b = a.idx ? a.idx + (int64_t)b * a.NS : nullptr;
        const float *sc_b = a.kv_scale + (int64_t)b * a.seq_stride_rows;
        float mx = 0.f;
        for (int64_t t = t0 + tid; t < t1; t += 8 * kPrepBlock) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t tu = t + (int64_t)u * kPrepBlock;
                int64_t ri = tu < t1 ? (idx_b ? (int64_t)__ldg(idx_b + tu) : tu) : -1;
                v[u] = (ri >= 0 && ri < a.T) ? __ldg(sc_b + ri) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) mx = fmaxf(mx, fabsf(v[u]));
        }
        mx = warp_max(mx);
        if (lane == 0) red[warp] = mx;
        __syncthreads();
        if (tid == 0) {
            float m = 0.f;
            for (int k = 0; k < kPrepBlock / 32; ++k) m = fmaxf(m, red[k]);
            a.smax[bp] = m;
        }
    }
}

}  // namespace

// The driver's tensor-map encoder, looked up once (null if the driver does not provide it).
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

// Launch the tensor-core kernel.  The grid covers B items x P partitions x the head halves.  Dense
// rows are loaded as 128-row tiles through tensor maps over all items' caches; selected rows are
// copied by the kernel's producer warp.  Returns cudaErrorNotSupported if the tensor-map encoder is
// unavailable.
cudaError_t launch_attn_tc(const AttnArgs &x, cudaStream_t st) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const bool sel = x.idx != nullptr;
    // the tensor maps cover every item's cache (items seq_stride_rows apart; 0 when they share one)
    const int64_t rows = (int64_t)(x.B - 1) * x.seq_stride_rows + x.T;
    if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;  // tensor-map row coordinates are 32-bit
    CUtensorMap m_lc, m_rc;
    const cuuint64_t dims[2] = {(cuuint64_t)kRow, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kRow};
    const cuuint32_t box_h = sel ? 1u : (cuuint32_t)kTile;  // selection does not use the maps
    const cuuint32_t box_lc[2] = {128, box_h}, box_rc[2] = {64, box_h}, es[2] = {1, 1};
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
    a.kv8 = x.kv8;
    a.kv_scale = x.kv_scale;
    a.T = x.T;
    a.pos0 = x.pos0;
    a.lens = x.lens;
    a.idx = x.idx;
    a.NS = x.NS;
    a.seq_stride_rows = x.seq_stride_rows;
    a.sm_scale_log2 = x.sm_scale_log2;
    a.ws = x.ws;
    a.out = x.out;
    a.err_word = x.err_word;
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const int64_t grid = (int64_t)a.B * a.P * a.n_half;
    if (x.tc_scratch) {
        // decode / selection: prepare the queries once, then start the partial kernel as a
        // programmatic dependent
        const int n_heads_pad = a.n_half * kHeadsPerCta;
        PrepArgs pa{};
        pa.q_lat = a.q_lat;
        pa.q_rope = a.q_rope;
        pa.B = a.B;
        pa.H = a.H;
        pa.n_heads_pad = n_heads_pad;
        pa.P = a.P;
        pa.sm_scale_log2 = a.sm_scale_log2;
        pa.kv_scale = a.kv_scale;
        pa.T = a.T;
        pa.idx = a.idx;
        pa.NS = a.NS;
        pa.seq_stride_rows = a.seq_stride_rows;
        pa.lens = a.lens;
        pa.img = static_cast<uint8_t *>(x.tc_scratch);
        pa.c_head = reinterpret_cast<float *>(pa.img + (size_t)a.B * 2 * kImg);
        pa.smax = pa.c_head + (size_t)a.B * 2 * kHeadsPerCta;
        a.qimg = pa.img;
        a.c_head = pa.c_head;
        a.smax = pa.smax;
        cudaLaunchConfig_t pcfg = {};
        // partition blocks (largest row scale per partition) only for selected rows; dense rows take the
        // maximum inside the partial kernel
        pcfg.gridDim = dim3((unsigned)((int64_t)a.B * (n_heads_pad / kPrepHeads + (sel ? a.P : 0))));
        pcfg.blockDim = dim3(kPrepBlock);
        pcfg.stream = st;
        cudaLaunchAttribute pattr[1];
        pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pattr[0].val.programmaticStreamSerializationAllowed = 1;
        pcfg.attrs = pattr;
        pcfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&pcfg, tc_prep_kernel, pa)) != cudaSuccess) return e;
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, attn_tc_kernel, m_lc, m_rc, a);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if (sel) return cudaErrorInvalidValue;  // selection always takes the prepared-query path
    attn_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, st>>>(m_lc, m_rc, a);
    return cudaGetLastError();
}

size_t tc_scratch_bytes(int B, int P) {
    // query images (2 head groups per item), per-head factors, per-partition row-scale maxima
    return (size_t)B * (2 * (size_t)kImg + 2 * kHeadsPerCta * sizeof(float)) +
           (((size_t)B * P * sizeof(float) + 255) & ~(size_t)255);
}

}  // namespace kv8
