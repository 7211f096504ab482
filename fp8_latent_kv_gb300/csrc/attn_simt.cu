// attn_simt.cu -- absorbed MLA attention over e4m3 cache rows on the CUDA cores (sm_103a).
//
// Page "KV8 long-context CUDA: fp8 device shadow, split-T kernels, DSA-aware gather":
//   first commit message  -- the latent row serves as key and value; the row scale is hoisted out of the
//                            dot (score = sm_scale * s_t * q.e4m3(row)); context = softmax-weighted
//                            sum of s_t * e4m3(Lc_t).
//   second commit message -- split-T: partial online-softmax blocks (cl[K], m, z) plus a log-sum-exp
//                            merge kernel; DSA gather: attend the selected rows of the device cache
//                            by absolute index; batch/prefill path tiled over the rows.
//
// This is the general kernel: f32 or bf16 queries, any H in [1, 128], dense / selected / causal row
// lists.  A block owns 32 heads and one partition of the row list; it streams 64-row tiles of the
// cache through shared memory (16-byte loads), computes the 64x32 score tile, updates the online
// softmax per head and accumulates the 32x512 context in registers (2 latent columns per thread).
#include "internal.h"
#include "sm100.cuh"

#include <cudaTypedefs.h>

#include <math.h>

namespace kv8 {
namespace {

constexpr int kHB = 32;        // heads per block
constexpr int kTR = 64;        // rows per tile
constexpr int kThreads = 256;  // 8 warps
constexpr int kTileStride = kRow + 4;  // 580 bytes = 145 words: odd, so row-per-lane reads are conflict-free
constexpr int kSStride = kHB + 1;

struct Smem {
    float q[kHB][kRow];               // queries of this block's heads (f32)
    uint8_t tile[kTR][kTileStride];   // current cache tile
    float s[kTR][kSStride];           // scores (log2 domain)
    float p[kTR][kHB];                // weights p * s_t, row-major for broadcast reads
    float rscale[kTR];                // row scale, 0 for an invalid row
    int rvalid[kTR];
    const uint8_t *rowptr[kTR];
    float m_run[kHB], z_run[kHB], corr[kHB];
};

__device__ __forceinline__ float load_q(const void *base, int64_t i, int bf16) {
    if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[i]);
    return reinterpret_cast<const float *>(base)[i];
}

__global__ void __launch_bounds__(kThreads, 1) attn_simt_kernel(AttnArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int part = blockIdx.x, hb0 = blockIdx.y * kHB, b = blockIdx.z;
    const int nh = min(kHB, a.H - hb0);

    // ---- row list of this batch item and this partition
    int64_t n_list;
    if (a.idx) n_list = a.NS;
    else if (a.pos0 >= 0) n_list = (a.pos0 + b + 1 < a.T) ? a.pos0 + b + 1 : a.T;
    else if (a.lens) n_list = min((int64_t)max(__ldg(a.lens + b), 0), a.T);
    else n_list = a.T;
    const int64_t j0 = n_list * part / a.P, j1 = n_list * (part + 1) / a.P;
    const uint8_t *kv_b = a.kv8 + (int64_t)b * a.seq_stride_rows * kRow;
    const float *sc_b = a.kv_scale + (int64_t)b * a.seq_stride_rows;
    const int32_t *idx_b = a.idx ? a.idx + (int64_t)b * a.NS : nullptr;

    // ---- queries -> shared (f32, exact)
    for (int i = tid; i < kHB * kRow; i += kThreads) {
        const int h = i / kRow, k = i - h * kRow;
        float v = 0.f;
        if (h < nh) {
            const int64_t qh = (int64_t)b * a.H + hb0 + h;
            v = (k < kKL) ? load_q(a.q_lat, qh * kKL + k, a.q_bf16) : load_q(a.q_rope, qh * kKR + (k - kKL), a.q_bf16);
        }
        sm.q[h][k] = v;
    }
    if (tid < kHB) {
        sm.m_run[tid] = -INFINITY;
        sm.z_run[tid] = 0.f;
    }

    float acc[kHB][2];
#pragma unroll
    for (int h = 0; h < kHB; ++h) acc[h][0] = acc[h][1] = 0.f;
    bool bad_index = false;

    for (int64_t jt = j0; jt < j1; jt += kTR) {
        __syncthreads();  // previous tile fully consumed
        // ---- row pointers and scales for this tile
        if (tid < kTR) {
            const int64_t j = jt + tid;
            int valid = 0;
            int64_t t = 0;
            if (j < j1) {
                t = idx_b ? (int64_t)idx_b[j] : j;
                if (t >= 0 && t < a.T) valid = 1;
                else bad_index = true;
            }
            sm.rvalid[tid] = valid;
            sm.rowptr[tid] = valid ? kv_b + t * kRow : nullptr;
            sm.rscale[tid] = valid ? sc_b[t] : 0.f;
        }
        __syncthreads();
        // ---- tile load: 64 rows x 36 uint4
        for (int c = tid; c < kTR * (kRow / 16); c += kThreads) {
            const int r = c / (kRow / 16), col = c - r * (kRow / 16);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            const uint8_t *rp = sm.rowptr[r];
            if (rp) v = __ldg(reinterpret_cast<const uint4 *>(rp) + col);
            uint32_t *dst = reinterpret_cast<uint32_t *>(&sm.tile[r][col * 16]);
            dst[0] = v.x;
            dst[1] = v.y;
            dst[2] = v.z;
            dst[3] = v.w;
        }
        __syncthreads();
        // ---- scores: warp w -> heads (w&3)*8..+7, rows (w>>2)*32 + lane
        {
            const int g = warp & 3, r = (warp >> 2) * 32 + lane;
            float s8[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) s8[j] = 0.f;
            const uint32_t *rw = reinterpret_cast<const uint32_t *>(&sm.tile[r][0]);
#pragma unroll 4
            for (int k4 = 0; k4 < kRow / 4; ++k4) {
                float e0, e1, e2, e3;
                e4m3x4_to_f32(rw[k4], e0, e1, e2, e3);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(&sm.q[g * 8 + j][k4 * 4]);
                    s8[j] = fmaf(q4.x, e0, s8[j]);
                    s8[j] = fmaf(q4.y, e1, s8[j]);
                    s8[j] = fmaf(q4.z, e2, s8[j]);
                    s8[j] = fmaf(q4.w, e3, s8[j]);
                }
            }
            const float f = sm.rscale[r] * a.sm_scale_log2;
            const bool ok = sm.rvalid[r] != 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) sm.s[r][g * 8 + j] = ok ? s8[j] * f : -INFINITY;
        }
        __syncthreads();
        // ---- online softmax: thread -> head tid/8, rows (tid%8)*8..+7
        {
            const int h = tid >> 3, sub = tid & 7;
            float mloc = -INFINITY;
#pragma unroll
            for (int i = 0; i < 8; ++i) mloc = fmaxf(mloc, sm.s[sub * 8 + i][h]);
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
            const float m_old = sm.m_run[h];
            const float m_new = fmaxf(m_old, mloc);
            float corr = 1.f, zloc = 0.f;
            if (m_new == -INFINITY) {
#pragma unroll
                for (int i = 0; i < 8; ++i) sm.p[sub * 8 + i][h] = 0.f;
            } else {
                corr = exp2f(m_old - m_new);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = sub * 8 + i;
                    const float pr = exp2f(sm.s[r][h] - m_new);
                    zloc += pr;
                    sm.p[r][h] = pr * sm.rscale[r];
                }
            }
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) zloc += __shfl_xor_sync(0xffffffffu, zloc, o);
            __syncwarp();
            if (sub == 0) {
                sm.m_run[h] = m_new;
                sm.z_run[h] = sm.z_run[h] * corr + zloc;
                sm.corr[h] = corr;
            }
        }
        __syncthreads();
        // ---- context: thread -> latent columns 2*tid, 2*tid+1
        {
#pragma unroll
            for (int h = 0; h < kHB; ++h) {
                const float c = sm.corr[h];
                acc[h][0] *= c;
                acc[h][1] *= c;
            }
            const int nr = (j1 - jt) < kTR ? (int)(j1 - jt) : kTR;
            for (int r = 0; r < nr; ++r) {
                float v0, v1;
                e4m3x2_to_f32(*reinterpret_cast<const uint16_t *>(&sm.tile[r][2 * tid]), v0, v1);
#pragma unroll
                for (int h4 = 0; h4 < kHB / 4; ++h4) {
                    const float4 w = *reinterpret_cast<const float4 *>(&sm.p[r][h4 * 4]);
                    acc[h4 * 4 + 0][0] = fmaf(w.x, v0, acc[h4 * 4 + 0][0]);
                    acc[h4 * 4 + 0][1] = fmaf(w.x, v1, acc[h4 * 4 + 0][1]);
                    acc[h4 * 4 + 1][0] = fmaf(w.y, v0, acc[h4 * 4 + 1][0]);
                    acc[h4 * 4 + 1][1] = fmaf(w.y, v1, acc[h4 * 4 + 1][1]);
                    acc[h4 * 4 + 2][0] = fmaf(w.z, v0, acc[h4 * 4 + 2][0]);
                    acc[h4 * 4 + 2][1] = fmaf(w.z, v1, acc[h4 * 4 + 2][1]);
                    acc[h4 * 4 + 3][0] = fmaf(w.w, v0, acc[h4 * 4 + 3][0]);
                    acc[h4 * 4 + 3][1] = fmaf(w.w, v1, acc[h4 * 4 + 3][1]);
                }
            }
        }
    }
    if (bad_index && a.err_word) atomicOr(a.err_word, (int)KV8_ERR_INDEX);
    __syncthreads();

    // ---- write the partial set, or the normalised output
    if (a.ws) {
        PartialView pv(a.ws, a.B, a.P, a.H);
        const int64_t base = ((int64_t)b * a.P + part) * a.H + hb0;
        for (int h = 0; h < nh; ++h)
            reinterpret_cast<float2 *>(pv.cl + (base + h) * kKL)[tid] = make_float2(acc[h][0], acc[h][1]);
        if (tid < nh) {
            pv.m[base + tid] = sm.m_run[tid];
            pv.z[base + tid] = sm.z_run[tid];
        }
    } else {
        for (int h = 0; h < nh; ++h) {
            const float z = sm.z_run[h];
            const float inv = z > 0.f ? 1.f / z : 0.f;
            reinterpret_cast<float2 *>(a.out + ((int64_t)b * a.H + hb0 + h) * kKL)[tid] =
                make_float2(acc[h][0] * inv, acc[h][1] * inv);
        }
    }
}

// Log-sum-exp merge: block (h, quarter, b) -- 128 threads, one latent column each.
//
// P <= kMergeTma: one 3-D TMA box brings the block's 128 columns of all P partitions' cl rows of head h
// into shared memory (a tensor map over cl viewed as [B*P][H][512]), while warp 0 loads every maximum and
// row sum at once (up to four per lane, one round trip) and turns them into weights 2^(m_p - M); every
// thread then sums its column.  Per-thread loads of the columns (the kernels below) keep far more lines
// in flight per SM than the load units track, so they wait on memory-level parallelism, not bandwidth.
constexpr int kMergeTma = 128;
// byte offset of the merge block's mbarrier: after the P x 128 columns and the P + 1 weights
__host__ __device__ constexpr size_t merge_tma_bar_offset(int P) {
    return ((size_t)P * 129 * sizeof(float) + sizeof(float) + 15) & ~(size_t)15;
}

__global__ void __launch_bounds__(128) lse_merge_tma_kernel(const __grid_constant__ CUtensorMap map,
                                                            const float *__restrict__ ws, int B, int P, int H,
                                                            float *__restrict__ out) {
    extern __shared__ __align__(1024) uint8_t msm[];
    float *cs = reinterpret_cast<float *>(msm);  // [P][128]
    float *wsh = cs + (size_t)P * 128;           // [P] weights, then Z
    uint64_t *full = reinterpret_cast<uint64_t *>(msm + merge_tma_bar_offset(P));
    const int h = blockIdx.x, quarter = blockIdx.y, b = blockIdx.z, tid = threadIdx.x, lane = tid & 31;
    PartialView pv(const_cast<float *>(ws), B, P, H);
    const int64_t base = (int64_t)b * P * H + h;
    float *o = out + ((int64_t)b * H + h) * kKL + quarter * 128 + tid;
    if ((sm100::smem_u32(msm) & 127u) != 0) {  // a tensor copy needs a 128-byte aligned destination
        *o = NAN;
        return;
    }
    if (tid == 0) {
        sm100::prefetch_tensormap(&map);
        sm100::mbar_init(full, 1);
        sm100::fence_barrier_init();
    }
    __syncthreads();
    // launched as a programmatic dependent of the partial kernel: wait until its partials are written
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) {
        sm100::mbar_arrive_expect_tx(full, (uint32_t)P * 512u);
        sm100::tma_load_3d(cs, &map, quarter * 128, h, b * P, full);
    }
    if (tid < 32) {
        float mv[kMergeTma / 32], zv[kMergeTma / 32];
#pragma unroll
        for (int k = 0; k < kMergeTma / 32; ++k) {
            const int p = lane + 32 * k;
            mv[k] = p < P ? pv.m[base + (int64_t)p * H] : -INFINITY;
            zv[k] = p < P ? pv.z[base + (int64_t)p * H] : 0.f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMergeTma / 32; ++k) M = fmaxf(M, mv[k]);
        M = warp_max(M);
        float Z = 0.f;
#pragma unroll
        for (int k = 0; k < kMergeTma / 32; ++k) {
            const int p = lane + 32 * k;
            const float w = (mv[k] == -INFINITY || M == -INFINITY) ? 0.f : exp2f(mv[k] - M);
            if (p < P) wsh[p] = w;
            Z = fmaf(w, zv[k], Z);
        }
        Z = warp_sum(Z);
        if (tid == 0) wsh[P] = Z;
    }
    __syncthreads();
    // the copy lands long before the limit; if it did not, the block reports NaN and still waits for it
    // before it ends (its destination is this block's shared memory)
    const bool ok = sm100::mbar_wait(full, 0, nullptr, nullptr, 200000000ull);
    if (!ok) (void)sm100::mbar_wait(full, 0, nullptr, nullptr, 200000000ull);
    float acc0 = 0.f, acc1 = 0.f;
    for (int p = 0; p < P; ++p) {
        const float w = wsh[p];
        // a partition with weight 0 may hold anything (it attended no row): do not touch its values
        if (w != 0.f) {
            if (p & 1) acc1 = fmaf(w, cs[p * 128 + tid], acc1);
            else acc0 = fmaf(w, cs[p * 128 + tid], acc0);
        }
    }
    const float Z = wsh[P];
    *o = !ok ? NAN : Z > 0.f ? (acc0 + acc1) / Z : 0.f;
}

// Without a tensor-map encoder, or for P > kMergeTma.  Small P (<= kMergeFast): every load the block
// needs is issued before any result is used -- each thread's P partial columns, and each warp's own copy
// of the P maxima and row sums -- so the partials' latency is paid about once.  Each warp turns the
// maxima into weights 2^(m_p - M) itself (lane p % 32 holds partition p's) and every thread sums its
// column.
constexpr int kMergeFast = 128;
constexpr int kMergeMaxP = 1024;  // larger P: weights kept in shared memory, loops over slices

template <int NP>
__device__ __forceinline__ void merge_small(const PartialView &pv, int64_t base, int P, int H, int d, float *out) {
    const int lane = threadIdx.x & 31;
    const float *cl = pv.cl + base * kKL + d;
    const int64_t pstride = (int64_t)H * kKL;
    float c[NP];
#pragma unroll
    for (int u = 0; u < NP; ++u) c[u] = u < P ? cl[(int64_t)u * pstride] : 0.f;
    constexpr int K = (NP + 31) / 32;
    float mv[K], zv[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int p = lane + 32 * k;
        mv[k] = p < P ? pv.m[base + (int64_t)p * H] : -INFINITY;
        zv[k] = p < P ? pv.z[base + (int64_t)p * H] : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < K; ++k) M = fmaxf(M, mv[k]);
    M = warp_max(M);
    float wv[K], Z = 0.f;
#pragma unroll
    for (int k = 0; k < K; ++k) {
        wv[k] = (mv[k] == -INFINITY || M == -INFINITY) ? 0.f : exp2f(mv[k] - M);
        Z = fmaf(wv[k], zv[k], Z);
    }
    Z = warp_sum(Z);
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int u = 0; u < NP; ++u) {
        const float w = __shfl_sync(0xffffffffu, wv[u >> 5], u & 31);
        // a partition with weight 0 may hold anything (it attended no row): do not touch its values
        if (w != 0.f) {
            if (u & 1) acc1 = fmaf(w, c[u], acc1);
            else acc0 = fmaf(w, c[u], acc0);
        }
    }
    *out = Z > 0.f ? (acc0 + acc1) / Z : 0.f;
}

// NP > 0: P <= NP, every load issued up front (one instantiation per size, so a small P does not pay
// for the registers of a large one); NP == 0: any P, weights through shared memory.
template <int NP>
__global__ void __launch_bounds__(128) lse_merge_kernel(const float *__restrict__ ws, int B, int P, int H,
                                                        float *__restrict__ out) {
    // launched as a programmatic dependent of the partial kernel: wait until its partials are written
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int h = blockIdx.x, quarter = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
    PartialView pv(const_cast<float *>(ws), B, P, H);
    const int64_t base = (int64_t)b * P * H + h;
    const int d = quarter * 128 + tid;
    float *o = out + ((int64_t)b * H + h) * kKL + d;
    if constexpr (NP > 0) {
        merge_small<NP>(pv, base, P, H, d, o);
        return;
    }
    // large P: warp 0 turns the maxima into weights in shared memory
    __shared__ float wsh[kMergeMaxP];
    __shared__ float zsh;
    float M = -INFINITY;
    if (tid < 32) {
        for (int p = tid; p < P; p += 32) M = fmaxf(M, pv.m[base + (int64_t)p * H]);
        M = warp_max(M);
        float Z = 0.f;
        for (int p = tid; p < P; p += 32) {
            const float mp = pv.m[base + (int64_t)p * H];
            const float w = (mp == -INFINITY || M == -INFINITY) ? 0.f : exp2f(mp - M);
            if (p < kMergeMaxP) wsh[p] = w;
            Z = fmaf(w, pv.z[base + (int64_t)p * H], Z);
        }
        Z = warp_sum(Z);
        if (tid == 0) zsh = Z;
    }
    __syncthreads();
    const float *cl = pv.cl + base * kKL + d;
    const int64_t pstride = (int64_t)H * kKL;
    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
    const int pw = P < kMergeMaxP ? P : kMergeMaxP;
    // rounds of kBatch independent loads (one per partition)
    constexpr int kBatch = 32;
    for (int p0 = 0; p0 < pw; p0 += kBatch) {
        float c[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) c[u] = p0 + u < pw ? cl[(int64_t)(p0 + u) * pstride] : 0.f;
#pragma unroll
        for (int u = 0; u < kBatch; u += 4) {
            const int q = p0 + u;
            if (q + 0 < pw && wsh[q + 0] != 0.f) acc0 = fmaf(wsh[q + 0], c[u + 0], acc0);
            if (q + 1 < pw && wsh[q + 1] != 0.f) acc1 = fmaf(wsh[q + 1], c[u + 1], acc1);
            if (q + 2 < pw && wsh[q + 2] != 0.f) acc2 = fmaf(wsh[q + 2], c[u + 2], acc2);
            if (q + 3 < pw && wsh[q + 3] != 0.f) acc3 = fmaf(wsh[q + 3], c[u + 3], acc3);
        }
    }
    // partitions beyond the shared-memory slice (P > kMergeMaxP): weights recomputed on the fly
    if (P > kMergeMaxP) {
        float Mx = -INFINITY;
        for (int q = 0; q < P; ++q) Mx = fmaxf(Mx, pv.m[base + (int64_t)q * H]);
        for (int q = kMergeMaxP; q < P; ++q) {
            const float mp = pv.m[base + (int64_t)q * H];
            if (mp == -INFINITY) continue;
            acc1 = fmaf(exp2f(mp - Mx), cl[(int64_t)q * pstride], acc1);
        }
    }
    const float Z = zsh;
    const float inv = Z > 0.f ? 1.f / Z : 0.f;
    *o = ((acc0 + acc1) + (acc2 + acc3)) * inv;
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs &a, cudaStream_t st) {
    const size_t smem = sizeof(Smem);
    cudaError_t e = cudaFuncSetAttribute(attn_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.P, (unsigned)((a.H + kHB - 1) / kHB), (unsigned)a.B);
    attn_simt_kernel<<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_lse_merge(const float *ws, int B, int P, int H, float *out, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)H, 4u, (unsigned)B);
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (encode && P <= kMergeTma) {
        // cl viewed as [B*P][H][512] f32: one box = 128 columns x 1 head x the item's P partitions
        CUtensorMap map;
        const cuuint64_t dims[3] = {(cuuint64_t)kKL, (cuuint64_t)H, (cuuint64_t)B * (cuuint64_t)P};
        const cuuint64_t strides[2] = {(cuuint64_t)kKL * sizeof(float), (cuuint64_t)H * kKL * sizeof(float)};
        const cuuint32_t box[3] = {128u, 1u, (cuuint32_t)P}, es[3] = {1u, 1u, 1u};
        if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(ws), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
            cudaError_t e = cudaFuncSetAttribute(lse_merge_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)(merge_tma_bar_offset(kMergeTma) + sizeof(uint64_t)));
            if (e != cudaSuccess) return e;
            cfg.dynamicSmemBytes = merge_tma_bar_offset(P) + sizeof(uint64_t);
            e = cudaLaunchKernelEx(&cfg, lse_merge_tma_kernel, map, ws, B, P, H, out);
            if (e != cudaSuccess) return e;
            return cudaGetLastError();
        }
    }
    cudaError_t e = P <= 16   ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<16>, ws, B, P, H, out)
                    : P <= 32 ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<32>, ws, B, P, H, out)
                    : P <= 64 ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<64>, ws, B, P, H, out)
                    : P <= 96 ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<96>, ws, B, P, H, out)
                    : P <= kMergeFast ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<kMergeFast>, ws, B, P, H, out)
                                      : cudaLaunchKernelEx(&cfg, lse_merge_kernel<0>, ws, B, P, H, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kv8
