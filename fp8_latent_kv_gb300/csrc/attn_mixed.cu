// attn_mixed.cu -- decode over the mixed-precision cache (sm_103a, CUDA cores).
//
// Page "B1 Mixed FP8/BF16 FMHA first pass": each KV row keeps its no-position part (448 values) as e4m3
// bytes with a per-row f32 scale and its RoPE part (64 values) as bf16; the query's no-position part is
// quantized from bf16 to e4m3 right before the attention; the head width is 512 = 448 + 64 and the row
// is both key and value.  Per head h and row t:
//     score = sm_scale * ( q_scale[h] * k_scale[t] * sum_i e4m3(q8[h][i]) e4m3(k8[t][i]) + q_rope[h] . k_rope[t] )
//     value = [ k_scale[t] * e4m3(k8[t][0..447]) , k_rope[t][0..63] ]
// The output is split-T partial sets in the layout of the other decode calls (cl[512], m, z), merged by
// the same log-sum-exp merge.
//
// A block owns 32 heads and one partition of the rows.  It quantizes its heads' no-position queries
// with the row quantizer's f32 steps (the bytes the reference quantizer gives) and keeps their decoded
// values; 64-row tiles (448 + 128 bytes per row, 16-byte loads) stream through shared memory; the
// scores of a tile are two dot products per (row, head); the context accumulates 512 columns per head
// in registers (2 per thread: warps 0..6 the no-position columns, warp 7 the RoPE columns).
#include "internal.h"
#include "quant_row.cuh"

#include <math.h>

namespace kv8 {
namespace {

constexpr int kMxNope = KV8_MX_NOPE;   // 448
constexpr int kMxRope = KV8_MX_ROPE;   // 64
constexpr int kMxD = kMxNope + kMxRope;
constexpr int kMHB = 32;               // heads per block
constexpr int kMTR = 64;               // rows per tile
constexpr int kMThreads = 256;
constexpr int kMRowBytes = kMxNope + 2 * kMxRope;  // 576 bytes per staged row
constexpr int kMTileStride = kMRowBytes + 4;        // 580 bytes = 145 words (odd): conflict-free row reads
constexpr int kMSStride = kMHB + 1;

struct MixedSmem {
    float qn[kMHB][kMxNope];          // e4m3 values of the quantized no-position queries (unscaled)
    float qr[kMHB][kMxRope];          // RoPE queries (f32)
    float qscale[kMHB];
    uint8_t tile[kMTR][kMTileStride]; // [448 e4m3 | 64 bf16] per row
    float s[kMTR][kMSStride];         // scores (log2 domain)
    float p[kMTR][kMHB];              // softmax weights of the tile
    float rscale[kMTR];               // row scale, 0 for a row past the end
    float m_run[kMHB], z_run[kMHB], corr[kMHB];
};

struct MixedArgs {
    const void *q_nope, *q_rope;
    int q_bf16, H;
    const uint8_t *k8;
    const float *k_scale;
    const __nv_bfloat16 *k_rope;
    int64_t T;
    float sm_scale_log2;
    int P;
    float *ws;
};

__device__ __forceinline__ float mx_load(const void *base, int64_t i, int bf16) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(base)[i]) : static_cast<const float *>(base)[i];
}

__global__ void __launch_bounds__(kMThreads, 1) attn_mixed_kernel(MixedArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    MixedSmem &sm = *reinterpret_cast<MixedSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int part = blockIdx.x, hb0 = blockIdx.y * kMHB;
    const int nh = min(kMHB, a.H - hb0);
    const int64_t j0 = a.T * part / a.P, j1 = a.T * (part + 1) / a.P;

    // ---- queries: warp w quantizes heads w, w+8, ... (the row quantizer's steps on 448 values)
    for (int h = warp; h < kMHB; h += kMThreads / 32) {
        constexpr int kF4 = kMxNope / 4, kPer = (kF4 + 31) / 32;  // 112 float4, up to 4 per lane
        float4 v[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int f = j * 32 + lane;
            v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (h < nh && f < kF4) {
                const int64_t e = (int64_t)(hb0 + h) * kMxNope + 4 * f;
                v[j] = make_float4(mx_load(a.q_nope, e, a.q_bf16), mx_load(a.q_nope, e + 1, a.q_bf16),
                                   mx_load(a.q_nope, e + 2, a.q_bf16), mx_load(a.q_nope, e + 3, a.q_bf16));
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            amax = finite_abs_max(amax, v[j].x);
            amax = finite_abs_max(amax, v[j].y);
            amax = finite_abs_max(amax, v[j].z);
            amax = finite_abs_max(amax, v[j].w);
        }
        amax = warp_max(amax);
        float pre, mul, qs;
        row_quant_factors(amax, pre, mul, qs);
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const int f = j * 32 + lane;
            if (f < kF4) {
                float e0, e1, e2, e3;
                e4m3x4_to_f32(enc4(scale4(v[j], pre, mul)), e0, e1, e2, e3);
                *reinterpret_cast<float4 *>(&sm.qn[h][4 * f]) = make_float4(e0, e1, e2, e3);
            }
        }
        if (lane == 0) sm.qscale[h] = qs;
        for (int k = lane; k < kMxRope; k += 32)
            sm.qr[h][k] = h < nh ? mx_load(a.q_rope, (int64_t)(hb0 + h) * kMxRope + k, a.q_bf16) : 0.f;
    }
    if (tid < kMHB) {
        sm.m_run[tid] = -INFINITY;
        sm.z_run[tid] = 0.f;
    }
    float acc[kMHB][2];
#pragma unroll
    for (int h = 0; h < kMHB; ++h) acc[h][0] = acc[h][1] = 0.f;

    for (int64_t jt = j0; jt < j1; jt += kMTR) {
        __syncthreads();  // previous tile consumed (and the queries written, on the first tile)
        const int nr = (j1 - jt) < kMTR ? (int)(j1 - jt) : kMTR;
        if (tid < kMTR) sm.rscale[tid] = tid < nr ? __ldg(a.k_scale + jt + tid) : 0.f;
        // ---- tile: per row 28 uint4 of e4m3 bytes + 8 uint4 of bf16 RoPE
        for (int c = tid; c < kMTR * 36; c += kMThreads) {
            const int r = c / 36, col = c - r * 36;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < nr) {
                const int64_t t = jt + r;
                v = col < 28 ? __ldg(reinterpret_cast<const uint4 *>(a.k8 + t * kMxNope) + col)
                             : __ldg(reinterpret_cast<const uint4 *>(a.k_rope + t * kMxRope) + (col - 28));
            }
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
            float sn[8], sr[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) sn[j] = sr[j] = 0.f;
            const uint32_t *rw = reinterpret_cast<const uint32_t *>(&sm.tile[r][0]);
#pragma unroll 4
            for (int k4 = 0; k4 < kMxNope / 4; ++k4) {
                float e0, e1, e2, e3;
                e4m3x4_to_f32(rw[k4], e0, e1, e2, e3);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(&sm.qn[g * 8 + j][k4 * 4]);
                    sn[j] = fmaf(q4.x, e0, sn[j]);
                    sn[j] = fmaf(q4.y, e1, sn[j]);
                    sn[j] = fmaf(q4.z, e2, sn[j]);
                    sn[j] = fmaf(q4.w, e3, sn[j]);
                }
            }
#pragma unroll 4
            for (int k2 = 0; k2 < kMxRope / 2; ++k2) {
                const float2 kr = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&rw[kMxNope / 4 + k2]));
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 q2 = *reinterpret_cast<const float2 *>(&sm.qr[g * 8 + j][k2 * 2]);
                    sr[j] = fmaf(q2.x, kr.x, sr[j]);
                    sr[j] = fmaf(q2.y, kr.y, sr[j]);
                }
            }
            const bool ok = r < nr;
            const float ks = sm.rscale[r];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                sm.s[r][g * 8 + j] = ok ? a.sm_scale_log2 * fmaf(sm.qscale[g * 8 + j] * ks, sn[j], sr[j]) : -INFINITY;
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
                    sm.p[r][h] = pr;
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
        // ---- context: thread -> columns 2*tid, 2*tid+1 (tid < 224: no-position values x row scale;
        // warp 7: the RoPE values)
        {
#pragma unroll
            for (int h = 0; h < kMHB; ++h) {
                const float c = sm.corr[h];
                acc[h][0] *= c;
                acc[h][1] *= c;
            }
            const bool rope = tid >= kMxNope / 2;
            for (int r = 0; r < nr; ++r) {
                float v0, v1;
                if (!rope) {
                    e4m3x2_to_f32(*reinterpret_cast<const uint16_t *>(&sm.tile[r][2 * tid]), v0, v1);
                    const float ks = sm.rscale[r];
                    v0 *= ks;
                    v1 *= ks;
                } else {
                    const float2 f = __bfloat1622float2(
                        *reinterpret_cast<const __nv_bfloat162 *>(&sm.tile[r][kMxNope + 4 * (tid - kMxNope / 2)]));
                    v0 = f.x;
                    v1 = f.y;
                }
#pragma unroll
                for (int h4 = 0; h4 < kMHB / 4; ++h4) {
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
    __syncthreads();
    // ---- the partial set of this partition (cl relative to m, z)
    PartialView pv(a.ws, 1, a.P, a.H);
    const int64_t base = (int64_t)part * a.H + hb0;
    for (int h = 0; h < nh; ++h)
        reinterpret_cast<float2 *>(pv.cl + (base + h) * kKL)[tid] = make_float2(acc[h][0], acc[h][1]);
    if (tid < nh) {
        pv.m[base + tid] = sm.m_run[tid];
        pv.z[base + tid] = sm.z_run[tid];
    }
}

}  // namespace

int mixed_partitions(int H, int64_t T) {
    // one wave of CUDA-core blocks (one per SM of a 152-SM part): P partitions x ceil(H/32) head blocks
    const int64_t hb = (H + kMHB - 1) / kMHB;
    int64_t cap = 152 / hb;
    if (cap < 1) cap = 1;
    const int64_t p = (T + kMTR - 1) / kMTR;
    return (int)(p < cap ? p : cap);
}

cudaError_t launch_attn_mixed(const void *q_nope, const void *q_rope, int q_bf16, int H, const uint8_t *k8,
                              const float *k_scale, const void *k_rope, int64_t T, float sm_scale_log2, int P,
                              float *ws, cudaStream_t st) {
    MixedArgs a{};
    a.q_nope = q_nope;
    a.q_rope = q_rope;
    a.q_bf16 = q_bf16;
    a.H = H;
    a.k8 = k8;
    a.k_scale = k_scale;
    a.k_rope = static_cast<const __nv_bfloat16 *>(k_rope);
    a.T = T;
    a.sm_scale_log2 = sm_scale_log2;
    a.P = P;
    a.ws = ws;
    const size_t smem = sizeof(MixedSmem);
    cudaError_t e = cudaFuncSetAttribute(attn_mixed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)P, (unsigned)((H + kMHB - 1) / kMHB));
    attn_mixed_kernel<<<grid, kMThreads, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kv8
