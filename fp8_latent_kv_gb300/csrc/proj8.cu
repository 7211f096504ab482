// proj8.cu -- the absorb projections through an fmt=8 kv_b_proj (page "feat: fmt=8 (fp8-e4m3)
// decode on the kv_b absorb path, CPU and CUDA": raw e4m3 bytes, one f32 scale per 128x128 block,
// block-row-major).  kv_b has H*256 rows of 512: head h's rows 256h..256h+127 are W_UK (the key's
// no-position part), rows 256h+128..256h+255 are W_UV (the value part).
//
//   q absorb:     q_lat[s][h][c] = sum_j q_nope[s][h][j] * W[256h + j][c]         (j < 128, c < 512)
//   out project:  out[s][h][v]   = sum_c W[256h + 128 + v][c] * ctx[s][h][c]     (v < 128, c < 512)
//
// A head's W_UK rows are one block row, so a q_lat column's scale is one factor (applied after the
// sum); an output row of W_UV crosses four blocks, so each block's partial sum takes its own scale.
// Weights are decoded exactly (e4m3 -> f16 -> f32) and products summed in f32.
//
// This file holds the shape for a few query rows (decode: every weight byte is read once, coalesced,
// and used for all rows, on the CUDA cores); more rows (prefill chunks) go to the tensor-core kernels of
// proj8_tc.cu.
#include "internal.h"
#include "sm100.cuh"

namespace kv8 {
namespace {

constexpr int kNope = KV8_NOPE;  // 128
constexpr int kVH = KV8_VHEAD;   // 128
constexpr int kKvbRows = kNope + kVH;
constexpr int kBlk = 128;        // scale block edge
constexpr int kNbc = kKL / kBlk; // scale blocks per kv_b row (4)
constexpr int kSmallS = 8;       // up to this many rows: the weight-streaming kernels

// four e4m3 bytes (byte 0 first) -> four floats, exactly
__device__ __forceinline__ float4 dec4(uint32_t w) {
    uint32_t lo, hi;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((uint16_t)(w & 0xFFFFu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((uint16_t)(w >> 16)));
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
    return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ float load_act(const void *p, int64_t i, int bf16) {
    return bf16 ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]) : static_cast<const float *>(p)[i];
}

// ------------------------------------------------------------------------------------------------
// q absorb, few rows.  CTA (h, column block cb): 8 warps; warp g sums rows j = 16g..16g+15, lane l
// owns columns 4l..4l+3 of the block.  Each warp instruction reads 128 contiguous weight bytes.
// ------------------------------------------------------------------------------------------------
template <int NS>
__global__ void __launch_bounds__(256) q_absorb_small(const void *__restrict__ q_nope, int q_bf16, int S, int H,
                                                      const uint8_t *__restrict__ w8, const float *__restrict__ w_scale,
                                                      void *__restrict__ q_lat, int out_bf16) {
    __shared__ float qs[NS][kNope];
    __shared__ float4 red[8][NS][32];
    const int h = blockIdx.x, cb = blockIdx.y, tid = threadIdx.x, g = tid >> 5, lane = tid & 31;
    // launched as a programmatic dependent: the weights (never written by the kernel before this one on the
    // stream) stream in while that kernel finishes; the activations only after it has completed
    sm100::grid_launch_dependents();
    const uint8_t *wb = w8 + ((int64_t)h * kKvbRows + 16 * g) * kKL + cb * kBlk + 4 * lane;
    uint32_t wv[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) wv[r] = __ldg(reinterpret_cast<const uint32_t *>(wb + (int64_t)r * kKL));
    sm100::grid_dependency_wait();
    for (int i = tid; i < NS * kNope; i += 256) {
        const int s = i / kNope, j = i - s * kNope;
        qs[s][j] = s < S ? load_act(q_nope, ((int64_t)s * H + h) * kNope + j, q_bf16) : 0.f;
    }
    __syncthreads();
    float4 acc[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) acc[s] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float4 w = dec4(wv[r]);
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const float q = qs[s][16 * g + r];
            acc[s].x = fmaf(q, w.x, acc[s].x);
            acc[s].y = fmaf(q, w.y, acc[s].y);
            acc[s].z = fmaf(q, w.z, acc[s].z);
            acc[s].w = fmaf(q, w.w, acc[s].w);
        }
    }
#pragma unroll
    for (int s = 0; s < NS; ++s) red[g][s][lane] = acc[s];
    __syncthreads();
    const float sc = __ldg(w_scale + (int64_t)(2 * h) * kNbc + cb);
    for (int i = tid; i < NS * 32; i += 256) {
        const int s = i >> 5, l = i & 31;
        if (s >= S) continue;
        float4 t = red[0][s][l];
#pragma unroll
        for (int gg = 1; gg < 8; ++gg) {
            const float4 u = red[gg][s][l];
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
        const int64_t o = ((int64_t)s * H + h) * kKL + cb * kBlk + 4 * l;
        if (out_bf16) {
            __nv_bfloat162 *d = reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(q_lat) + o);
            d[0] = __floats2bfloat162_rn(t.x * sc, t.y * sc);
            d[1] = __floats2bfloat162_rn(t.z * sc, t.w * sc);
        } else {
            *reinterpret_cast<float4 *>(static_cast<float *>(q_lat) + o) = make_float4(t.x * sc, t.y * sc, t.z * sc, t.w * sc);
        }
    }
}

// ------------------------------------------------------------------------------------------------
// out project, few rows.  CTA (h, 32 value rows): warp w takes rows 4w..4w+3 of them.  For a row, lane
// l reads the 4 weight bytes at columns 128k + 4l (k = 0..3: one per scale block; each warp
// instruction reads 128 contiguous bytes) and the matching context values (consecutive lanes,
// consecutive 16 bytes of shared memory); each block's partial sum takes its scale, the warp sums.
// ------------------------------------------------------------------------------------------------
template <int NS>
__global__ void __launch_bounds__(256) out_project_small(const float *__restrict__ ctx, int S, int H,
                                                         const uint8_t *__restrict__ w8,
                                                         const float *__restrict__ w_scale, float *__restrict__ out) {
    __shared__ __align__(16) float xs[NS][kKL];
    const int h = blockIdx.x, v0 = blockIdx.y * 32, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // launched as a programmatic dependent: the weights (never written by the kernel before this one on the
    // stream) stream in while that kernel finishes; the context rows only after it has completed
    sm100::grid_launch_dependents();
    uint32_t wv[4][kNbc];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const uint8_t *row = w8 + ((int64_t)h * kKvbRows + kNope + v0 + 4 * warp + r) * kKL + 4 * lane;
#pragma unroll
        for (int k = 0; k < kNbc; ++k) wv[r][k] = __ldg(reinterpret_cast<const uint32_t *>(row + k * kBlk));
    }
    float sc[kNbc];
#pragma unroll
    for (int k = 0; k < kNbc; ++k) sc[k] = __ldg(w_scale + (int64_t)(2 * h + 1) * kNbc + k);
    sm100::grid_dependency_wait();
    for (int i = tid; i < NS * kKL / 4; i += 256) {
        const int s = i / (kKL / 4), c4 = i - s * (kKL / 4);
        *reinterpret_cast<float4 *>(&xs[s][4 * c4]) =
            s < S ? __ldg(reinterpret_cast<const float4 *>(ctx + ((int64_t)s * H + h) * kKL) + c4)
                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        float4 w[kNbc];
#pragma unroll
        for (int k = 0; k < kNbc; ++k) w[k] = dec4(wv[r][k]);
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            if (s >= S) break;
            float a = 0.f;
#pragma unroll
            for (int k = 0; k < kNbc; ++k) {
                const float4 x = *reinterpret_cast<const float4 *>(&xs[s][k * kBlk + 4 * lane]);
                float p = w[k].x * x.x;
                p = fmaf(w[k].y, x.y, p);
                p = fmaf(w[k].z, x.z, p);
                p = fmaf(w[k].w, x.w, p);
                a = fmaf(sc[k], p, a);
            }
            a = warp_sum(a);
            if (lane == 0) out[((int64_t)s * H + h) * kVH + v0 + 4 * warp + r] = a;
        }
    }
}

}  // namespace

cudaError_t launch_q_absorb(const void *q_nope, int q_bf16, int S, int H, const uint8_t *w8, const float *w_scale,
                            void *q_lat, int out_bf16, int *err_word, cudaStream_t st) {
    if (S > kSmallS) return launch_q_absorb_tc(q_nope, q_bf16, S, H, w8, w_scale, q_lat, out_bf16, err_word, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)H, (unsigned)kNbc);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e =
        S <= 1   ? cudaLaunchKernelEx(&cfg, q_absorb_small<1>, q_nope, q_bf16, S, H, w8, w_scale, q_lat, out_bf16)
        : S <= 4 ? cudaLaunchKernelEx(&cfg, q_absorb_small<4>, q_nope, q_bf16, S, H, w8, w_scale, q_lat, out_bf16)
                 : cudaLaunchKernelEx(&cfg, q_absorb_small<kSmallS>, q_nope, q_bf16, S, H, w8, w_scale, q_lat, out_bf16);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_out_project(const float *ctx, int S, int H, const uint8_t *w8, const float *w_scale, float *out,
                               int *err_word, cudaStream_t st) {
    if (S > kSmallS) return launch_out_project_tc(ctx, S, H, w8, w_scale, out, err_word, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)H, (unsigned)(kVH / 32));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = S <= 1   ? cudaLaunchKernelEx(&cfg, out_project_small<1>, ctx, S, H, w8, w_scale, out)
                          : S <= 4 ? cudaLaunchKernelEx(&cfg, out_project_small<4>, ctx, S, H, w8, w_scale, out)
                                   : cudaLaunchKernelEx(&cfg, out_project_small<kSmallS>, ctx, S, H, w8, w_scale, out);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kv8
