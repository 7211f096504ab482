// quant8.cu -- e4m3 row quantizer and element encoder (sm_103a).
//
// Page "KV8 long-context CUDA: fp8 device shadow, split-T kernels, DSA-aware gather", first commit
// message, c/kv_fp8.h item: round-to-nearest-even encoder clamped to +-448 that keeps the sign of zero
// and turns NaN into a zero byte; per-row quantizer with a per-row f32 amax/448 scale and a guard for
// an amax so small that 448/amax is not finite.
//
// Design: one warp per 576-element row.  Each lane loads 4 or 5 float4 (coalesced 16-byte loads:
// the row is 144 float4), the warp takes amax with a shuffle reduction, every f32 step is an
// explicit round-to-nearest intrinsic (no contraction), and the encode is the hardware
// cvt.rn.satfinite.e4m3x2.f32 (RNE, saturating, sign-preserving) with NaN inputs forced to 0x00.
#include "internal.h"

namespace kv8 {

// Encode two f32 values; returns (byte(hi_elem) << 8) | byte(lo_elem).
__device__ __forceinline__ uint32_t enc2(float lo_elem, float hi_elem) {
    uint16_t v;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(hi_elem), "f"(lo_elem));
    uint32_t r = v;
    if (isnan(lo_elem)) r &= 0xFF00u;
    if (isnan(hi_elem)) r &= 0x00FFu;
    return r;
}

__device__ __forceinline__ uint32_t enc4(float4 v) {
    return enc2(v.x, v.y) | (enc2(v.z, v.w) << 16);
}

__device__ __forceinline__ float4 scale4(float4 v, float pre, float mul) {
    // y = (x * pre) * mul, each product rounded to nearest f32 (pre is 1 or 2^64: exact)
    v.x = __fmul_rn(__fmul_rn(v.x, pre), mul);
    v.y = __fmul_rn(__fmul_rn(v.y, pre), mul);
    v.z = __fmul_rn(__fmul_rn(v.z, pre), mul);
    v.w = __fmul_rn(__fmul_rn(v.w, pre), mul);
    return v;
}

__device__ __forceinline__ float finite_abs_max(float acc, float x) {
    float a = fabsf(x);
    return (a <= 3.402823466e38f) ? fmaxf(acc, a) : acc;  // NaN and inf fail the compare
}

__global__ void __launch_bounds__(256) quant_rows_kernel(const float *__restrict__ x, int64_t n,
                                                          uint8_t *__restrict__ q, float *__restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= n) return;
    const float4 *xr = reinterpret_cast<const float4 *>(x + row * kRow);
    float4 v[5];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __ldg(xr + j * 32 + lane);
    const bool has5 = lane < 16;  // 144 = 4*32 + 16
    v[4] = has5 ? __ldg(xr + 128 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);

    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 5; ++j) {
        amax = finite_abs_max(amax, v[j].x);
        amax = finite_abs_max(amax, v[j].y);
        amax = finite_abs_max(amax, v[j].z);
        amax = finite_abs_max(amax, v[j].w);
    }
    amax = warp_max(amax);

    float pre = 1.f, mul = 1.f;
    if (amax != 0.f) {
        mul = __fdiv_rn(448.f, amax);
        if (isinf(mul)) {  // subnormal-amax guard
            pre = 18446744073709551616.f;  // 2^64
            mul = __fdiv_rn(448.f, __fmul_rn(amax, pre));
        }
    }
    if (lane == 0) scale[row] = __fdiv_rn(amax, 448.f);

    uint32_t *qr = reinterpret_cast<uint32_t *>(q + row * kRow);
#pragma unroll
    for (int j = 0; j < 4; ++j) qr[j * 32 + lane] = enc4(scale4(v[j], pre, mul));
    if (has5) qr[128 + lane] = enc4(scale4(v[4], pre, mul));
}

__global__ void __launch_bounds__(256) encode_kernel(const float *__restrict__ y, int64_t n,
                                                      uint8_t *__restrict__ out) {
    const int64_t n4 = n >> 2;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(y) + i);
        reinterpret_cast<uint32_t *>(out)[i] = enc4(v);
    }
    const int64_t tail = n - (n4 << 2);
    if (blockIdx.x == 0 && threadIdx.x < tail) {
        const int64_t i = (n4 << 2) + threadIdx.x;
        out[i] = (uint8_t)(enc2(y[i], 0.f) & 0xFFu);
    }
}

cudaError_t launch_quant_rows(const float *x, int64_t n, uint8_t *q, float *scale, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int rows_per_block = 8;  // 256 threads
    const int64_t blocks = (n + rows_per_block - 1) / rows_per_block;
    quant_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, n, q, scale);
    return cudaGetLastError();
}

cudaError_t launch_encode(const float *y, int64_t n, uint8_t *out, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    int64_t n4 = (n + 3) / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    encode_kernel<<<(unsigned)blocks, 256, 0, st>>>(y, n, out);
    return cudaGetLastError();
}

}  // namespace kv8
