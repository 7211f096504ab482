// quant8.cu -- e4m3 row quantizer and element encoder (sm_103a).
//
// Page "KV8 long-context CUDA: fp8 device shadow, split-T kernels, DSA-aware gather", first commit
// message, c/kv_fp8.h item: round-to-nearest-even encoder clamped to +-448 that keeps the sign of zero
// and turns NaN into a zero byte; per-row quantizer with a per-row f32 amax/448 scale and a guard for
// an amax so small that 448/amax is not finite.
//
// Design: one warp per row (576 cache elements, or 128 for index keys).  Each lane loads every 32nd
// float4 (coalesced 16-byte loads: a cache row is 144 float4), the warp takes amax with a shuffle
// reduction, every f32 step is an
// explicit round-to-nearest intrinsic (no contraction), and the encode is the hardware
// cvt.rn.satfinite.e4m3x2.f32 (RNE, saturating, sign-preserving) with NaN inputs forced to 0x00.
#include "internal.h"
#include "quant_row.cuh"
#include "sm100.cuh"

namespace kv8 {

// One warp per row of W elements (W/4 float4, coalesced: lane l takes float4 l, l+32, ...).  With
// `dst`, input row r is written to output row dst[r] (appending one row to each of several caches); a
// destination outside [0, cache_rows) is skipped and reported.
template <int W>
__global__ void __launch_bounds__(256) quant_rows_kernel(const float *__restrict__ x, int64_t n,
                                                          uint8_t *__restrict__ q, float *__restrict__ scale,
                                                          const int64_t *__restrict__ dst, int64_t cache_rows,
                                                          int *err_word) {
    // a programmatic dependent (the next call's query prep) may launch now; it waits for this grid
    // before it reads anything
    sm100::grid_launch_dependents();
    constexpr int kF4 = W / 4, kPer = (kF4 + 31) / 32;
    const int lane = threadIdx.x & 31;
    const int64_t in_row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (in_row >= n) return;
    int64_t row = in_row;
    if (dst) {
        row = __ldg(dst + in_row);
        if (row < 0 || row >= cache_rows) {
            if (lane == 0 && err_word) atomicOr(err_word, (int)KV8_ERR_INDEX);
            return;
        }
    }
    const float4 *xr = reinterpret_cast<const float4 *>(x + in_row * W);
    float4 v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int f = j * 32 + lane;
        v[j] = f < kF4 ? __ldg(xr + f) : make_float4(0.f, 0.f, 0.f, 0.f);
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
    float pre, mul, sc;
    row_quant_factors(amax, pre, mul, sc);
    if (lane == 0) scale[row] = sc;
    uint32_t *qr = reinterpret_cast<uint32_t *>(q + row * W);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int f = j * 32 + lane;
        if (f < kF4) qr[f] = enc4(scale4(v[j], pre, mul));
    }
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

cudaError_t launch_quant_rows_w(const float *x, int64_t n, int width, uint8_t *q, float *scale, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int rows_per_block = 8;  // 256 threads
    const int64_t blocks = (n + rows_per_block - 1) / rows_per_block;
    if (width == kRow)
        quant_rows_kernel<kRow><<<(unsigned)blocks, 256, 0, st>>>(x, n, q, scale, nullptr, 0, nullptr);
    else if (width == KV8_IDX_D)
        quant_rows_kernel<KV8_IDX_D><<<(unsigned)blocks, 256, 0, st>>>(x, n, q, scale, nullptr, 0, nullptr);
    else if (width == KV8_MX_NOPE)
        quant_rows_kernel<KV8_MX_NOPE><<<(unsigned)blocks, 256, 0, st>>>(x, n, q, scale, nullptr, 0, nullptr);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_quant_rows_scatter(const float *x, int64_t n, const int64_t *dst, int64_t cache_rows, uint8_t *q,
                                      float *scale, int *err_word, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int64_t blocks = (n + 7) / 8;
    quant_rows_kernel<kRow><<<(unsigned)blocks, 256, 0, st>>>(x, n, q, scale, dst, cache_rows, err_word);
    return cudaGetLastError();
}

cudaError_t launch_quant_rows(const float *x, int64_t n, uint8_t *q, float *scale, cudaStream_t st) {
    return launch_quant_rows_w(x, n, kRow, q, scale, st);
}

cudaError_t launch_encode(const float *y, int64_t n, uint8_t *out, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    int64_t n4 = (n + 3) / 4;
    int64_t blocks = (n4 + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 16;  // a grid-stride loop: a few waves suffice
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    encode_kernel<<<(unsigned)blocks, 256, 0, st>>>(y, n, out);
    return cudaGetLastError();
}

}  // namespace kv8
