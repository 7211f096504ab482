// quant_row.cuh -- the e4m3 encoder and the per-row quantizer's f32 steps, shared by every kernel that
// quantizes (cache rows, index keys, index queries), so all of them produce the same bytes.
//
// Page "KV8 long-context CUDA: fp8 device shadow, split-T kernels, DSA-aware gather", first commit
// message, c/kv_fp8.h item: round-to-nearest-even encoder clamped to +-448 that keeps the sign of zero
// and turns NaN into a zero byte; per-row scale amax/448 with a guard for an amax so small that
// 448/amax is not finite.
#pragma once

#include "common.cuh"

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

// The row's f32 factors: y = (x * pre) * mul encodes to the row's bytes; scale = amax / 448.
__device__ __forceinline__ void row_quant_factors(float amax, float &pre, float &mul, float &scale) {
    pre = 1.f;
    mul = 1.f;
    if (amax != 0.f) {
        mul = __fdiv_rn(448.f, amax);
        if (isinf(mul)) {  // subnormal-amax guard
            pre = 18446744073709551616.f;  // 2^64
            mul = __fdiv_rn(448.f, __fmul_rn(amax, pre));
        }
    }
    scale = __fdiv_rn(amax, 448.f);
}

}  // namespace kv8
