// common.cuh -- device helpers shared by the library's kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "kv8mla.h"

namespace kv8 {

constexpr int kRow = KV8_ROW_BYTES;  // 576 e4m3 bytes per cache row
constexpr int kKL = KV8_KL;          // 512 latent
constexpr int kKR = KV8_KR;          // 64 rope
constexpr float kLog2e = 1.4426950408889634f;

// Partial-set layout in a workspace, for batch item b of B, partition count P, H heads.
struct PartialView {
    float *cl;  // [B][P][H][512]
    float *m;   // [B][P][H]
    float *z;   // [B][P][H]
    __host__ __device__ static size_t floats(int B, int P, int H) {
        return (size_t)B * P * H * (kKL + 2);
    }
    __host__ __device__ PartialView(void *ws, int B, int P, int H) {
        cl = static_cast<float *>(ws);
        m = cl + (size_t)B * P * H * kKL;
        z = m + (size_t)B * P * H;
    }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Four e4m3 bytes (little-endian in w: byte 0 = element 0) -> four f32 values, exactly
// (every e4m3 value is a half value; the hardware conversion is exact).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float &a, float &b, float &c, float &d) {
    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xFFFFu), __NV_E4M3);
    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    float2 f0 = __half22float2(*reinterpret_cast<__half2 *>(&lo));
    float2 f1 = __half22float2(*reinterpret_cast<__half2 *>(&hi));
    a = f0.x;
    b = f0.y;
    c = f1.x;
    d = f1.y;
}

__device__ __forceinline__ void e4m3x2_to_f32(uint16_t w, float &a, float &b) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)w, __NV_E4M3);
    float2 f = __half22float2(*reinterpret_cast<__half2 *>(&h));
    a = f.x;
    b = f.y;
}

}  // namespace kv8
