// copy.cu -- kv8_copy: byte copies between device-accessible buffers, moved by the SMs.
//
// On a GPU whose host memory is coherently attached (NVLink-C2C), page-locked host memory is mapped
// into the device's address space and SM loads and stores reach it directly.  A step's inputs and
// outputs are small (a query, a fresh row, one context); a kernel moves them with less fixed cost
// than a copy-engine transfer.
#include "internal.h"
#include "sm100.cuh"

namespace kv8 {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte loads in flight per thread (the host side has a long latency)

__global__ void __launch_bounds__(kCopyThreads) copy16_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                              int64_t n16) {
    sm100::grid_launch_dependents();  // a programmatic dependent waits for this grid before it reads
    const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
    for (int64_t i0 = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; i0 < n16; i0 += stride * kCopyUnroll) {
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n16) v[u] = src[i];
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n16) dst[i] = v[u];
        }
    }
}

__global__ void __launch_bounds__(kCopyThreads) copy1_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                                                             int64_t n) {
    sm100::grid_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * kCopyThreads;
    for (int64_t i = (int64_t)blockIdx.x * kCopyThreads + threadIdx.x; i < n; i += stride) dst[i] = src[i];
}

unsigned copy_blocks(int64_t items, int unroll) {
    int64_t b = (items + (int64_t)kCopyThreads * unroll - 1) / ((int64_t)kCopyThreads * unroll);
    const int64_t cap = 152 * 8;  // 8 blocks per SM of a 152-SM part
    return (unsigned)(b < 1 ? 1 : b > cap ? cap : b);
}

}  // namespace

cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t st) {
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    if (((d | s) & 15u) == 0) {
        const int64_t n16 = (int64_t)(bytes / 16);
        if (n16 > 0)
            copy16_kernel<<<copy_blocks(n16, kCopyUnroll), kCopyThreads, 0, st>>>(
                static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16);
        const int64_t tail = (int64_t)(bytes % 16);
        if (tail > 0)
            copy1_kernel<<<1, kCopyThreads, 0, st>>>(static_cast<const uint8_t *>(src) + n16 * 16,
                                                      static_cast<uint8_t *>(dst) + n16 * 16, tail);
    } else {
        copy1_kernel<<<copy_blocks((int64_t)bytes, 1), kCopyThreads, 0, st>>>(static_cast<const uint8_t *>(src),
                                                                              static_cast<uint8_t *>(dst),
                                                                              (int64_t)bytes);
    }
    return cudaGetLastError();
}

}  // namespace kv8
