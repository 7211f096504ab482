// selftest.cu -- a diagnostic for the bounded waits every tensor-core kernel of the library uses.
//
// One CTA initialises an mbarrier that nothing ever arrives at and waits on it through the same bounded
// wait (sm100.cuh: mbar_wait) the kernels use for their TMA, MMA and softmax hand-offs.  After the limit
// the wait gives up, sets KV8_ERR_TIMEOUT in the error word and the kernel returns normally: no fault, no
// trap, and the context stays usable.  The tests call it to check the timeout path end to end.
#include "internal.h"
#include "sm100.cuh"

namespace kv8 {
namespace {

using namespace sm100;

__global__ void wait_selftest_kernel(uint64_t limit_ns, int *err_word, int *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool done = mbar_wait(&bar, 0, nullptr, err_word, limit_ns);  // no arrival: gives up at the limit
        if (status) *status = done ? 1 : 2;
    }
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, int *err_word, int *status, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns, err_word, status);
    return cudaGetLastError();
}

}  // namespace kv8
