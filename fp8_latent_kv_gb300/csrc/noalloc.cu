// noalloc.cu -- the decode entry point for callers that cannot allocate device memory.
//
// The split-T partials normally live in a workspace the caller allocates.  Here they live in one
// fixed array that is part of the library's device image, so neither the caller nor the library
// allocates anything.  The array is shared by every call on a device and holds KV8_NOALLOC_SCRATCH_BYTES;
// requests whose partials do not fit are refused.  Calls that overlap on the GPU race on the array.
#include "internal.h"

namespace {

// One copy per device, resident from module load until the process exits.  Host code must not use
// this name as a pointer: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KV8_NOALLOC_SCRATCH_BYTES];

// Device address of the array in the current device's context, looked up on every call: a context
// that was destroyed and created again (cudaDeviceReset) reloads the module, possibly at another
// address, so no address is kept between calls.  The first lookup in a context loads the module.
int scratch_address(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return KV8_ECUDA;
    }
    *out = p;
    return KV8_OK;
}

}  // namespace

extern "C" int mla_absorb_decode8_noalloc(const void *q_lat, const void *q_rope, int q_dtype, int H,
                                          const uint8_t *kv8, const float *kv_scale, int64_t T, float sm_scale,
                                          int P_req, int *err_word, float *out, void *stream) {
    int P = 0;
    int rc = mla_decode8_partitions(H, T, P_req, &P);
    if (rc != KV8_OK) return rc;
    size_t need = 0;
    rc = mla_decode8_workspace_bytes(H, T, P, &need);
    if (rc != KV8_OK) return rc;
    if (need > KV8_NOALLOC_SCRATCH_BYTES) {
        if (P_req != 0) return KV8_EWORKSPACE;  // an explicit partition count that does not fit
        while (P > 1 && need > KV8_NOALLOC_SCRATCH_BYTES) {
            --P;
            rc = mla_decode8_workspace_bytes(H, T, P, &need);
            if (rc != KV8_OK) return rc;
        }
        if (need > KV8_NOALLOC_SCRATCH_BYTES) return KV8_EWORKSPACE;
    }
    void *scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != KV8_OK) return rc;
    return mla_absorb_decode8(q_lat, q_rope, q_dtype, H, kv8, kv_scale, T, sm_scale, P, scratch,
                              KV8_NOALLOC_SCRATCH_BYTES, err_word, out, stream);
}
