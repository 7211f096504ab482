// Memory- and UB-sanitizer driver for the host side of the C ABI (include/kv8mla.h).  Built with
// -fsanitize=address,undefined together with the library's sources by tests/test_sanitizers.py and run
// with every GPU hidden (CUDA_VISIBLE_DEVICES empty), so no kernel can start:
//   * invalid arguments are rejected by host validation with KV8_EINVAL / KV8_EWORKSPACE;
//   * a well-formed call reaches its launch, the CUDA runtime refuses it (no device), and the call
//     returns KV8_ECUDA: the host-side launch failure path of every entry point.
// Pointers are aligned host addresses that the library never dereferences on the host.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kv8mla.h"

static int g_fail = 0;
#define EXPECT(call, want)                                                                               \
    do {                                                                                                 \
        const int rc_ = (call);                                                                          \
        if (rc_ != (want)) {                                                                             \
            fprintf(stderr, "line %d: %s returned %d, expected %d\n", __LINE__, #call, rc_, (int)(want)); \
            g_fail = 1;                                                                                  \
        }                                                                                                \
    } while (0)

int main() {
    // one arena of aligned fake buffers (never read or written by the host code under test)
    const size_t arena_bytes = (size_t)1 << 20;
    unsigned char *arena = static_cast<unsigned char *>(aligned_alloc(256, arena_bytes));
    memset(arena, 0, arena_bytes);
    void *a = arena, *b = arena + 65536, *c = arena + 131072, *d = arena + 196608, *w = arena + 262144;
    void *mis = arena + 4;  // 4-byte aligned only
    auto *f = static_cast<float *>(a);
    auto *u8 = static_cast<uint8_t *>(b);
    auto *sc = static_cast<float *>(c);
    auto *out = static_cast<float *>(d);
    auto *i32 = static_cast<int32_t *>(d);
    auto *i64 = static_cast<int64_t *>(d);
    int err_word = 0, status = 0;
    size_t sz = 0;
    int P = 0;

    // ---- strings and sizes
    for (int code = -6; code <= 1; ++code)
        if (!kv8_strerror(code) || !kv8_strerror(code)[0]) g_fail = 1;
    EXPECT(mla_decode8_partitions(128, 262144, 0, &P), KV8_OK);
    EXPECT(mla_decode8_partitions(0, 10, 0, &P), KV8_EINVAL);
    EXPECT(mla_decode8_partitions(16, 10, 0, nullptr), KV8_EINVAL);
    EXPECT(mla_decode8_workspace_bytes(128, 262144, 0, &sz), KV8_OK);
    EXPECT(mla_decode8_workspace_bytes(129, 10, 0, &sz), KV8_EINVAL);
    EXPECT(mla_decode8_workspace_bytes(16, 0, 0, &sz), KV8_EINVAL);
    EXPECT(mla_decode8_workspace_bytes(16, (1 << 20) + 1, 0, &sz), KV8_EINVAL);
    EXPECT(mla_sel8_workspace_bytes(8, 128, 2048, &sz), KV8_OK);
    EXPECT(mla_sel8_workspace_bytes(8, 128, 4097, &sz), KV8_EINVAL);
    EXPECT(mla_mixed_decode8_workspace_bytes(128, 65536, &sz), KV8_OK);
    EXPECT(mla_mixed_decode8_workspace_bytes(0, 65536, &sz), KV8_EINVAL);
    EXPECT(mla_batch_decode8_workspace_bytes(8, 128, 32768, &sz), KV8_OK);
    EXPECT(mla_batch_decode8_workspace_bytes(0, 128, 32768, &sz), KV8_EINVAL);
    EXPECT(dsa_index_workspace_bytes(8, &sz), KV8_OK);
    EXPECT(dsa_index_workspace_bytes(0, &sz), KV8_EINVAL);

    // ---- validation before any launch
    EXPECT(kv8_encode_e4m3(f, -1, u8, nullptr), KV8_EINVAL);
    EXPECT(kv8_encode_e4m3(static_cast<float *>(mis), 16, u8, nullptr), KV8_EINVAL);
    EXPECT(kv8_quant_rows(nullptr, 4, u8, sc, nullptr), KV8_EINVAL);
    EXPECT(kv8_quant_rows(f, 4, static_cast<uint8_t *>(mis), sc, nullptr), KV8_EINVAL);
    EXPECT(kv8_quant_rows_w(f, 4, 100, u8, sc, nullptr), KV8_EINVAL);
    EXPECT(mla_decode8_partial(a, b, KV8_BF16, 128, u8, sc, 1000, 0.07f, 0, w, 16, &err_word, nullptr), KV8_EWORKSPACE);
    EXPECT(mla_decode8_partial(a, b, 7, 128, u8, sc, 1000, 0.07f, 0, w, 1 << 20, &err_word, nullptr), KV8_EINVAL);
    EXPECT(mla_decode8_partial(mis, b, KV8_BF16, 128, u8, sc, 1000, 0.07f, 0, w, 1 << 20, &err_word, nullptr), KV8_EINVAL);
    EXPECT(mla_absorb_decode8(a, b, KV8_BF16, 128, u8, sc, 1000, __builtin_inff(), 0, w, 1 << 20, &err_word, out, nullptr), KV8_EINVAL);
    EXPECT(mla_lse_merge8(w, 0, 4, 16, out, nullptr), KV8_EINVAL);
    EXPECT(mla_absorb_sel8(a, b, KV8_BF16, 2, 16, u8, sc, 100, 50, i32, 8, 0.07f, w, 1 << 20, &err_word, out, nullptr), KV8_EINVAL);
    EXPECT(mla_absorb_prefill8(a, b, KV8_BF16, 4, 16, 98, u8, sc, 100, 0.07f, &err_word, out, nullptr), KV8_EINVAL);
    EXPECT(mla_absorb_decode8_noalloc(a, b, KV8_BF16, 0, u8, sc, 100, 0.07f, 0, &err_word, out, nullptr), KV8_EINVAL);
    EXPECT(mla_absorb_decode8_noalloc(a, b, KV8_BF16, 128, u8, sc, 262144, 0.07f, 100, &err_word, out, nullptr), KV8_EWORKSPACE);
    EXPECT(mla_absorb_mixed_decode8(a, b, KV8_BF16, 16, u8, sc, static_cast<uint8_t *>(mis), 100, 0.07f, w, 1 << 20, &err_word, out, nullptr), KV8_EINVAL);
    EXPECT(mla_absorb_batch_decode8(a, b, KV8_BF16, 2, 16, u8, sc, 100, 50, i32, 0.07f, w, 1 << 20, &err_word, out, nullptr), KV8_EINVAL);
    EXPECT(kv8_quant_rows_scatter(f, 2, static_cast<int64_t *>(mis), u8, sc, 100, &err_word, nullptr), KV8_EINVAL);
    EXPECT(mla_q_absorb8(a, KV8_BF16, 0, 16, u8, sc, out, KV8_F32, &err_word, nullptr), KV8_EINVAL);
    EXPECT(mla_out_project8(f, 1, 129, u8, sc, out, &err_word, nullptr), KV8_EINVAL);
    EXPECT(dsa_index_topk8(a, KV8_BF16, sc, 2, 17, u8, sc, 100, 100, 10, w, 1 << 20, out, i32, &err_word, nullptr), KV8_EINVAL);
    EXPECT(dsa_index_topk8(a, KV8_BF16, sc, 2, 16, u8, sc, 100, 100, 10, w, 16, out, i32, &err_word, nullptr), KV8_EWORKSPACE);
    EXPECT(kv8_copy(nullptr, a, 16, nullptr), KV8_EINVAL);
    EXPECT(kv8_copy(a, static_cast<unsigned char *>(a) + 8, 16, nullptr), KV8_EINVAL);  // overlapping ranges
    EXPECT(kv8_wait_selftest(10, &err_word, &status, nullptr), KV8_EINVAL);

    // ---- well-formed calls: the launch is refused (no visible device) and reported as KV8_ECUDA
    EXPECT(kv8_encode_e4m3(f, 16, u8, nullptr), KV8_ECUDA);
    EXPECT(kv8_quant_rows(f, 4, u8, sc, nullptr), KV8_ECUDA);
    EXPECT(kv8_quant_rows_w(f, 4, 128, u8, sc, nullptr), KV8_ECUDA);
    size_t need = 0;
    EXPECT(mla_decode8_workspace_bytes(128, 1000, 0, &need), KV8_OK);
    void *ws = aligned_alloc(256, (need + 255) & ~(size_t)255);
    EXPECT(mla_decode8_partial(a, b, KV8_BF16, 128, u8, sc, 1000, 0.07f, 0, ws, need, &err_word, nullptr), KV8_ECUDA);
    EXPECT(mla_decode8_partial(a, b, KV8_F32, 128, u8, sc, 1000, 0.07f, 0, ws, need, &err_word, nullptr), KV8_ECUDA);
    EXPECT(mla_absorb_decode8(a, b, KV8_BF16, 128, u8, sc, 1000, 0.07f, 0, ws, need, &err_word, out, nullptr), KV8_ECUDA);
    EXPECT(mla_lse_merge8(ws, 1, 4, 16, out, nullptr), KV8_ECUDA);
    EXPECT(mla_absorb_decode8_noalloc(a, b, KV8_BF16, 128, u8, sc, 1000, 0.07f, 0, &err_word, out, nullptr), KV8_ECUDA);
    free(ws);
    EXPECT(mla_sel8_workspace_bytes(2, 16, 8, &need), KV8_OK);
    ws = aligned_alloc(256, (need + 255) & ~(size_t)255);
    EXPECT(mla_absorb_sel8(a, b, KV8_BF16, 2, 16, u8, sc, 100, 100, i32, 8, 0.07f, ws, need, &err_word, out, nullptr), KV8_ECUDA);
    free(ws);
    EXPECT(mla_absorb_prefill8(a, b, KV8_BF16, 4, 16, 96, u8, sc, 100, 0.07f, &err_word, out, nullptr), KV8_ECUDA);
    EXPECT(mla_absorb_prefill8(a, b, KV8_F32, 4, 16, 96, u8, sc, 100, 0.07f, &err_word, out, nullptr), KV8_ECUDA);
    EXPECT(mla_mixed_decode8_workspace_bytes(16, 100, &need), KV8_OK);
    ws = aligned_alloc(256, (need + 255) & ~(size_t)255);
    EXPECT(mla_absorb_mixed_decode8(a, b, KV8_BF16, 16, u8, sc, u8, 100, 0.07f, ws, need, &err_word, out, nullptr), KV8_ECUDA);
    free(ws);
    EXPECT(mla_batch_decode8_workspace_bytes(2, 16, 100, &need), KV8_OK);
    ws = aligned_alloc(256, (need + 255) & ~(size_t)255);
    EXPECT(mla_absorb_batch_decode8(a, b, KV8_BF16, 2, 16, u8, sc, 100, 100, i32, 0.07f, ws, need, &err_word, out, nullptr), KV8_ECUDA);
    free(ws);
    EXPECT(kv8_quant_rows_scatter(f, 2, i64, u8, sc, 100, &err_word, nullptr), KV8_ECUDA);
    EXPECT(mla_q_absorb8(a, KV8_BF16, 1, 16, u8, sc, out, KV8_F32, &err_word, nullptr), KV8_ECUDA);
    EXPECT(mla_q_absorb8(a, KV8_BF16, 64, 16, u8, sc, out, KV8_F32, &err_word, nullptr), KV8_ECUDA);
    EXPECT(mla_out_project8(f, 1, 16, u8, sc, out, &err_word, nullptr), KV8_ECUDA);
    EXPECT(mla_out_project8(f, 64, 16, u8, sc, out, &err_word, nullptr), KV8_ECUDA);
    EXPECT(dsa_index_workspace_bytes(2, &need), KV8_OK);
    ws = aligned_alloc(256, (need + 255) & ~(size_t)255);
    EXPECT(dsa_index_topk8(a, KV8_BF16, sc, 2, 16, u8, sc, 100, 100, 10, ws, need, out, i32, &err_word, nullptr), KV8_ECUDA);
    free(ws);
    EXPECT(kv8_wait_selftest(100000, &err_word, &status, nullptr), KV8_ECUDA);
    EXPECT(kv8_copy(a, c, 64, nullptr), KV8_EINVAL);  // the pointers are not visible to any device

    free(arena);
    if (g_fail) return 1;
    printf("abi driver ok\n");
    return 0;
}
