/* Memory- and UB-sanitizer driver for the oracle (oracle/kv8_oracle.c): calls every function on small
 * inputs, edge cases included (T = 1, zero and subnormal rows, non-finite values, empty partitions,
 * out-of-range and duplicate selection indices, k > n).  Built with -fsanitize=address,undefined by
 * tests/test_sanitizers.py; any report aborts the run.  Values are checked by the oracle's pins, not here. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

double kv8o_e4m3_decode(uint8_t b);
void kv8o_e4m3_table(double *out256);
uint8_t kv8o_e4m3_encode(float y);
uint8_t kv8o_e4m3_encode_scan(float y);
void kv8o_encode_array(const float *y, int64_t n, uint8_t *out);
int64_t kv8o_encode_change_points(uint32_t *out, int64_t cap);
void kv8o_quant_rows_w(const float *x, int64_t n, int width, uint8_t *q, float *scale);
void kv8o_quant_rows(const float *x, int64_t n, uint8_t *q, float *scale);
void kv8o_dequant_rows(const uint8_t *q, const float *scale, int64_t n, double *out);
void kv8o_attn_decode(const float *q_lat, const float *q_rope, int H, const uint8_t *kv8, const float *scale,
                      int64_t T, float sm_scale, float *out);
void kv8o_attn_decode_split(const float *q_lat, const float *q_rope, int H, const uint8_t *kv8, const float *scale,
                            int64_t T, float sm_scale, int P, double *cl_part, double *m_part, double *z_part,
                            float *out);
void kv8o_attn_select(const float *q_lat, const float *q_rope, int B, int H, const uint8_t *kv8, const float *scale,
                      int64_t T, int64_t seq_stride_rows, const int32_t *idx, int NS, float sm_scale, float *out,
                      int64_t *bad);
void kv8o_attn_prefill(const float *q_lat, const float *q_rope, int nq, int H, const int64_t *pos,
                       const uint8_t *kv8, const float *scale, int64_t T, float sm_scale, float *out);
void kv8o_q_absorb(const float *q_nope, int S, int H, const uint8_t *w8, const float *w_scale, float *q_lat);
void kv8o_out_project(const float *ctx, int S, int H, const uint8_t *w8, const float *w_scale, float *out);
void kv8o_index_scores(const uint8_t *q8, const float *q_scale, const float *w, int B, int HI, int DI,
                       const uint8_t *k8, const float *k_scale, int64_t T, int64_t seq_stride_rows, double *scores);
void kv8o_topk(const double *scores, int64_t n, int k, int32_t *idx);
void kv8o_attn_mixed_decode(const uint8_t *q8, const float *q_scale, const float *q_rope, int H, const uint8_t *k8,
                            const float *k_scale, const float *k_rope, int64_t T, float sm_scale, float *out);
int kv8o_num_threads(void);
void kv8o_set_num_threads(int n);

static uint64_t g_state = 0x9E3779B97F4A7C15ull;
static double unif(void) {  /* splitmix64 -> [0, 1) */
    uint64_t z = (g_state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return (double)(z >> 11) * (1.0 / 9007199254740992.0);
}
static float gauss(void) { return (float)(sqrt(-2.0 * log(unif() + 1e-300)) * cos(6.283185307179586 * unif())); }
static void *xalloc(size_t n) {
    void *p = malloc(n ? n : 1);
    if (!p) { fprintf(stderr, "out of memory\n"); exit(2); }
    return p;
}
static float *frand(size_t n, float mag) {
    float *p = (float *)xalloc(n * sizeof(float));
    for (size_t i = 0; i < n; ++i) p[i] = gauss() * mag;
    return p;
}

int main(void) {
    kv8o_set_num_threads(2);
    (void)kv8o_num_threads();
    double tab[256];
    kv8o_e4m3_table(tab);
    for (int b = 0; b < 256; ++b) (void)kv8o_e4m3_decode((uint8_t)b);
    const float specials[] = {0.f, -0.f, 1e-30f, -1e-30f, 448.f, 464.f, 1e30f, INFINITY, -INFINITY, NAN, 0.0009765625f};
    for (size_t i = 0; i < sizeof specials / sizeof specials[0]; ++i) {
        (void)kv8o_e4m3_encode(specials[i]);
        (void)kv8o_e4m3_encode_scan(specials[i]);
    }
    uint8_t enc[11];
    kv8o_encode_array(specials, 11, enc);
    uint32_t cps[300];
    (void)kv8o_encode_change_points(cps, 300);

    /* rows: T = 37, one zero row, one subnormal row, one row with a NaN and an inf */
    const int T = 37, H = 3;
    float *rows = frand((size_t)T * 576, 1.f);
    memset(rows + 5 * 576, 0, 576 * sizeof(float));
    for (int i = 0; i < 576; ++i) rows[9 * 576 + i] *= 1e-39f;
    rows[11 * 576 + 3] = NAN;
    rows[11 * 576 + 4] = INFINITY;
    uint8_t *kv8 = (uint8_t *)xalloc((size_t)T * 576);
    float *sc = (float *)xalloc((size_t)T * sizeof(float));
    kv8o_quant_rows(rows, T, kv8, sc);
    double *deq = (double *)xalloc((size_t)T * 576 * sizeof(double));
    kv8o_dequant_rows(kv8, sc, T, deq);
    uint8_t *q128 = (uint8_t *)xalloc((size_t)T * 576);
    float *s128 = (float *)xalloc((size_t)T * 4 * sizeof(float));
    kv8o_quant_rows_w(rows, T, 128, q128, s128);
    kv8o_quant_rows_w(rows, T, 448, q128, s128);

    float *ql = frand((size_t)H * 512, 1.f), *qr = frand((size_t)H * 64, 1.f);
    float *out = (float *)xalloc((size_t)H * 512 * sizeof(float));
    const float sm = 0.0721687836f;
    kv8o_attn_decode(ql, qr, H, kv8, sc, T, sm, out);
    kv8o_attn_decode(ql, qr, H, kv8, sc, 1, sm, out);
    for (int P = 1; P <= 64; P = P * 2 + 1) {  /* P = 1, 3, 7, 15, 31, 63 (more partitions than rows too) */
        double *cl = (double *)xalloc((size_t)P * H * 512 * sizeof(double));
        double *mp = (double *)xalloc((size_t)P * H * sizeof(double)), *zp = (double *)xalloc((size_t)P * H * sizeof(double));
        kv8o_attn_decode_split(ql, qr, H, kv8, sc, T, sm, P, cl, mp, zp, out);
        free(cl); free(mp); free(zp);
    }
    /* selection: 2 items in one cache (stride 16), duplicates and out-of-range indices */
    const int B = 2, NS = 6;
    const int32_t idx[12] = {0, 3, 3, 15, -1, 40, 1, 2, 16, 7, 7, 100000};
    float *qls = frand((size_t)B * H * 512, 1.f), *qrs = frand((size_t)B * H * 64, 1.f);
    float *outs = (float *)xalloc((size_t)B * H * 512 * sizeof(float));
    int64_t bad = 0;
    kv8o_attn_select(qls, qrs, B, H, kv8, sc, 16, 16, idx, NS, sm, outs, &bad);
    /* prefill: 3 queries at positions 0, 20, 36 */
    const int64_t pos[3] = {0, 20, 36};
    float *qlp = frand((size_t)3 * H * 512, 1.f), *qrp = frand((size_t)3 * H * 64, 1.f);
    float *outp = (float *)xalloc((size_t)3 * H * 512 * sizeof(float));
    kv8o_attn_prefill(qlp, qrp, 3, H, pos, kv8, sc, T, sm, outp);
    /* absorb projections: S = 3, H = 2; kv_b [H*256][512] e4m3 with block scales */
    const int S = 3, Hp = 2;
    uint8_t *w8 = (uint8_t *)xalloc((size_t)Hp * 256 * 512);
    for (size_t i = 0; i < (size_t)Hp * 256 * 512; ++i) w8[i] = (uint8_t)((unif() * 254.0)) & 0x7E;
    float *wsc = frand((size_t)((Hp * 256 + 127) / 128) * 4, 1e-2f);
    float *qn = frand((size_t)S * Hp * 128, 1.f), *qlo = (float *)xalloc((size_t)S * Hp * 512 * sizeof(float));
    kv8o_q_absorb(qn, S, Hp, w8, wsc, qlo);
    float *ctx = frand((size_t)S * Hp * 512, 1.f), *ho = (float *)xalloc((size_t)S * Hp * 128 * sizeof(float));
    kv8o_out_project(ctx, S, Hp, w8, wsc, ho);
    /* indexer: 2 queries x 16 index heads x 128 over 2 x 50 keys; top-k with ties and k > n */
    const int HI = 16, DI = 128, TK = 50;
    float *qx = frand((size_t)2 * HI * DI, 1.f), *kx = frand((size_t)2 * TK * DI, 1.f), *wi = frand((size_t)2 * HI, 0.1f);
    uint8_t *q8 = (uint8_t *)xalloc((size_t)2 * HI * DI), *k8 = (uint8_t *)xalloc((size_t)2 * TK * DI);
    float *qs = (float *)xalloc((size_t)2 * HI * sizeof(float)), *ks = (float *)xalloc((size_t)2 * TK * sizeof(float));
    kv8o_quant_rows_w(qx, 2 * HI, DI, q8, qs);
    kv8o_quant_rows_w(kx, 2 * TK, DI, k8, ks);
    double *scores = (double *)xalloc((size_t)2 * TK * sizeof(double));
    kv8o_index_scores(q8, qs, wi, 2, HI, DI, k8, ks, TK, TK, scores);
    int32_t tk[64];
    kv8o_topk(scores, TK, 10, tk);
    kv8o_topk(scores, TK, 64, tk);
    double ties[40];
    for (int i = 0; i < 40; ++i) ties[i] = (double)(i % 3);
    kv8o_topk(ties, 40, 7, tk);
    /* mixed cache: 448 e4m3 + 64 rope values per row */
    const int TM = 9;
    float *mn = frand((size_t)TM * 448, 1.f), *mr = frand((size_t)TM * 64, 1.f);
    uint8_t *m8 = (uint8_t *)xalloc((size_t)TM * 448);
    float *ms = (float *)xalloc((size_t)TM * sizeof(float));
    kv8o_quant_rows_w(mn, TM, 448, m8, ms);
    float *qmn = frand((size_t)H * 448, 1.f), *qmr = frand((size_t)H * 64, 1.f);
    uint8_t *qm8 = (uint8_t *)xalloc((size_t)H * 448);
    float *qms = (float *)xalloc((size_t)H * sizeof(float));
    kv8o_quant_rows_w(qmn, H, 448, qm8, qms);
    kv8o_attn_mixed_decode(qm8, qms, qmr, H, m8, ms, mr, TM, sm, out);

    free(rows); free(kv8); free(sc); free(deq); free(q128); free(s128); free(ql); free(qr); free(out);
    free(qls); free(qrs); free(outs); free(qlp); free(qrp); free(outp); free(w8); free(wsc); free(qn); free(qlo);
    free(ctx); free(ho); free(qx); free(kx); free(wi); free(q8); free(k8); free(qs); free(ks); free(scores);
    free(mn); free(mr); free(m8); free(ms); free(qmn); free(qmr); free(qm8); free(qms);
    printf("oracle driver ok\n");
    return 0;
}
