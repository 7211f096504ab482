/*
 * kv8_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, CPU-only restatement of fp8 latent-KV absorbed MLA attention, used to check the
 * CUDA library and to time a CPU baseline.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference legs may load this library; the product path never does.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (web pages; cited by title and section):
 *   [KV8]  "KV8 long-context CUDA: fp8 device shadow, split-T kernels, DSA-aware gather"
 *          (colibri pull request #300).  First commit message = the KV8 base (fp8 row format,
 *          c/kv_fp8.h codec, absorb score/context loops); second commit message = device
 *          shadow, split-T partial blocks + log-sum-exp merge, DSA gather.
 *   [FMT8] "feat: fmt=8 (fp8-e4m3) decode on the kv_b absorb path, CPU and CUDA"
 *          (colibri pull request #1102), commit "qt_addrow and qt_matvec_rows gain explicit
 *          fmt=8 branches": widen each product to double and accumulate in double.
 *
 * Conventions fixed here (readings of the pages, each listed in the design notes):
 *   - A cache row is D = 576 bytes: Lc (kv_lora, 512) then Rc (qk_rope, 64), one f32 scale.
 *   - e4m3 is the OCP "FN" format: bias 7, no infinities, 0x7F/0xFF are NaN, max 448.
 *   - The encoder rounds to nearest, ties to the even code, saturates at +-448, copies the sign
 *     bit (so -0.0 and negative underflow give 0x80) and stores NaN as +0 (0x00).
 *   - The row quantizer works in f32 with IEEE round-to-nearest and no contraction.
 *   - Attention accumulates in double over the dequantized rows and rounds once to f32.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -fPIC -shared (no -ffast-math).
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* f32 expressions must be evaluated in f32 (no x87 extended precision). */
_Static_assert(FLT_EVAL_METHOD == 0, "f32 arithmetic must be evaluated in f32");

#define KV8O_D 576
#define KV8O_KL 512
#define KV8O_KR 64

/* ---------------------------------------------------------------------------------------------
 * e4m3 decode, by the closed form of the format ([KV8] first commit decodes through a table of all 256 codes).
 * byte b = s eeee mmm; e == 0 is subnormal (m * 2^-9); e == 15, m == 7 is NaN; otherwise
 * (1 + m/8) * 2^(e-7).  The largest finite magnitude is 0x7E = 448.
 * ------------------------------------------------------------------------------------------- */
double kv8o_e4m3_decode(uint8_t b)
{
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 15;
    int m = b & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* The 256-entry table of the page, filled from the closed form above. */
static double g_lut[256];
static int g_lut_ready = 0;

static void lut_init(void)
{
    if (g_lut_ready)
        return;
    for (int b = 0; b < 256; ++b)
        g_lut[b] = kv8o_e4m3_decode((uint8_t)b);
    g_lut_ready = 1;
}

void kv8o_e4m3_table(double *out256)
{
    lut_init();
    memcpy(out256, g_lut, sizeof(g_lut));
}

/* ---------------------------------------------------------------------------------------------
 * e4m3 encode ([KV8] first commit, c/kv_fp8.h item: round to nearest with ties to even,
 * clamped to +-448, the sign of zero kept, NaN turned into a zero byte).
 *
 * Definition used: the nearest of the 127 non-negative finite e4m3 magnitudes (codes 0x00..0x7E,
 * ascending), distance measured exactly in double; on an exact tie the code whose mantissa LSB is
 * 0 wins.  |y| >= 448 (including inf) gives 0x7E.  The sign bit of y is copied.  NaN gives 0x00.
 * The nearest magnitude is found by bisection over the ascending table, then the two neighbours
 * are compared -- the same answer as scanning all 127 values, which a test checks.
 * ------------------------------------------------------------------------------------------- */
uint8_t kv8o_e4m3_encode(float y)
{
    lut_init();
    if (isnan(y))
        return 0x00;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0)
        return sign | 0x7E;
    /* largest code lo in [0, 0x7E] with value(lo) <= a */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (g_lut[mid] <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    int best = lo;
    if (lo < 0x7E) {
        double dl = a - g_lut[lo];
        double du = g_lut[lo + 1] - a;
        if (du < dl || (du == dl && ((lo + 1) & 1) == 0))
            best = lo + 1;
    }
    return sign | (uint8_t)best;
}

/* Brute-force form of the same definition: scan all 127 magnitudes.  Used by a pin test to check
 * the bisection above; slow. */
uint8_t kv8o_e4m3_encode_scan(float y)
{
    lut_init();
    if (isnan(y))
        return 0x00;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0)
        return sign | 0x7E;
    int best = 0;
    double bestd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(a - g_lut[c]);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return sign | (uint8_t)best;
}

void kv8o_encode_array(const float *y, int64_t n, uint8_t *out)
{
    lut_init();
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = kv8o_e4m3_encode(y[i]);
}

/* ---------------------------------------------------------------------------------------------
 * Change points of the encoder over f32 bit patterns.  Over [0x00000000, 0x7F800000] (+0 to +inf)
 * and over [0x80000000, 0xFF800000] (-0 to -inf) the magnitude |y| grows with the pattern, so the
 * magnitude code is non-decreasing and each of codes 1..126 is first reached at one pattern.  This
 * lists every pattern p at which encode(p) differs from encode(p-1), over all 2^32 patterns
 * (including the steps into and out of the two NaN ranges), in ascending order.  A GPU test scans
 * all 2^32 patterns and must find exactly this list, with equal codes at each point.
 * ------------------------------------------------------------------------------------------- */
static uint8_t enc_bits(uint32_t p)
{
    float f;
    memcpy(&f, &p, 4);
    return kv8o_e4m3_encode(f);
}

static int64_t range_changes(uint32_t lo, uint32_t hi, uint32_t *out, int64_t n, int64_t cap)
{
    for (int c = 1; c <= 0x7E; ++c) {
        /* smallest p in [lo, hi] with (enc(p) & 0x7F) >= c */
        uint32_t a = lo, b = hi;
        if ((enc_bits(hi) & 0x7F) < c)
            break;
        while (a < b) {
            uint32_t mid = a + (b - a) / 2;
            if ((enc_bits(mid) & 0x7F) >= c)
                b = mid;
            else
                a = mid + 1;
        }
        if (a > lo && (n == 0 || out[n - 1] != a)) {
            if (n < cap)
                out[n] = a;
            ++n;
        }
    }
    return n;
}

int64_t kv8o_encode_change_points(uint32_t *out, int64_t cap)
{
    lut_init();
    int64_t n = 0;
    n = range_changes(0x00000000u, 0x7F800000u, out, n, cap);
    if (n < cap) out[n] = 0x7F800001u; /* +inf (0x7E) -> first +NaN (0x00) */
    ++n;
    if (n < cap) out[n] = 0x80000000u; /* last +NaN (0x00) -> -0 (0x80) */
    ++n;
    n = range_changes(0x80000000u, 0xFF800000u, out, n, cap);
    if (n < cap) out[n] = 0xFF800001u; /* -inf (0xFE) -> first -NaN (0x00) */
    ++n;
    return n;
}

/* ---------------------------------------------------------------------------------------------
 * Row quantizer ([KV8] first commit, c/kv_fp8.h item: a per-row quantizer guarded against an
 * amax so small that 448/amax overflows; the row format: e4m3 bytes with a per-row f32
 * amax/448 scale).  All arithmetic in f32 with IEEE round-to-nearest:
 *   amax  = max |x_i| over finite elements
 *   scale = amax / 448
 *   amax == 0:           y_i = x_i
 *   inv = 448 / amax finite:  y_i = x_i * inv
 *   inv overflows:       y_i = (x_i * 2^64) * (448 / (amax * 2^64))   (the guard)
 *   byte_i = encode(y_i)
 * ------------------------------------------------------------------------------------------- */
void kv8o_quant_rows_w(const float *x, int64_t n, int width, uint8_t *q, float *scale)
{
    lut_init();
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r) {
        const float *xr = x + r * width;
        uint8_t *qr = q + r * width;
        float amax = 0.0f;
        for (int i = 0; i < width; ++i) {
            float a = fabsf(xr[i]);
            if (isfinite(a) && a > amax)
                amax = a;
        }
        float s = amax / 448.0f;
        scale[r] = s;
        if (amax == 0.0f) {
            for (int i = 0; i < width; ++i)
                qr[i] = kv8o_e4m3_encode(xr[i]);
            continue;
        }
        float inv = 448.0f / amax;
        if (isinf(inv)) {
            const float two64 = 18446744073709551616.0f; /* 2^64 */
            float amax_up = amax * two64;
            float inv_up = 448.0f / amax_up;
            for (int i = 0; i < width; ++i) {
                float xi = xr[i] * two64;
                float yi = xi * inv_up;
                qr[i] = kv8o_e4m3_encode(yi);
            }
        } else {
            for (int i = 0; i < width; ++i) {
                float yi = xr[i] * inv;
                qr[i] = kv8o_e4m3_encode(yi);
            }
        }
    }
}

/* The cache rows: width 576. */
void kv8o_quant_rows(const float *x, int64_t n, uint8_t *q, float *scale)
{
    kv8o_quant_rows_w(x, n, KV8O_D, q, scale);
}

/* Dequantize rows to double: value = table[byte] * scale (exact in double). */
void kv8o_dequant_rows(const uint8_t *q, const float *scale, int64_t n, double *out)
{
    lut_init();
    for (int64_t r = 0; r < n; ++r)
        for (int i = 0; i < KV8O_D; ++i)
            out[r * KV8O_D + i] = g_lut[q[r * KV8O_D + i]] * (double)scale[r];
}

/* ---------------------------------------------------------------------------------------------
 * Absorbed attention of one query head over a list of rows ([KV8] first commit, attention_rows
 * item: the latent row serves as key and as value; the absorb score loop dequantizes inline with the row
 * scale hoisted out of the dot):
 *   score_t = sm_scale * s_t * ( sum_{i<512} q_lat[i] e4m3(Lc8_t[i]) + sum_{j<64} q_rope[j] e4m3(Rc8_t[j]) )
 *   cl[i]   = sum_t softmax(score)_t * s_t * e4m3(Lc8_t[i])
 * in double.  `rows` lists the row indices attended (any order); rows outside [0, T) are skipped
 * and counted in *bad.  With no valid rows the output is 0.
 * ------------------------------------------------------------------------------------------- */
static void attend_rows(const float *q_lat, const float *q_rope, const uint8_t *kv8, const float *scale,
                        int64_t T, const int64_t *rows, int64_t n_rows, double sm_scale, double *score,
                        double *acc /*[512]*/, double *m_out, double *z_out, int64_t *bad)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < n_rows; ++j) {
        int64_t t = rows[j];
        if (t < 0 || t >= T) {
            score[j] = -INFINITY;
            if (bad)
                ++*bad;
            continue;
        }
        const uint8_t *row = kv8 + t * KV8O_D;
        double dot = 0.0;
        for (int i = 0; i < KV8O_KL; ++i)
            dot += (double)q_lat[i] * g_lut[row[i]];
        for (int i = 0; i < KV8O_KR; ++i)
            dot += (double)q_rope[i] * g_lut[row[KV8O_KL + i]];
        score[j] = sm_scale * (double)scale[t] * dot;
        if (score[j] > m)
            m = score[j];
    }
    for (int i = 0; i < KV8O_KL; ++i)
        acc[i] = 0.0;
    double z = 0.0;
    if (m != -INFINITY) {
        for (int64_t j = 0; j < n_rows; ++j) {
            if (score[j] == -INFINITY)
                continue;
            int64_t t = rows[j];
            double p = exp(score[j] - m);
            z += p;
            double w = p * (double)scale[t];
            const uint8_t *row = kv8 + t * KV8O_D;
            for (int i = 0; i < KV8O_KL; ++i)
                acc[i] += w * g_lut[row[i]];
        }
    }
    *m_out = m;
    *z_out = z;
}

/* Dense decode: H heads (q_lat [H][512], q_rope [H][64]) over rows 0..T-1; out [H][512] f32. */
void kv8o_attn_decode(const float *q_lat, const float *q_rope, int H, const uint8_t *kv8, const float *scale,
                      int64_t T, float sm_scale, float *out)
{
    lut_init();
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(T > 0 ? T : 1));
    for (int64_t t = 0; t < T; ++t)
        rows[t] = t;
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < H; ++h) {
        double *score = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double acc[KV8O_KL], m, z;
        attend_rows(q_lat + (int64_t)h * KV8O_KL, q_rope + (int64_t)h * KV8O_KR, kv8, scale, T, rows, T,
                    (double)sm_scale, score, acc, &m, &z, NULL);
        for (int i = 0; i < KV8O_KL; ++i)
            out[(int64_t)h * KV8O_KL + i] = z > 0.0 ? (float)(acc[i] / z) : 0.0f;
        free(score);
    }
    free(rows);
}

/* ---------------------------------------------------------------------------------------------
 * Split-T decode ([KV8] second commit, split-T item: partial online-softmax blocks (cl[K], m, z)
 * plus a log-sum-exp merge).  Partition p covers rows [T*p/P, T*(p+1)/P).  Each partition keeps
 * its own max m_p, sum z_p = sum exp(score - m_p) and unnormalised context cl_p; an empty
 * partition has m_p = -inf, z_p = 0.  The merge: M = max_p m_p; w_p = exp(m_p - M) (0 for an
 * empty partition); Z = sum_p w_p z_p; cl = sum_p w_p cl_p / Z.  Partials are returned in double
 * (cl_part [P][H][512], m_part [P][H], z_part [P][H]) and the merged output in f32.
 * ------------------------------------------------------------------------------------------- */
void kv8o_attn_decode_split(const float *q_lat, const float *q_rope, int H, const uint8_t *kv8, const float *scale,
                            int64_t T, float sm_scale, int P, double *cl_part, double *m_part, double *z_part,
                            float *out)
{
    lut_init();
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(T > 0 ? T : 1));
    for (int64_t t = 0; t < T; ++t)
        rows[t] = t;
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < H; ++h) {
        double *score = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        for (int p = 0; p < P; ++p) {
            int64_t t0 = T * p / P, t1 = T * (p + 1) / P;
            double *acc = cl_part + ((int64_t)p * H + h) * KV8O_KL;
            attend_rows(q_lat + (int64_t)h * KV8O_KL, q_rope + (int64_t)h * KV8O_KR, kv8, scale, T, rows + t0,
                        t1 - t0, (double)sm_scale, score, acc, &m_part[(int64_t)p * H + h],
                        &z_part[(int64_t)p * H + h], NULL);
        }
        double M = -INFINITY;
        for (int p = 0; p < P; ++p)
            if (m_part[(int64_t)p * H + h] > M)
                M = m_part[(int64_t)p * H + h];
        double Z = 0.0, cl[KV8O_KL];
        for (int i = 0; i < KV8O_KL; ++i)
            cl[i] = 0.0;
        for (int p = 0; p < P; ++p) {
            double mp = m_part[(int64_t)p * H + h];
            if (mp == -INFINITY)
                continue; /* empty partition: weight 0, no (-inf) - (-inf) */
            double w = exp(mp - M);
            Z += w * z_part[(int64_t)p * H + h];
            const double *acc = cl_part + ((int64_t)p * H + h) * KV8O_KL;
            for (int i = 0; i < KV8O_KL; ++i)
                cl[i] += w * acc[i];
        }
        for (int i = 0; i < KV8O_KL; ++i)
            out[(int64_t)h * KV8O_KL + i] = Z > 0.0 ? (float)(cl[i] / Z) : 0.0f;
        free(score);
    }
    free(rows);
}

/* ---------------------------------------------------------------------------------------------
 * Selected-row decode ([KV8] second commit, DSA gather item: attend the selected rows, absolute
 * indices, NS <= 4096; a selection means only those rows).  B sequences; sequence b has its own
 * cache of T rows starting at row b*seq_stride_rows of kv8/scale, its own queries
 * (q_lat [B][H][512], q_rope [B][H][64]) and its own index list idx [B][NS] (int32).  Every list
 * entry counts once per occurrence; an index outside [0, T) is skipped and counted in *bad.
 * out [B][H][512].
 * ------------------------------------------------------------------------------------------- */
void kv8o_attn_select(const float *q_lat, const float *q_rope, int B, int H, const uint8_t *kv8, const float *scale,
                      int64_t T, int64_t seq_stride_rows, const int32_t *idx, int NS, float sm_scale, float *out,
                      int64_t *bad)
{
    lut_init();
    int64_t nbad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : nbad)
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        int64_t b = bh / H;
        int64_t *rowp = (int64_t *)malloc(sizeof(int64_t) * (size_t)(NS > 0 ? NS : 1));
        double *score = (double *)malloc(sizeof(double) * (size_t)(NS > 0 ? NS : 1));
        for (int j = 0; j < NS; ++j)
            rowp[j] = idx[b * NS + j];
        double acc[KV8O_KL], m, z;
        int64_t bad_here = 0;
        attend_rows(q_lat + bh * KV8O_KL, q_rope + bh * KV8O_KR, kv8 + b * seq_stride_rows * KV8O_D,
                    scale + b * seq_stride_rows, T, rowp, NS, (double)sm_scale, score, acc, &m, &z, &bad_here);
        if (bh % H == 0)
            nbad += bad_here; /* count each sequence's bad indices once */
        for (int i = 0; i < KV8O_KL; ++i)
            out[bh * KV8O_KL + i] = z > 0.0 ? (float)(acc[i] / z) : 0.0f;
        free(score);
        free(rowp);
    }
    if (bad)
        *bad = nbad;
}

/* ---------------------------------------------------------------------------------------------
 * Causal prefill ([KV8] first/second commit: the batch/prefill absorb path; causal by position).
 * nq queries; query i sits at absolute position pos[i] and attends rows 0..pos[i] (row index =
 * position).  q_lat [nq][H][512], q_rope [nq][H][64]; out [nq][H][512].
 * ------------------------------------------------------------------------------------------- */
void kv8o_attn_prefill(const float *q_lat, const float *q_rope, int nq, int H, const int64_t *pos,
                       const uint8_t *kv8, const float *scale, int64_t T, float sm_scale, float *out)
{
    lut_init();
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(T > 0 ? T : 1));
    for (int64_t t = 0; t < T; ++t)
        rows[t] = t;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t qh = 0; qh < (int64_t)nq * H; ++qh) {
        int64_t i = qh / H;
        int64_t n = pos[i] + 1;
        if (n > T)
            n = T;
        if (n < 0)
            n = 0;
        double *score = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double acc[KV8O_KL], m, z;
        attend_rows(q_lat + qh * KV8O_KL, q_rope + qh * KV8O_KR, kv8, scale, T, rows, n, (double)sm_scale, score,
                    acc, &m, &z, NULL);
        for (int k = 0; k < KV8O_KL; ++k)
            out[qh * KV8O_KL + k] = z > 0.0 ? (float)(acc[k] / z) : 0.0f;
        free(score);
    }
    free(rows);
}

/* ---------------------------------------------------------------------------------------------
 * Absorb projections through kv_b_proj stored as fmt=8 ([FMT8]: raw e4m3 bytes, one f32 scale per
 * 128x128 block, block-row-major, ceil(O/128) x ceil(I/128) scales).  kv_b has O = H*256 rows of
 * I = 512 columns; head h owns rows 256h..256h+127 (W_UK: the no-position key part, qk_nope = 128)
 * and rows 256h+128..256h+255 (W_UV: the value part, v_head = 128).  The dequantized weight is
 *     W[o][i] = e4m3(w8[o][i]) * w_scale[(o/128) * nbc + i/128],   nbc = ceil(I/128) = 4.
 * Every product is widened to double and summed in double; each output is rounded once to f32.
 *
 * Query side (the absorbed query, [KV8] first commit: the latent is the key):
 *     q_lat[s][h][c] = sum_{j<128} q_nope[s][h][j] * W[256h + j][c]          (c < 512)
 * Output side (the context leaves the latent space through the value rows):
 *     out[s][h][v]   = sum_{c<512} W[256h + 128 + v][c] * ctx[s][h][c]        (v < 128)
 * ------------------------------------------------------------------------------------------- */
#define KV8O_NOPE 128
#define KV8O_VH 128
#define KV8O_BLK 128

static double kvb_weight(const uint8_t *w8, const float *w_scale, int64_t o, int i)
{
    const int nbc = (KV8O_KL + KV8O_BLK - 1) / KV8O_BLK;
    return kv8o_e4m3_decode(w8[o * KV8O_KL + i]) * (double)w_scale[(o / KV8O_BLK) * nbc + i / KV8O_BLK];
}

void kv8o_q_absorb(const float *q_nope, int S, int H, const uint8_t *w8, const float *w_scale, float *q_lat)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t sh = 0; sh < (int64_t)S * H; ++sh) {
        const int h = (int)(sh % H);
        const float *q = q_nope + sh * KV8O_NOPE;
        for (int c = 0; c < KV8O_KL; ++c) {
            double acc = 0.0;
            for (int j = 0; j < KV8O_NOPE; ++j)
                acc += (double)q[j] * kvb_weight(w8, w_scale, (int64_t)h * (KV8O_NOPE + KV8O_VH) + j, c);
            q_lat[sh * KV8O_KL + c] = (float)acc;
        }
    }
}

void kv8o_out_project(const float *ctx, int S, int H, const uint8_t *w8, const float *w_scale, float *out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t sh = 0; sh < (int64_t)S * H; ++sh) {
        const int h = (int)(sh % H);
        const float *x = ctx + sh * KV8O_KL;
        for (int v = 0; v < KV8O_VH; ++v) {
            const int64_t o = (int64_t)h * (KV8O_NOPE + KV8O_VH) + KV8O_NOPE + v;
            double acc = 0.0;
            for (int c = 0; c < KV8O_KL; ++c)
                acc += kvb_weight(w8, w_scale, o, c) * (double)x[c];
            out[sh * KV8O_VH + v] = (float)acc;
        }
    }
}

/* ---------------------------------------------------------------------------------------------
 * DSA lightning-indexer score and top-k ([B1] page, the indexer_fp8_score_topk commit: the index
 * query (64 heads x 128) quantized from bf16 to e4m3, the index keys read as e4m3; dequantize with
 * q_scale * k_scale, ReLU, weighted sum over the heads, then top-k).  Our reading of the formula:
 *     I[b][t] = sum_h w[b][h] * max(0, q_scale[b][h] * k_scale[t'] * sum_i e4m3(q8[b][h][i]) e4m3(k8[t'][i]))
 * with t' = b * seq_stride_rows + t the key row of item b's position t, and the scales the per-row
 * amax/448 of the row quantizer above (index keys: rows of width DI; index query: one row per head).
 * Products of two e4m3 values and their sums over DI <= 512 terms are exact in double.
 * ------------------------------------------------------------------------------------------- */
void kv8o_index_scores(const uint8_t *q8, const float *q_scale, const float *w, int B, int HI, int DI,
                       const uint8_t *k8, const float *k_scale, int64_t T, int64_t seq_stride_rows, double *scores)
{
    lut_init();
#pragma omp parallel for schedule(static)
    for (int64_t bt = 0; bt < (int64_t)B * T; ++bt) {
        const int b = (int)(bt / T);
        const int64_t row = (int64_t)b * seq_stride_rows + (bt - (int64_t)b * T);
        const uint8_t *kr = k8 + row * DI;
        double acc = 0.0;
        for (int h = 0; h < HI; ++h) {
            const uint8_t *qr = q8 + ((int64_t)b * HI + h) * DI;
            double dot = 0.0;
            for (int i = 0; i < DI; ++i)
                dot += g_lut[qr[i]] * g_lut[kr[i]];
            const double v = (double)q_scale[b * HI + h] * (double)k_scale[row] * dot;
            if (v > 0.0)
                acc += (double)w[b * HI + h] * v;
        }
        scores[bt] = acc;
    }
}

/* The k largest of n scores, the smaller index first among equal scores; indices returned in
 * ascending order (the order the selected-row attention takes them in). */
static const double *g_topk_scores;
static int topk_cmp(const void *a, const void *b)
{
    const int64_t i = *(const int64_t *)a, j = *(const int64_t *)b;
    const double si = g_topk_scores[i], sj = g_topk_scores[j];
    if (si != sj)
        return si > sj ? -1 : 1;
    return i < j ? -1 : (i > j ? 1 : 0);
}
static int idx_cmp(const void *a, const void *b)
{
    const int32_t i = *(const int32_t *)a, j = *(const int32_t *)b;
    return i < j ? -1 : (i > j ? 1 : 0);
}
void kv8o_topk(const double *scores, int64_t n, int k, int32_t *idx)
{
    int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i)
        order[i] = i;
    g_topk_scores = scores;  /* single-threaded: qsort has no context argument in C11 */
    qsort(order, (size_t)n, sizeof(int64_t), topk_cmp);
    const int kk = (int64_t)k < n ? k : (int)n;
    for (int i = 0; i < kk; ++i)
        idx[i] = (int32_t)order[i];
    qsort(idx, (size_t)kk, sizeof(int32_t), idx_cmp);
    free(order);
}

/* ---------------------------------------------------------------------------------------------
 * Mixed-precision cache decode ([B1] page, "B1 Mixed FP8/BF16 FMHA first pass": each KV row keeps its
 * no-position part (448) as e4m3 bytes with a per-row f32 scale and its RoPE part (64) as bf16; the
 * query's no-position part is quantized from bf16 to e4m3 just before the attention; head width 512).
 * Our reading (K and V are the same 512-wide row):
 *   q8 [H][448] u8 and q_scale [H]: the row quantizer above applied to each head's q_nope;
 *   score[h][t] = sm_scale * ( q_scale[h] * k_scale[t] * sum_i e4m3(q8[h][i]) e4m3(k8[t][i])
 *                              + sum_j q_rope[h][j] * k_rope[t][j] )
 *   value_t     = [ k_scale[t] * e4m3(k8[t][i]) for i < 448 ,  k_rope[t][j] for j < 64 ]
 *   out[h]      = sum_t softmax_t(score[h][t]) * value_t             (double; rounded once to f32)
 * q_rope and k_rope are passed as f32 holding the bf16 values.
 * ------------------------------------------------------------------------------------------- */
#define KV8O_MX_NOPE 448
#define KV8O_MX_ROPE 64
#define KV8O_MX_D (KV8O_MX_NOPE + KV8O_MX_ROPE)

void kv8o_attn_mixed_decode(const uint8_t *q8, const float *q_scale, const float *q_rope, int H, const uint8_t *k8,
                            const float *k_scale, const float *k_rope, int64_t T, float sm_scale, float *out)
{
    lut_init();
#pragma omp parallel for schedule(dynamic, 1)
    for (int h = 0; h < H; ++h) {
        double *score = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
        double m = -INFINITY;
        for (int64_t t = 0; t < T; ++t) {
            double dn = 0.0, dr = 0.0;
            for (int i = 0; i < KV8O_MX_NOPE; ++i)
                dn += g_lut[q8[(int64_t)h * KV8O_MX_NOPE + i]] * g_lut[k8[t * KV8O_MX_NOPE + i]];
            for (int j = 0; j < KV8O_MX_ROPE; ++j)
                dr += (double)q_rope[(int64_t)h * KV8O_MX_ROPE + j] * (double)k_rope[t * KV8O_MX_ROPE + j];
            score[t] = (double)sm_scale * ((double)q_scale[h] * (double)k_scale[t] * dn + dr);
            if (score[t] > m)
                m = score[t];
        }
        double acc[KV8O_MX_D], z = 0.0;
        for (int i = 0; i < KV8O_MX_D; ++i)
            acc[i] = 0.0;
        for (int64_t t = 0; t < T; ++t) {
            const double p = exp(score[t] - m);
            z += p;
            const double ks = (double)k_scale[t];
            for (int i = 0; i < KV8O_MX_NOPE; ++i)
                acc[i] += p * ks * g_lut[k8[t * KV8O_MX_NOPE + i]];
            for (int j = 0; j < KV8O_MX_ROPE; ++j)
                acc[KV8O_MX_NOPE + j] += p * (double)k_rope[t * KV8O_MX_ROPE + j];
        }
        for (int i = 0; i < KV8O_MX_D; ++i)
            out[(int64_t)h * KV8O_MX_D + i] = z > 0.0 ? (float)(acc[i] / z) : 0.0f;
        free(score);
    }
}

int kv8o_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void kv8o_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
