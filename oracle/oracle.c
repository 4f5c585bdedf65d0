/*
 * oracle.c -- plain, slow CPU reference for the W4A16 skinny GEMM and the
 * int4 lm_head greedy verify.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it follows (page titles and sections of the source pages):
 *  - "qwen-warp and llamAmpere: two RTX 3090 engines for Qwen3.8, and what each one calls the same answer", section "qwen-warp: keep the activations in
 *    bf16": weights are uint32 words of eight 4-bit nibbles along K with one
 *    bf16 scale per 128 columns of a row; a nibble n stands for the signed
 *    level n - 8; the group scale multiplies the fp32 sum of the group, after
 *    that group's accumulation.
 *  - same page, table "What one cycle reads from VRAM": the int4 lm_head is
 *    248,320 rows of 5,120 columns.
 *  - same page, section "What each one calls the same answer": greedy
 *    acceptance is an argmax equality over the verify rows.
 *  - "swift-qwen3.8-rtx3090", section "Body, heads and drafter": the model
 *    keeps drafted tokens up to the first one it disagrees with.
 *  - "OpenJet Engine: CUDA LLM inference for Qwen3.8-27B", sections "How it works" and "How it gets its speed":
 *    lm_head and verification run over T = 1 + n_draft rows; a restricted
 *    draft head scores a fixed id list.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - nibble i of word w holds column k = 8w + i, in bits 4i..4i+3;
 *  - a weight row is one output row (N or V), K contiguous;
 *  - the zero point is the constant 8 (symmetric);
 *  - logits stay fp32 (never rounded to bf16) before the argmax;
 *  - argmax ties go to the lowest token id (over a vocab_map: lowest id, not
 *    lowest map position);
 *  - row 0 of a verify block is the last committed token; draft i is
 *    compared with the argmax of row i; accept_len is the first mismatch
 *    index (n_draft if none) and the bonus token is the argmax of row
 *    accept_len.
 *
 * Arithmetic: every product level * x is exact in fp32 (a 4-bit integer
 * times an 8-bit significand).  Within a group the products are summed in
 * fp32 in ascending k; the group sum is multiplied by float(scale) (one
 * rounding) and added to the row accumulator (one rounding), groups in
 * ascending order.  Build with -ffp-contract=off so no fused multiply-add
 * changes that.  An fp64 twin of the same sum measures the fp32 rounding.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#include <omp.h>

#define OR_OK 0
#define OR_EINVAL (-1)

static float bf16_to_float(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE round-to-nearest-even from fp32 to bf16 (finite inputs). */
static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {          /* inf / nan: keep class */
        return (uint16_t)((u >> 16) | ((u & 0xffffu) ? 0x40u : 0u));
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* The signed level of column k of one packed weight row. */
static int level_at(const uint32_t *wrow, int k)
{
    uint32_t word = wrow[k / 8];
    uint32_t nib = (word >> (4 * (k % 8))) & 0xfu;
    return (int)nib - 8;
}

/*
 * Dot products of one weight row with T activation rows.
 * out32[t] (fp32 as specified above), out64[t] (fp64 twin); either may be
 * NULL.  lv is caller scratch of K ints.
 */
static void row_dot(const uint16_t *x, const uint32_t *wrow, const uint16_t *srow,
                    int T, int K, int *lv, float *acc32, double *acc64,
                    float *gacc32, double *gacc64)
{
    int G = K / 128;
    for (int k = 0; k < K; ++k)
        lv[k] = level_at(wrow, k);
    for (int t = 0; t < T; ++t) {
        acc32[t] = 0.0f;
        acc64[t] = 0.0;
    }
    for (int g = 0; g < G; ++g) {
        for (int t = 0; t < T; ++t) {
            gacc32[t] = 0.0f;
            gacc64[t] = 0.0;
        }
        for (int k = 128 * g; k < 128 * g + 128; ++k) {
            float w = (float)lv[k];
            for (int t = 0; t < T; ++t) {
                float xv = bf16_to_float(x[(size_t)t * K + k]);
                float p = w * xv;                 /* exact */
                gacc32[t] = gacc32[t] + p;
                gacc64[t] = gacc64[t] + (double)w * (double)xv;
            }
        }
        float s = bf16_to_float(srow[g]);
        for (int t = 0; t < T; ++t) {
            float sp = s * gacc32[t];
            acc32[t] = acc32[t] + sp;
            acc64[t] = acc64[t] + (double)s * gacc64[t];
        }
    }
}

/*
 * y[t][n] = sum_g scale[n][g] * sum_{k in g} (q(n,k) - 8) * x[t][k]
 * x: [T][K] bf16 bits; Wq: [N][K/8]; scales: [N][K/128] bf16 bits.
 * Outputs (any may be NULL): y32 [T][N] fp32, y64 [T][N] fp64,
 * ybf [T][N] bf16 bits = round-to-nearest-even(y32).
 */
int or_w4a16_gemm(const uint16_t *x, const uint32_t *Wq, const uint16_t *scales,
                  int T, int K, int N, float *y32, double *y64, uint16_t *ybf)
{
    if (!x || !Wq || !scales || T < 1 || K < 128 || K % 128 || N < 1)
        return OR_EINVAL;
    int G = K / 128;
    int bad = 0;
#pragma omp parallel
    {
        int *lv = (int *)malloc(sizeof(int) * (size_t)K);
        float *a32 = (float *)malloc(sizeof(float) * (size_t)T * 2);
        double *a64 = (double *)malloc(sizeof(double) * (size_t)T * 2);
        int ok = lv && a32 && a64;
        if (!ok) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int n = 0; n < N; ++n) {
            if (!ok)
                continue;
            row_dot(x, Wq + (size_t)n * (K / 8), scales + (size_t)n * G, T, K, lv,
                    a32, a64, a32 + T, a64 + T);
            for (int t = 0; t < T; ++t) {
                size_t o = (size_t)t * N + n;
                if (y32) y32[o] = a32[t];
                if (y64) y64[o] = a64[t];
                if (ybf) ybf[o] = float_to_bf16_rne(a32[t]);
            }
        }
        free(lv);
        free(a32);
        free(a64);
    }
    return bad ? OR_EINVAL : OR_OK;
}

/*
 * lm_head logits over a row list: logits[t][j] = dot(row rows[j], x[t]),
 * fp32 as in or_w4a16_gemm and never rounded to bf16.  rows == NULL means
 * rows[j] = j for j < n_rows.  Rows outside [0, V) are an error.
 */
int or_lmhead_logits(const uint16_t *x, const uint32_t *Wq, const uint16_t *scales,
                     int K, int T, const int32_t *rows, int n_rows, int V,
                     float *logits32, double *logits64)
{
    if (!x || !Wq || !scales || T < 1 || K < 128 || K % 128 || n_rows < 1 || V < 1)
        return OR_EINVAL;
    if (!rows && n_rows > V)
        return OR_EINVAL;
    for (int j = 0; rows && j < n_rows; ++j)
        if (rows[j] < 0 || rows[j] >= V)
            return OR_EINVAL;
    int G = K / 128;
    int bad = 0;
#pragma omp parallel
    {
        int *lv = (int *)malloc(sizeof(int) * (size_t)K);
        float *a32 = (float *)malloc(sizeof(float) * (size_t)T * 2);
        double *a64 = (double *)malloc(sizeof(double) * (size_t)T * 2);
        int ok = lv && a32 && a64;
        if (!ok) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int j = 0; j < n_rows; ++j) {
            if (!ok)
                continue;
            size_t v = rows ? (size_t)rows[j] : (size_t)j;
            row_dot(x, Wq + v * (K / 8), scales + v * G, T, K, lv, a32, a64,
                    a32 + T, a64 + T);
            for (int t = 0; t < T; ++t) {
                size_t o = (size_t)t * n_rows + j;
                if (logits32) logits32[o] = a32[t];
                if (logits64) logits64[o] = a64[t];
            }
        }
        free(lv);
        free(a32);
        free(a64);
    }
    return bad ? OR_EINVAL : OR_OK;
}

/*
 * bf16 lm_head logits over a row list: logits[t][j] = sum_k
 * float(Wbf[rows[j]][k]) * float(x[t][k]), each product exact in fp32 (two
 * 8-bit significands), summed in fp32 in ascending k.  The head the
 * quantized lm_head's candidates are rescored with (page "qwen-warp and
 * llamAmpere: two RTX 3090 engines for Qwen3.8, and what each one calls the
 * same answer", section "What each one calls the same answer"; table "What
 * one cycle reads from VRAM": 16 to 64 candidates).  rows == NULL means
 * rows[j] = j.
 */
int or_bf16_logits(const uint16_t *x, const uint16_t *Wbf, int K, int T, const int32_t *rows,
                   int n_rows, int V, float *logits32)
{
    if (!x || !Wbf || !logits32 || T < 1 || K < 1 || n_rows < 1 || V < 1)
        return OR_EINVAL;
    if (!rows && n_rows > V)
        return OR_EINVAL;
    for (int j = 0; rows && j < n_rows; ++j)
        if (rows[j] < 0 || rows[j] >= V)
            return OR_EINVAL;
#pragma omp parallel for schedule(static)
    for (int j = 0; j < n_rows; ++j) {
        size_t v = rows ? (size_t)rows[j] : (size_t)j;
        const uint16_t *w = Wbf + v * (size_t)K;
        for (int t = 0; t < T; ++t) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                float p = bf16_to_float(w[k]) * bf16_to_float(x[(size_t)t * K + k]);   /* exact */
                acc = acc + p;
            }
            logits32[(size_t)t * n_rows + j] = acc;
        }
    }
    return OR_OK;
}

/*
 * Row-wise argmax of logits[T][n] with the lowest token id winning ties.
 * ids[j] is the token id of column j (NULL: ids[j] = j).  Also returns the
 * best value, the runner-up value over the other columns (-INFINITY when
 * n == 1) and the margin best - runner_up.  Logits must be finite.
 */
int or_argmax(const float *logits, int T, int n, const int32_t *ids,
              int32_t *a, float *best, float *second)
{
    if (!logits || T < 1 || n < 1 || !a)
        return OR_EINVAL;
    for (int t = 0; t < T; ++t) {
        const float *row = logits + (size_t)t * n;
        int bj = -1;
        for (int j = 0; j < n; ++j) {
            if (!isfinite(row[j]))
                return OR_EINVAL;
            if (bj < 0 || row[j] > row[bj])
                bj = j;
            else if (row[j] == row[bj]) {
                int32_t idj = ids ? ids[j] : j;
                int32_t idb = ids ? ids[bj] : bj;
                if (idj < idb)
                    bj = j;
            }
        }
        float sec = -INFINITY;
        for (int j = 0; j < n; ++j)
            if (j != bj && row[j] > sec)
                sec = row[j];
        a[t] = ids ? ids[bj] : bj;
        if (best) best[t] = row[bj];
        if (second) second[t] = sec;
    }
    return OR_OK;
}

/*
 * Greedy verification of one block of 1 + n_draft rows.
 * a: argmax token of each row (n_draft + 1 entries); drafts: n_draft ids.
 * accept_len = first i with drafts[i] != a[i], or n_draft if none;
 * next_token = a[accept_len].
 */
int or_verify(const int32_t *a, const int32_t *drafts, int n_draft,
              int32_t *accept_len, int32_t *next_token)
{
    if (!a || n_draft < 0 || (n_draft > 0 && !drafts) || !accept_len || !next_token)
        return OR_EINVAL;
    int i = 0;
    while (i < n_draft && drafts[i] == a[i])
        ++i;
    *accept_len = i;
    *next_token = a[i];
    return OR_OK;
}

/* Number of threads an OpenMP region of this library uses. */
int or_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
}

/* Set the number of threads later OpenMP regions of this library use
   (n >= 1); used to time the oracle on one core as well as on all. */
void or_set_num_threads(int n)
{
    if (n >= 1)
        omp_set_num_threads(n);
}
