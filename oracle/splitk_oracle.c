/*
 * CPU oracle for the split-K BF16 decode GEMM.  TEST INFRASTRUCTURE ONLY:
 * the tests, the package's smoke check and the benchmark's CPU-baseline leg
 * load this file's library; the product path never does.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it computes (plain definition, float64 throughout):
 *
 *     C[l][m][n] = RNE_bf16( sum_{k<K} f64(A[l][n][k]) * f64(B[l][m][k]) )
 *
 *   A[L][N][K]  bf16 weights, K contiguous ("A (M, K, L) K-major" in kernel
 *               terms, where kernel-M carries the public N),
 *   B[L][M][K]  bf16 token activations, K contiguous,
 *   C[L][M][N]  bf16 output, N contiguous.
 *
 * Sources (the vLLM "splitk" API page, module
 * vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.gemm.splitk):
 *   - module docstring: each cluster rank accumulates an exact K slice in
 *     FP32, rank 0 reduces, casts and stores once; kernel-M carries public N
 *     and kernel-N public M (the swapped operand roles);
 *   - SplitKGemm.kernel docstring: A and B are K-major, C has the kernel-M
 *     (public N) mode contiguous;
 *   - SplitKGemm.epilog_warp: the FP32 sum is converted to the C dtype once.
 * The split of K and its FP32 rounding are implementation detail of the GPU
 * path; the oracle sums exactly enough (float64) that its only rounding that
 * matters is the single final one.
 *
 * BF16 bit rules (the DeepSeek-V4.1 AMD "mono" ops page, bf_lo / bf_hi, and
 * the Muse Spark AMD dev page, bf16_pair): a bf16 value is the high 16 bits
 * of an IEEE binary32, so widening is a 16-bit left shift; narrowing rounds to
 * nearest, ties to even.  Readings where the pages are silent: NaN maps to the
 * canonical quiet NaN 0x7FC0 (sign kept), overflow maps to +-Inf, subnormals
 * are kept (never flushed).
 *
 * The A16W4 functions at the end (4-bit weights with 8-bit power-of-two
 * scales, bf16 activations) follow the Muse Spark AMD dev page's e8m0_f32
 * and fp4x8_bf16; see their block comment.
 *
 * Every function here is pinned by tests/test_oracle_pins.py against values
 * fixed independently of this file (exact rational arithmetic, closed forms,
 * library conversions).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bits -> float64.  Exact: bf16 is the top half of a binary32. */
double oracle_bf16_to_f64(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * float64 -> bf16 bits, one rounding to nearest with ties to even.
 *
 * bf16 keeps 8 significant bits (1 implicit + 7 stored), exponent range of
 * binary32: normal numbers down to 2^-126, subnormals spaced 2^-133, largest
 * finite (2 - 2^-7) * 2^127.  The definition used: let q be the spacing of
 * bf16 numbers in the binade of |x| (2^(e-8) for |x| in [2^(e-1), 2^e), but
 * never below the subnormal spacing 2^-133).  Then |x|/q is exact (a power of
 * two scaling), rint() rounds it to the nearest integer with ties to even in
 * the default rounding mode, and the rounded magnitude is that integer times
 * q.  Results at or beyond 2^128 overflow to infinity.
 */
uint16_t oracle_f64_to_bf16(double x)
{
    if (isnan(x)) {
        return (uint16_t)(signbit(x) ? 0xFFC0u : 0x7FC0u);
    }
    uint16_t sign = (uint16_t)(signbit(x) ? 0x8000u : 0u);
    double ax = fabs(x);
    if (isinf(ax)) {
        return (uint16_t)(sign | 0x7F80u);
    }
    if (ax == 0.0) {
        return sign;
    }
    int e;
    (void)frexp(ax, &e);            /* ax = f * 2^e, f in [0.5, 1) */
    int qexp = e - 8;               /* spacing of 8-significant-bit numbers */
    if (qexp < -133) {
        qexp = -133;                /* subnormal spacing of bf16 */
    }
    double n = rint(ldexp(ax, -qexp));  /* exact scaling, then RNE */
    double r = ldexp(n, qexp);          /* exact: n < 2^9 */
    if (r >= 0x1p128) {
        return (uint16_t)(sign | 0x7F80u);
    }
    /* r is a bf16 value, hence exactly a binary32 whose low 16 bits are 0. */
    float rf = (float)r;
    uint32_t bits;
    memcpy(&bits, &rf, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* The float64 dot product behind one output element (before rounding). */
double oracle_dot_f64(const uint16_t *A, const uint16_t *B,
                      int64_t M, int64_t N, int64_t K,
                      int64_t l, int64_t m, int64_t n)
{
    const uint16_t *arow = A + (l * N + n) * K;
    const uint16_t *brow = B + (l * M + m) * K;
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        s += oracle_bf16_to_f64(arow[k]) * oracle_bf16_to_f64(brow[k]);
    }
    return s;
}

/* One output element, rounded once to bf16. */
uint16_t oracle_element(const uint16_t *A, const uint16_t *B,
                        int64_t M, int64_t N, int64_t K,
                        int64_t l, int64_t m, int64_t n)
{
    return oracle_f64_to_bf16(oracle_dot_f64(A, B, M, N, K, l, m, n));
}

/* Selected output elements: idx[i] is the flat index l*M*N + m*N + n. */
void oracle_elements(const uint16_t *A, const uint16_t *B, uint16_t *out,
                     int64_t M, int64_t N, int64_t K, int64_t L,
                     const int64_t *idx, int64_t count)
{
    (void)L;
    for (int64_t i = 0; i < count; ++i) {
        int64_t f = idx[i];
        int64_t l = f / (M * N);
        int64_t m = (f / N) % M;
        int64_t n = f % N;
        out[i] = oracle_element(A, B, M, N, K, l, m, n);
    }
}

/* The whole GEMM, one thread. */
void oracle_gemm(const uint16_t *A, const uint16_t *B, uint16_t *C,
                 int64_t M, int64_t N, int64_t K, int64_t L)
{
    for (int64_t l = 0; l < L; ++l)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n)
                C[(l * M + m) * N + n] = oracle_element(A, B, M, N, K, l, m, n);
}

/*
 * The same GEMM with the output elements divided among host threads.  Each
 * element is still computed by oracle_element alone, so the result is
 * identical to oracle_gemm for any thread count.
 */
struct oracle_job {
    const uint16_t *A, *B;
    uint16_t *C;
    int64_t M, N, K, L;
    int64_t begin, end;  /* flat output range */
};

static void *oracle_worker(void *arg)
{
    struct oracle_job *j = (struct oracle_job *)arg;
    for (int64_t f = j->begin; f < j->end; ++f) {
        int64_t l = f / (j->M * j->N);
        int64_t m = (f / j->N) % j->M;
        int64_t n = f % j->N;
        j->C[f] = oracle_element(j->A, j->B, j->M, j->N, j->K, l, m, n);
    }
    return NULL;
}

int oracle_gemm_threaded(const uint16_t *A, const uint16_t *B, uint16_t *C,
                         int64_t M, int64_t N, int64_t K, int64_t L,
                         int threads)
{
    int64_t total = L * M * N;
    if (threads < 1) threads = 1;
    if (threads == 1 || total < threads) {
        oracle_gemm(A, B, C, M, N, K, L);
        return 1;
    }
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    int *live = (int *)calloc((size_t)threads, sizeof(int));
    struct oracle_job *jobs =
        (struct oracle_job *)calloc((size_t)threads, sizeof(struct oracle_job));
    if (!tid || !live || !jobs) {
        free(tid);
        free(live);
        free(jobs);
        oracle_gemm(A, B, C, M, N, K, L);
        return 1;
    }
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        jobs[t] = (struct oracle_job){A, B, C, M, N, K, L,
                                      total * t / threads,
                                      total * (t + 1) / threads};
        if (pthread_create(&tid[t], NULL, oracle_worker, &jobs[t]) == 0) {
            live[t] = 1;
            ++started;
        } else {
            oracle_worker(&jobs[t]);  /* run it here if no thread is available */
        }
    }
    for (int t = 0; t < threads; ++t) {
        if (live[t]) pthread_join(tid[t], NULL);
    }
    free(tid);
    free(live);
    free(jobs);
    return started > 0 ? started : 1;
}

/*
 * GEMM with a per-output-feature bias (the bias argument of SplitKGemm's
 * launcher on the vLLM "splitk" page, unused there):
 *     C[l][m][n] = RNE_bf16( sum_k f64(A[l][n][k]) * f64(B[l][m][k]) + f64(bias[l][n]) )
 * bias is [L][N] bf16; the sum and the bias are added in float64 and rounded
 * once.
 */
void oracle_gemm_bias(const uint16_t *A, const uint16_t *B, const uint16_t *bias,
                      uint16_t *C, int64_t M, int64_t N, int64_t K, int64_t L)
{
    for (int64_t l = 0; l < L; ++l)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n)
                C[(l * M + m) * N + n] = oracle_f64_to_bf16(
                    oracle_dot_f64(A, B, M, N, K, l, m, n) +
                    oracle_bf16_to_f64(bias[l * N + n]));
}

/* ------------------------------------------------------------------------
 * A16W4: 4-bit weights, bf16 activations (the Muse Spark AMD dev page,
 * e8m0_f32 and fp4x8_bf16, "the aiter Muse a16w4 decode").
 *
 *   E2M1 code c (4 bits): sign = bit 3, exponent e = bits 2..1 (bias 1),
 *   mantissa m = bit 0.  e = 0: (-1)^s * m * 2^-1;  e >= 1:
 *   (-1)^s * (1 + m/2) * 2^(e-1).  Magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 *   E8M0 code x: the power of two 2^(x - 127) (the page's domain is 1..254,
 *   where this is the f32 with exponent field x; 255 is not a number).
 *
 *   Weights: A_q[l][n][k/2] bytes, element k in the low nibble when k is
 *   even ("low nibble first"); scales A_s[l][n][k/32], one code per 32
 *   consecutive k of a weight row (the OCP microscaling block -- a reading:
 *   the page decodes one dword of 8 codes with one scale but does not print
 *   the block length).
 *
 *   C[l][m][n] = RNE_bf16( sum_k w(l,n,k) * f64(B[l][m][k]) ),
 *   w(l,n,k) = e2m1(code of k) * e8m0(scale of k / 32), exact in float64.
 * ------------------------------------------------------------------------ */
double oracle_e2m1_to_f64(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = e == 0 ? 0.5 * (double)m : (1.0 + 0.5 * (double)m) * ldexp(1.0, (int)e - 1);
    return s ? -mag : mag;
}

double oracle_e8m0_to_f64(unsigned code)
{
    code &= 0xFFu;
    if (code == 255u) return NAN;
    return ldexp(1.0, (int)code - 127);
}

/* The dequantized weight w(l, n, k). */
double oracle_w4_weight(const uint8_t *Aq, const uint8_t *As, int64_t N, int64_t K,
                        int64_t l, int64_t n, int64_t k)
{
    const uint8_t byte = Aq[(l * N + n) * (K / 2) + k / 2];
    const unsigned code = (k % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);
    const uint8_t scale = As[(l * N + n) * (K / 32) + k / 32];
    return oracle_e2m1_to_f64(code) * oracle_e8m0_to_f64(scale);
}

void oracle_w4_dequant(const uint8_t *Aq, const uint8_t *As, double *W, int64_t N, int64_t K, int64_t L)
{
    for (int64_t l = 0; l < L; ++l)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t k = 0; k < K; ++k)
                W[(l * N + n) * K + k] = oracle_w4_weight(Aq, As, N, K, l, n, k);
}

double oracle_w4_dot_f64(const uint8_t *Aq, const uint8_t *As, const uint16_t *B, int64_t M, int64_t N,
                         int64_t K, int64_t l, int64_t m, int64_t n)
{
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
        s += oracle_w4_weight(Aq, As, N, K, l, n, k) * oracle_bf16_to_f64(B[(l * M + m) * K + k]);
    return s;
}

void oracle_gemm_w4a16(const uint8_t *Aq, const uint8_t *As, const uint16_t *B, uint16_t *C,
                       int64_t M, int64_t N, int64_t K, int64_t L)
{
    for (int64_t l = 0; l < L; ++l)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n)
                C[(l * M + m) * N + n] = oracle_f64_to_bf16(oracle_w4_dot_f64(Aq, As, B, M, N, K, l, m, n));
}

void oracle_w4_elements(const uint8_t *Aq, const uint8_t *As, const uint16_t *B, uint16_t *out, int64_t M,
                        int64_t N, int64_t K, int64_t L, const int64_t *flat, int64_t count)
{
    (void)L;
    for (int64_t i = 0; i < count; ++i) {
        const int64_t f = flat[i];
        const int64_t l = f / (M * N), m = (f / N) % M, n = f % N;
        out[i] = oracle_f64_to_bf16(oracle_w4_dot_f64(Aq, As, B, M, N, K, l, m, n));
    }
}

/* ------------------------------------------------------------------------
 * A16W8: 8-bit E4M3 weights with E8M0 scales per 32 k, bf16 activations.
 *
 *   E4M3 (the DeepSeek-V4.1 AMD mono ops page's fp8_pack4 packs four f32 into
 *   "four E4M3 bytes, RNE"; the bit layout is the OCP 8-bit floating-point
 *   E4M3 definition, a reading: the page names the format, not its fields):
 *   sign bit 7, exponent bits 6..3 with bias 7, mantissa bits 2..0.
 *   Exponent 0 is subnormal, m * 2^-9; exponent field 15 with mantissa 7 is
 *   not a number (no infinities; largest finite 448).
 *
 *   Weights: A_q[l][n][k] bytes, one code per k; scales A_s[l][n][k/32], one
 *   E8M0 code per 32 consecutive k of a weight row, as for the 4-bit weights
 *   above (the OCP microscaling block -- a reading: the pages give no block
 *   scale for 8-bit weights; this is the plainest one that matches the 4-bit
 *   path).
 *
 *   C[l][m][n] = RNE_bf16( sum_k w(l,n,k) * f64(B[l][m][k]) ),
 *   w(l,n,k) = e4m3(A_q[l][n][k]) * e8m0(A_s[l][n][k/32]), exact in float64.
 * ------------------------------------------------------------------------ */
double oracle_e4m3_to_f64(unsigned code)
{
    code &= 0xFFu;
    const unsigned s = code >> 7, e = (code >> 3) & 15u, m = code & 7u;
    if (e == 15u && m == 7u) return NAN;
    double mag = e == 0 ? (double)m * ldexp(1.0, -9) : (1.0 + (double)m / 8.0) * ldexp(1.0, (int)e - 7);
    return s ? -mag : mag;
}

/* The dequantized 8-bit weight w(l, n, k). */
double oracle_w8_weight(const uint8_t *Aq, const uint8_t *As, int64_t N, int64_t K,
                        int64_t l, int64_t n, int64_t k)
{
    const uint8_t code = Aq[(l * N + n) * K + k];
    const uint8_t scale = As[(l * N + n) * (K / 32) + k / 32];
    return oracle_e4m3_to_f64(code) * oracle_e8m0_to_f64(scale);
}

void oracle_w8_dequant(const uint8_t *Aq, const uint8_t *As, double *W, int64_t N, int64_t K, int64_t L)
{
    for (int64_t l = 0; l < L; ++l)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t k = 0; k < K; ++k)
                W[(l * N + n) * K + k] = oracle_w8_weight(Aq, As, N, K, l, n, k);
}

void oracle_gemm_w8a16(const uint8_t *Aq, const uint8_t *As, const uint16_t *B, uint16_t *C,
                       int64_t M, int64_t N, int64_t K, int64_t L)
{
    for (int64_t l = 0; l < L; ++l)
        for (int64_t m = 0; m < M; ++m)
            for (int64_t n = 0; n < N; ++n) {
                double s = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    s += oracle_w8_weight(Aq, As, N, K, l, n, k) * oracle_bf16_to_f64(B[(l * M + m) * K + k]);
                C[(l * M + m) * N + n] = oracle_f64_to_bf16(s);
            }
}
