/*
 * oracle.c -- plain, slow CPU oracle for the rotated-INT8 linear / FFN path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark use it (through oracle/oracle.py).  It shares no code,
 * header, table or constant with the CUDA path.
 *
 * Source of every formula: the PyPI page "xpu-kernels 0.2.0"
 * (pypi.org/project/xpu-kernels/0.2.0), sections "Use from Python",
 * "The backward: dL/dx, weight-only", "API" and "Algorithm: fused ConvRot
 * rotation".  Where the page leaves a step open, the reading taken is
 * named at the function (R-n tags; the same list is kept in the design
 * notes of the repository).
 *
 * Arithmetic policy (no blocking, no fusion, no reordering beyond the
 * definitions):
 *   - rotation: explicit integer Hadamard factors, sums in fp64, one
 *     rounding to fp32 at the end;
 *   - quantizer: fp32, IEEE division, round-half-even, clamp +-127;
 *   - integer GEMM: int64, with a check that every result fits in int32;
 *   - dequant epilogue: fp32 multiply then fmaf, then bf16 RNE.
 * Compile with -ffp-contract=off and without -ffast-math.
 *
 * Parallelism: independent rows are spread over OpenMP threads.  Each row
 * is computed exactly as the serial definition states.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32 (bfloat16: the upper 16 bits of an IEEE binary32).     */
/* ------------------------------------------------------------------ */

static float bf16_bits_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round-to-nearest-even from binary32 to bfloat16; NaN -> quiet NaN. */
static uint16_t f32_to_bf16_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

void orc_bf16_to_f32(const uint16_t *h, float *f, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) f[i] = bf16_bits_to_f32(h[i]);
}

void orc_f32_to_bf16(const float *f, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = f32_to_bf16_bits(f[i]);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* Hadamard factors.                                                   */
/* ------------------------------------------------------------------ */

/* The 4-point factor printed in "Algorithm: fused ConvRot rotation". */
static const int32_t H4[4][4] = {
    { 1,  1,  1, -1},
    { 1,  1, -1,  1},
    { 1, -1,  1,  1},
    {-1,  1,  1,  1},
};
static const int32_t H2[2][2] = {{1, 1}, {1, -1}};

static int is_pow2(int64_t n) { return n >= 1 && (n & (n - 1)) == 0; }

/*
 * Integer factor H_n, n a power of two, row-major [n][n].
 * The page builds the transform as a Kronecker power of H4 ("Algorithm:
 * fused ConvRot rotation").  For n = 4^j: H_n = H4 (x) ... (x) H4.
 * Reading R-2 (the page is silent for n not a power of four, e.g. 128):
 * H_n = H2 (x) H4^(x)j, with H2 = [[1,1],[1,-1]] on the most significant
 * index bit.  Kronecker convention: (A(x)B)[i*nb+i', j*nb+j'] = A[i,j]*B[i',j'].
 * Returns 0, or -1 when n is not a power of two.
 */
int orc_hadamard(int n, int32_t *H)
{
    if (!is_pow2(n)) return -1;
    int32_t *cur = (int32_t *)malloc(sizeof(int32_t) * (size_t)n * n);
    int32_t *nxt = (int32_t *)malloc(sizeof(int32_t) * (size_t)n * n);
    int size = 1;
    cur[0] = 1;
    int lg = 0;
    while ((1 << lg) < n) ++lg;
    if (lg & 1) { /* H2 first, so it lands on the most significant bit */
        for (int i = 0; i < 2; ++i)
            for (int j = 0; j < 2; ++j) cur[i * 2 + j] = H2[i][j];
        size = 2;
    }
    while (size < n) { /* cur <- cur (x) H4 */
        int ns = size * 4;
        for (int i = 0; i < size; ++i)
            for (int j = 0; j < size; ++j)
                for (int ip = 0; ip < 4; ++ip)
                    for (int jp = 0; jp < 4; ++jp)
                        nxt[(i * 4 + ip) * ns + (j * 4 + jp)] = cur[i * size + j] * H4[ip][jp];
        int32_t *t = cur; cur = nxt; nxt = t;
        size = ns;
    }
    memcpy(H, cur, sizeof(int32_t) * (size_t)n * n);
    free(cur);
    free(nxt);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Rotation  v = (H_a (x) H_b) x / sqrt(a*b), per group of a*b columns. */
/* ------------------------------------------------------------------ */

/*
 * Rotate each row of x (fp32 [M][K]) with the block-diagonal transform
 * I_groups (x) (H_a (x) H_b)/sqrt(a*b), where K = groups*a*b.
 * groups = 1 is the full-width transform; a = b = 16 with groups = K/256 is
 * the page's 256-group form ("API": groupsize 256).
 * Each group, viewed as X[a][b] with x[p*b + q] = X[p][q], becomes
 *   Y[i][j] = sum_p H_a[i][p] * sum_q H_b[j][q] * X[p][q]
 * (the Kronecker definition applied factor by factor), summed in fp64,
 * divided by sqrt(a*b) in fp64 and rounded once to fp32.
 * Returns 0, or -1 on bad descriptors.
 */
int orc_rotate_rows(const float *x, float *v, int64_t M, int64_t K,
                    int a, int b, int groups)
{
    if (!is_pow2(a) || !is_pow2(b) || groups < 1) return -1;
    if ((int64_t)a * b * groups != K) return -1;
    int32_t *Ha = (int32_t *)malloc(sizeof(int32_t) * (size_t)a * a);
    int32_t *Hb = (int32_t *)malloc(sizeof(int32_t) * (size_t)b * b);
    orc_hadamard(a, Ha);
    orc_hadamard(b, Hb);
    const double norm = sqrt((double)a * (double)b);
    int64_t ab = (int64_t)a * b;

    #pragma omp parallel
    {
        double *T = (double *)malloc(sizeof(double) * (size_t)ab);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t m = 0; m < M; ++m) {
            for (int g = 0; g < groups; ++g) {
                const float *xg = x + m * K + (int64_t)g * ab;
                float *vg = v + m * K + (int64_t)g * ab;
                /* T[p][j] = sum_q H_b[j][q] * X[p][q] */
                for (int p = 0; p < a; ++p)
                    for (int j = 0; j < b; ++j) {
                        double s = 0.0;
                        for (int q = 0; q < b; ++q)
                            s += (double)Hb[j * b + q] * (double)xg[p * b + q];
                        T[p * b + j] = s;
                    }
                /* Y[i][j] = sum_p H_a[i][p] * T[p][j] */
                for (int i = 0; i < a; ++i)
                    for (int j = 0; j < b; ++j) {
                        double s = 0.0;
                        for (int p = 0; p < a; ++p)
                            s += (double)Ha[i * a + p] * T[p * b + j];
                        vg[i * b + j] = (float)(s / norm);
                    }
            }
        }
        free(T);
    }
    free(Ha);
    free(Hb);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Per-row symmetric INT8 quantizer (fp32).                            */
/* ------------------------------------------------------------------ */

/*
 * "bf16 [M,K] -> int8 [M,K] + fp32 [M] row scales" (page section "API").
 * Per row:  amax = max_k |v_k|;  s = fp32(amax / 127);
 *           q_k  = clamp(rne(fp32(v_k / s)), -127, 127).
 * Readings: R-3 round-half-even and clamp to +-127 (-128 never produced);
 * R-4 IEEE fp32 division v/s; R-5 a row whose s is 0 (amax = 0, or amax/127
 * underflowing to 0) gets s = 0 and q = 0.
 */
void orc_quantize_rows(const float *v, int8_t *q, float *s, int64_t M, int64_t K)
{
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        const float *vr = v + m * K;
        int8_t *qr = q + m * K;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float a = fabsf(vr[k]);
            if (a > amax) amax = a;
        }
        float sc = amax / 127.0f;
        s[m] = sc;
        if (sc == 0.0f) {
            for (int64_t k = 0; k < K; ++k) qr[k] = 0;
            continue;
        }
        for (int64_t k = 0; k < K; ++k) {
            float t = vr[k] / sc;
            float r = rintf(t); /* default rounding mode: nearest, ties to even */
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            qr[k] = (int8_t)r;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Integer GEMM  acc[m][n] = sum_k q[m][k] * w[n][k]  (int64).          */
/* ------------------------------------------------------------------ */

/*
 * The int8 x int8 -> int32 product of "Use from C" (torch._int_mm on the
 * page), both operands K-contiguous.  Returns the number of results whose
 * magnitude does not fit in int32 (0 on every valid input, since
 * |acc| <= 127*127*K).
 */
int64_t orc_gemm_s8(const int8_t *q, const int8_t *w, int64_t *acc,
                    int64_t M, int64_t N, int64_t K)
{
    int64_t bad = 0;
    #pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
    for (int64_t m = 0; m < M; ++m) {
        const int8_t *qr = q + m * K;
        for (int64_t n = 0; n < N; ++n) {
            const int8_t *wr = w + n * K;
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k) s += (int64_t)qr[k] * (int64_t)wr[k];
            if (s > 2147483647LL || s < -2147483648LL) ++bad;
            acc[m * N + n] = s;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Dequant epilogue.                                                   */
/* ------------------------------------------------------------------ */

/*
 * "out = acc * x_scale[m] * w_scale[n] + bias[n]" (page section "API").
 * Reading R-6 for the operation order: t = fp32(acc) * x_scale[m] in fp32,
 * then fmaf(t, w_scale[n], bias[n]) and one bf16 RNE rounding; a missing
 * bias is +0.  bias is given as fp32 values (bf16 bias widened exactly).
 * acc has leading dimension ld_acc, y has leading dimension ld_y.
 */
void orc_dequant(const int64_t *acc, int64_t ld_acc, const float *xs, const float *ws,
                 const float *bias, uint16_t *y, int64_t ld_y, int64_t M, int64_t N)
{
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            float t = (float)acc[m * ld_acc + n] * xs[m];
            float r = fmaf(t, ws[n], bias ? bias[n] : 0.0f);
            y[m * ld_y + n] = f32_to_bf16_bits(r);
        }
}

/* Same epilogue, fp32 result (no bf16 rounding); used by the dx route. */
void orc_dequant_f32(const int64_t *acc, const float *xs, float *y, int64_t M, int64_t N)
{
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            y[m * N + n] = (float)acc[m * N + n] * xs[m];
}

/* ------------------------------------------------------------------ */
/* SwiGLU middle of the FFN.                                           */
/* ------------------------------------------------------------------ */

/*
 * h = silu(g) * u with silu(x) = x / (1 + exp(-x)), all in fp32, from the
 * bf16 dequant outputs g and u.  Reading R-8: the page's "situ" activation
 * is SiLU in GLU form; reading R-9: g and u are rounded to bf16 (they are
 * dequant outputs) and h stays fp32 (activation fused into the quantizer,
 * page section "Use from Python").
 */
void orc_silu_glu(const uint16_t *g, const uint16_t *u, float *h, int64_t n)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        float gf = bf16_bits_to_f32(g[i]);
        float uf = bf16_bits_to_f32(u[i]);
        float e = expf(-gf);
        float d = 1.0f + e;
        float sg = gf / d;
        h[i] = sg * uf;
    }
}

/* ------------------------------------------------------------------ */
/* Backward helpers.                                                   */
/* ------------------------------------------------------------------ */

/* w[n][k] = fp32(W8[n][k]) * s[n]  (the weight-only dequant of "The backward"). */
void orc_scale_rows_s8(const int8_t *w8, const float *s, float *w, int64_t N, int64_t K)
{
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = (float)w8[n * K + k] * s[n];
}

/* dyp[m][n] = fp32(dy[m][n]) * s[n]: the weight scale as a column scale on dy. */
void orc_scale_cols_bf16(const uint16_t *dy, const float *s, float *dyp, int64_t M, int64_t N)
{
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            dyp[m * N + n] = bf16_bits_to_f32(dy[m * N + n]) * s[n];
}

/*
 * dx[m][k] = sum_n dy[m][n] * w[n][k] with bf16 inputs, summed in fp64,
 * rounded to fp32 and then to bf16 ("dx = dy @ W" of "The backward").
 */
void orc_matmul_bf16_nn(const uint16_t *dy, const uint16_t *w, uint16_t *dx,
                        int64_t M, int64_t N, int64_t K)
{
    #pragma omp parallel
    {
        double *row = (double *)malloc(sizeof(double) * (size_t)K);
        #pragma omp for schedule(dynamic, 1)
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t k = 0; k < K; ++k) row[k] = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                double d = (double)bf16_bits_to_f32(dy[m * N + n]);
                const uint16_t *wr = w + n * K;
                for (int64_t k = 0; k < K; ++k) row[k] += d * (double)bf16_bits_to_f32(wr[k]);
            }
            for (int64_t k = 0; k < K; ++k) dx[m * K + k] = f32_to_bf16_bits((float)row[k]);
        }
        free(row);
    }
}

/*
 * y[m][n] = bf16( sum_k x[m][k] * w[n][k] + bias[n] ) with bf16 inputs, the
 * sum and the bias add in fp64, rounded to fp32 and then to bf16: the linear
 * layer of the rotate-only BF16 path ("Use from C": the activation rotated by
 * the rotate-only kernel, then a bf16 linear against the pre-rotated weight).
 * bias may be NULL.
 */
void orc_linear_bf16(const uint16_t *x, const uint16_t *w, const uint16_t *bias,
                     uint16_t *y, int64_t M, int64_t N, int64_t K)
{
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *xr = x + m * K;
        for (int64_t n = 0; n < N; ++n) {
            const uint16_t *wr = w + n * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)bf16_bits_to_f32(xr[k]) * (double)bf16_bits_to_f32(wr[k]);
            if (bias) acc += (double)bf16_bits_to_f32(bias[n]);
            y[m * N + n] = f32_to_bf16_bits((float)acc);
        }
    }
}
