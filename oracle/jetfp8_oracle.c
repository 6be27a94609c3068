/*
 * jetfp8 CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded restatement of what the FP8 linear-layer
 * path computes, used to check the CUDA library.  Only the test suite, the
 * package smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never calls it and shares no code, header, table or constant
 * generator with it.
 *
 * Sources (Jet-RL: "Enabling On-Policy FP8 Reinforcement Learning with
 * Unified Training and Rollout Precision Flow", technical summaries on
 * gist.science, French and Portuguese pages):
 *   - "Schéma de Quantification" / "Esquema de Quantização": activations are
 *     quantised per 1x128 group, weights per 128x128 block; the backward
 *     DGrad/WGrad GEMMs run in FP8 with 1x128 / 128x1 groups for WGrad;
 *     gradients between operators stay BF16.
 *   - "Architecture Centrale" / "Arquitetura Central": rollout and training
 *     forward share one quantisation flow; master weights are BF16.
 * The pages say only "FP8".  Where they are silent this file takes the
 * readings below:
 *   - format: OCP FP8 E4M3 "FN" (bias 7, no infinities, S.1111.111 = NaN,
 *     largest finite 448);
 *   - scale: one fp32 per group, s = amax / 448 as one IEEE fp32 division;
 *   - code: q = E4M3(RNE, saturating)(fp32(x / s)), one IEEE fp32 division
 *     per element; an all-zero group stores s = 0 and codes 0x00;
 *   - GEMMs: the exact (fp64) sum over the whole contraction of
 *     (decode(qa) * sa) * (decode(qb) * sb).
 * Build: plain C99, -O2, no fast-math, no FMA contraction.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* The E4M3 format (OCP 8-bit floating point specification, E4M3).    */
/* Bit layout s|eeee|mmm, exponent bias 7.                            */
/*   eeee > 0 : (-1)^s * 2^(eeee-7) * (1 + mmm/8)                     */
/*   eeee = 0 : (-1)^s * 2^(-6)     * (mmm/8)        (subnormals)     */
/*   s.1111.111 : NaN (the FN variant has no infinities)              */
/* ------------------------------------------------------------------ */

double jo_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/*
 * Nearest E4M3 value to v, ties to the even mantissa, saturating to the
 * largest finite magnitude (448) instead of producing NaN.  The sign of v is
 * kept, so -0 and negative values that round to zero give 0x80.  NaN gives
 * 0x7F.  Works from the value itself: pick the binade, divide by its
 * quantum (a power of two, so exact), round to an integer with the default
 * IEEE rounding (nearest, ties to even).
 */
uint8_t jo_e4m3_encode(float v)
{
    uint8_t sign;
    double a, quantum, n;
    int x, E;

    if (isnan(v))
        return 0x7F;
    sign = signbit(v) ? 0x80 : 0x00;
    a = fabs((double)v);
    if (a >= 448.0)                       /* saturate (satfinite) */
        return (uint8_t)(sign | 0x7E);

    if (a < ldexp(1.0, -6)) {             /* subnormal binade: quantum 2^-9 */
        n = nearbyint(a / ldexp(1.0, -9));   /* 0..8; 8 is 2^-6 = code 0x08 */
        return (uint8_t)(sign | (uint8_t)n);
    }

    frexp(a, &x);                         /* a in [2^(x-1), 2^x) */
    E = x - 1;                            /* unbiased exponent, -6..8 */
    quantum = ldexp(1.0, E - 3);          /* 3 mantissa bits */
    n = nearbyint(a / quantum);           /* 8..16 */
    if (n == 16.0) {                      /* rounded up into the next binade */
        E += 1;
        n = 8.0;
    }
    return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | ((int)n - 8)));
}

/* bf16 is the upper half of an fp32 bit pattern. */
float jo_bf16_to_float(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

/* One group: s = amax / 448 (fp32), codes E4M3(x / s) (fp32 quotient). */
static float group_scale(float amax)
{
    return amax / 448.0f;
}

static uint8_t group_code(float x, float s)
{
    if (s == 0.0f)
        return 0x00;
    return jo_e4m3_encode(x / s);
}

/*
 * Activations / gradients, 1x128 groups along each row
 * ("Schéma de Quantification": activations 1x128 per group).
 *   x : bf16 bits [M][K]        q : codes [M][K]
 *   s : fp32 [K/128][M]  (group-major: s[g*M + m] belongs to row m, group g)
 */
void jo_quantize_act(const uint16_t *x, int64_t M, int64_t K, uint8_t *q, float *s)
{
    int64_t G = K / 128;
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < G; ++g) {
            float amax = 0.0f, sc;
            for (int64_t k = g * 128; k < g * 128 + 128; ++k) {
                float a = fabsf(jo_bf16_to_float(x[m * K + k]));
                if (a > amax)
                    amax = a;
            }
            sc = group_scale(amax);
            s[g * M + m] = sc;
            for (int64_t k = g * 128; k < g * 128 + 128; ++k)
                q[m * K + k] = group_code(jo_bf16_to_float(x[m * K + k]), sc);
        }
    }
}

/*
 * The WGrad operand: groups of 128 consecutive rows (tokens) of one column
 * ("128x1" in the [M][C] layout), written transposed so that each group is
 * 1x128 in the output (the summaries give WGrad 1x128 and 128x1 groups,
 * "Schéma de Quantification").
 *   x : bf16 bits [M][C]         qt : codes [C][M]
 *   st: fp32 [M/128][C]  (st[g*C + c] belongs to column c, row group g)
 */
void jo_quantize_act_transposed(const uint16_t *x, int64_t M, int64_t C, uint8_t *qt, float *st)
{
    int64_t G = M / 128;
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t g = 0; g < G; ++g) {
            float amax = 0.0f, sc;
            for (int64_t m = g * 128; m < g * 128 + 128; ++m) {
                float a = fabsf(jo_bf16_to_float(x[m * C + c]));
                if (a > amax)
                    amax = a;
            }
            sc = group_scale(amax);
            st[g * C + c] = sc;
            for (int64_t m = g * 128; m < g * 128 + 128; ++m)
                qt[c * M + m] = group_code(jo_bf16_to_float(x[m * C + c]), sc);
        }
    }
}

/*
 * Weights, 128x128 blocks ("Schéma de Quantification": weights 128x128 per
 * block).
 *   w : bf16 bits [N][K]     q : codes [N][K]     s : fp32 [N/128][K/128]
 *   qt: optional codes [K][N] (the same codes, transposed), may be NULL.
 */
void jo_quantize_weight(const uint16_t *w, int64_t N, int64_t K, uint8_t *q, float *s, uint8_t *qt)
{
    int64_t BN = N / 128, BK = K / 128;
    for (int64_t bn = 0; bn < BN; ++bn) {
        for (int64_t bk = 0; bk < BK; ++bk) {
            float amax = 0.0f, sc;
            for (int64_t n = bn * 128; n < bn * 128 + 128; ++n)
                for (int64_t k = bk * 128; k < bk * 128 + 128; ++k) {
                    float a = fabsf(jo_bf16_to_float(w[n * K + k]));
                    if (a > amax)
                        amax = a;
                }
            sc = group_scale(amax);
            s[bn * BK + bk] = sc;
            for (int64_t n = bn * 128; n < bn * 128 + 128; ++n)
                for (int64_t k = bk * 128; k < bk * 128 + 128; ++k) {
                    uint8_t c = group_code(jo_bf16_to_float(w[n * K + k]), sc);
                    q[n * K + k] = c;
                    if (qt)
                        qt[k * N + n] = c;
                }
        }
    }
}

/* ------------------------------------------------------------------ */
/* GEMMs: exact fp64 sums of dequantised products, one output element */
/* at a time.  Each returns the value and the sum of |terms| (for the */
/* tolerance).                                                        */
/* ------------------------------------------------------------------ */

/* Y[m][n] = sum_k deq(QX[m][k]) * deq(QW[n][k])      (Fprop, Y = X W^T)
 *   qx [M][K], sx [K/128][M], qw [N][K], sw [N/128][K/128]            */
static void fprop_elem(const uint8_t *qx, const float *sx, const uint8_t *qw, const float *sw,
                       int64_t M, int64_t N, int64_t K, int64_t m, int64_t n,
                       double *val, double *abssum)
{
    double acc = 0.0, aacc = 0.0;
    int64_t BK = K / 128;
    for (int64_t k = 0; k < K; ++k) {
        double a = jo_e4m3_decode(qx[m * K + k]) * (double)sx[(k / 128) * M + m];
        double b = jo_e4m3_decode(qw[n * K + k]) * (double)sw[(n / 128) * BK + k / 128];
        acc += a * b;
        aacc += fabs(a * b);
    }
    *val = acc;
    *abssum = aacc;
}

/* dX[m][k] = sum_n deq(QdY[m][n]) * deq(QW[n][k])    (Dgrad, dX = dY W)
 *   qdy [M][N], sdy [N/128][M], qw [N][K], sw [N/128][K/128]          */
static void dgrad_elem(const uint8_t *qdy, const float *sdy, const uint8_t *qw, const float *sw,
                       int64_t M, int64_t N, int64_t K, int64_t m, int64_t k,
                       double *val, double *abssum)
{
    double acc = 0.0, aacc = 0.0;
    int64_t BK = K / 128;
    for (int64_t n = 0; n < N; ++n) {
        double a = jo_e4m3_decode(qdy[m * N + n]) * (double)sdy[(n / 128) * M + m];
        double b = jo_e4m3_decode(qw[n * K + k]) * (double)sw[(n / 128) * BK + k / 128];
        acc += a * b;
        aacc += fabs(a * b);
    }
    *val = acc;
    *abssum = aacc;
}

/* dW[n][k] = sum_m deq(QdY^T[n][m]) * deq(QX^T[k][m])  (Wgrad, dW = dY^T X)
 *   qdyt [N][M], sdyt [M/128][N], qxt [K][M], sxt [M/128][K]          */
static void wgrad_elem(const uint8_t *qdyt, const float *sdyt, const uint8_t *qxt, const float *sxt,
                       int64_t M, int64_t N, int64_t K, int64_t n, int64_t k,
                       double *val, double *abssum)
{
    double acc = 0.0, aacc = 0.0;
    for (int64_t m = 0; m < M; ++m) {
        double a = jo_e4m3_decode(qdyt[n * M + m]) * (double)sdyt[(m / 128) * N + n];
        double b = jo_e4m3_decode(qxt[k * M + m]) * (double)sxt[(m / 128) * K + k];
        acc += a * b;
        aacc += fabs(a * b);
    }
    *val = acc;
    *abssum = aacc;
}

/*
 * Drivers.  `rows`/`cols` list the output elements to compute (count of
 * them: `count`); out[i] and abssum[i] receive element (rows[i], cols[i]).
 * A full GEMM passes every (row, col) pair.
 */
void jo_gemm_fprop(const uint8_t *qx, const float *sx, const uint8_t *qw, const float *sw,
                   int64_t M, int64_t N, int64_t K,
                   const int64_t *rows, const int64_t *cols, int64_t count,
                   double *out, double *abssum)
{
    for (int64_t i = 0; i < count; ++i)
        fprop_elem(qx, sx, qw, sw, M, N, K, rows[i], cols[i], &out[i], &abssum[i]);
}

void jo_gemm_dgrad(const uint8_t *qdy, const float *sdy, const uint8_t *qw, const float *sw,
                   int64_t M, int64_t N, int64_t K,
                   const int64_t *rows, const int64_t *cols, int64_t count,
                   double *out, double *abssum)
{
    for (int64_t i = 0; i < count; ++i)
        dgrad_elem(qdy, sdy, qw, sw, M, N, K, rows[i], cols[i], &out[i], &abssum[i]);
}

void jo_gemm_wgrad(const uint8_t *qdyt, const float *sdyt, const uint8_t *qxt, const float *sxt,
                   int64_t M, int64_t N, int64_t K,
                   const int64_t *rows, const int64_t *cols, int64_t count,
                   double *out, double *abssum)
{
    for (int64_t i = 0; i < count; ++i)
        wgrad_elem(qdyt, sdyt, qxt, sxt, M, N, K, rows[i], cols[i], &out[i], &abssum[i]);
}

/* Array forms of the codec, for the tests. */
void jo_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = jo_e4m3_encode(v[i]);
}

void jo_e4m3_decode_array(const uint8_t *c, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = jo_e4m3_decode(c[i]);
}

/* Encode every fp32 bit pattern in [lo, hi) and count mismatches against
 * `table` codes given for the same patterns (used to compare a bulk GPU
 * conversion against this encoder without shipping 4 GiB through Python). */
int64_t jo_e4m3_encode_check_range(uint32_t lo, uint64_t count, const uint8_t *codes,
                                   int64_t *first_bad)
{
    int64_t bad = 0;
    *first_bad = -1;
    for (uint64_t i = 0; i < count; ++i) {
        uint32_t bits = lo + (uint32_t)i;
        float f;
        memcpy(&f, &bits, sizeof f);
        if (jo_e4m3_encode(f) != codes[i]) {
            if (bad == 0)
                *first_bad = (int64_t)i;
            ++bad;
        }
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Producers fused in front of the linear layers.                      */
/*                                                                    */
/* The pages (technical summaries, "Implémentation") name fused      */
/* activation / RMSNorm kernels that emit the FP8 input of the next  */
/* GEMM, without their arithmetic.  The oracle takes the operators'  */
/* textbook definitions and evaluates them in fp64 (double), in the  */
/* plainest order; the bf16 value a kernel produces is checked        */
/* against this to within one bf16 ulp, and the kernel's FP8 codes    */
/* against jo_quantize_act of that bf16 value.                        */
/* ------------------------------------------------------------------ */

/*
 * RMSNorm (root-mean-square layer normalisation, Zhang and Sennrich 2019)
 * of x bf16 [M][H] with gain gamma bf16 [H]:
 *   y_i = x_i / sqrt( (1/H) sum_j x_j^2 + eps ) * gamma_i,
 * every operation in double, the sum over the row in natural order.
 *   y : fp64 [M][H]
 */
void jo_rmsnorm_f64(const uint16_t *x, const uint16_t *gamma, double eps, int64_t M, int64_t H, double *y)
{
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = x + m * H;
        double sum = 0.0, rms;
        for (int64_t j = 0; j < H; ++j) {
            double v = (double)jo_bf16_to_float(row[j]);
            sum += v * v;
        }
        rms = sqrt(sum / (double)H + eps);
        for (int64_t i = 0; i < H; ++i)
            y[m * H + i] = (double)jo_bf16_to_float(row[i]) / rms * (double)jo_bf16_to_float(gamma[i]);
    }
}

/*
 * SwiGLU of a gate_up projection output, gu bf16 [M][2I] (gate = columns
 * 0..I-1, up = columns I..2I-1):
 *   y = silu(g) * u,   silu(g) = g * sigmoid(g) = g / (1 + e^-g),
 * in double with the C library's exp.
 *   y : fp64 [M][I]
 */
void jo_swiglu_f64(const uint16_t *gu, int64_t M, int64_t I, double *y)
{
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *row = gu + m * 2 * I;
        for (int64_t i = 0; i < I; ++i) {
            double g = (double)jo_bf16_to_float(row[i]);
            double u = (double)jo_bf16_to_float(row[I + i]);
            y[m * I + i] = g / (1.0 + exp(-g)) * u;
        }
    }
}
