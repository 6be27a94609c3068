/*
 * jetfp8 -- group-wise FP8 (E4M3) quantisation and block-scaled FP8 GEMMs
 * for the forward (Fprop), input-gradient (Dgrad) and weight-gradient
 * (Wgrad) products of a linear layer, on NVIDIA GB300 (sm_103a).
 *
 * The method (Jet-RL: "Enabling On-Policy FP8 Reinforcement Learning with
 * Unified Training and Rollout Precision Flow"; technical summaries on
 * gist.science, French page "Schéma de Quantification", Portuguese page
 * "Esquema de Quantização"): the linear layers (GEMMs) quantise activations
 * with 1x128 groups and weights with 128x128 blocks; gradients passed
 * between operators stay BF16; the backward DGrad and WGrad GEMMs also run
 * in FP8, with 1x128 / 128x1 groups for WGrad; activations saved for the
 * backward pass are kept in FP8.  The same kernels serve rollout and the
 * training forward ("Architecture Centrale": one quantisation flow for both),
 * so both produce bit-identical results for the same inputs.
 *
 * Numerical definition (the pages say only "FP8"; these are this library's
 * stated choices):
 *   - codes are OCP FP8 E4M3 ("FN": bias 7, no infinities, max finite 448);
 *   - each group has one fp32 scale s = amax / 448 (IEEE fp32 division);
 *   - code = E4M3 round-to-nearest-even, saturating, of fp32(x / s) (IEEE
 *     fp32 division, no flush-to-zero); a group of zeros stores s = 0 and
 *     codes 0x00;
 *   - a GEMM sums, per 128-wide contraction group, the exact FP8 products in
 *     fp32 on the tensor cores, multiplies that partial by the two groups'
 *     scales in fp32, accumulates in fp32 and rounds the result once to bf16
 *     (round to nearest even).
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers to caller-owned memory, dense
 *     row-major with no padding (leading dimension = number of columns).
 *     The library never allocates, frees or synchronises inside these calls
 *     (jetfp8_poll_device_error excepted), and keeps no mutable state between
 *     them apart from a per-device cache of immutable facts (SM count, the
 *     driver's tensor-map encoder) and one per-device error word.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) in order, and is complete when the stream says so.
 *   - Outputs are fully overwritten; inputs are never modified.  An output
 *     that overlaps any input or another output is rejected.
 *   - Every argument check happens on the host before anything is launched;
 *     a call that returns an error has enqueued no work.
 *   - Empty inputs (M == 0) are accepted and launch nothing.
 *   - Base pointers must be 16-byte aligned.
 *   - Calls are thread-safe; calls on different streams may run concurrently.
 */
#ifndef JETFP8_H
#define JETFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define JETFP8_API __attribute__((visibility("default")))
#else
#define JETFP8_API
#endif

typedef enum jetfp8_status {
    JETFP8_OK = 0,
    JETFP8_ERR_INVALID_VALUE = 1,      /* NULL pointer, or an output overlaps an input/output */
    JETFP8_ERR_SHAPE = 2,              /* a size is negative, zero where it must not be, or not a
                                          multiple of 128 where the layout needs one, or too large */
    JETFP8_ERR_ALIGNMENT = 3,          /* a base pointer is not 16-byte aligned */
    JETFP8_ERR_UNSUPPORTED_DEVICE = 4, /* no CUDA device, or the current device is not sm_103 */
    JETFP8_ERR_LAUNCH = 5,             /* the CUDA runtime reported an error for the launch */
    JETFP8_ERR_TIMEOUT = 6             /* a kernel's bounded wait gave up (see poll_device_error) */
} jetfp8_status;

/*
 * Activation / gradient quantisation, 1x128 groups along each row
 * (Jet-RL, "Schéma de Quantification": activations 1x128 per group;
 *  gradients stay BF16 between operators and are quantised at the GEMM).
 *   x : bf16 [M][K]                       (input)
 *   q : uint8 E4M3 codes [M][K]           (output)
 *   s : fp32 [K/128][M], s[g*M + m] is the scale of row m, group g
 *       (group-major, so a tile's scales for one group are contiguous)
 * Requires M >= 0, K > 0, K % 128 == 0, M * K < 2^40.
 */
JETFP8_API jetfp8_status jetfp8_quantize_act(const void *x, int64_t M, int64_t K,
                                             uint8_t *q, float *s, void *stream);

/*
 * Quantise-transpose for the WGrad operand: groups of 128 consecutive rows
 * (tokens) of each column -- "128x1" in the [M][C] input, "1x128" in the
 * transposed output (Jet-RL, "Schéma de Quantification": 1x128 and 128x1
 * groups for WGrad; "Implémentation": quantisation and transposition
 * kernels).  Used for X (saved activation, kept in FP8) and for dY.
 *   x  : bf16 [M][C]                      (input)
 *   qt : uint8 E4M3 codes [C][M]          (output, qt[c*M + m] is the code of x[m][c])
 *   st : fp32 [M/128][C], st[g*C + c] is the scale of column c, rows 128g..128g+127
 * Requires M % 128 == 0, C > 0, C % 128 == 0, M * C < 2^40.
 */
JETFP8_API jetfp8_status jetfp8_quantize_act_transposed(const void *x, int64_t M, int64_t C,
                                                        uint8_t *qt, float *st, void *stream);

/*
 * Both activation layouts from one read of x: exactly the outputs of
 * jetfp8_quantize_act(x -> q, s) and jetfp8_quantize_act_transposed(x -> qt,
 * st), bit for bit, at the HBM cost of reading x once.  This is the training
 * forward's quantisation of X (the 1x128 codes feed Fprop, the transposed
 * 128x1 codes are the activation saved in FP8 for WGrad) and the backward's
 * quantisation of dY (DGrad and WGrad operands) -- Jet-RL, "Schéma de
 * Quantification": saved activations kept in FP8; "Implémentation": fused
 * quantisation and transposition kernels.
 *   x  : bf16 [M][K]
 *   q  : uint8 [M][K],  s  : fp32 [K/128][M]   (as jetfp8_quantize_act)
 *   qt : uint8 [K][M],  st : fp32 [M/128][K]   (as jetfp8_quantize_act_transposed)
 * Requires M % 128 == 0, K > 0, K % 128 == 0, M * K < 2^40.
 */
JETFP8_API jetfp8_status jetfp8_quantize_act_dual(const void *x, int64_t M, int64_t K, uint8_t *q, float *s,
                                                  uint8_t *qt, float *st, void *stream);

/*
 * Fused RMSNorm producer: the 1x128 FP8 input of the next linear layer
 * straight from the residual stream (Jet-RL, "Implémentation": fused
 * activation / RMSNorm kernels in front of the FP8 GEMMs).  Per row:
 *   y_i = x_i / sqrt( (1/H) sum_j x_j^2 + eps ) * gamma_i,
 * returned as bf16 within one bf16 ulp of the exact value (computed in
 * fp32 in a fixed order, so a row's bits never depend on the launch or the
 * other rows).  Rows whose sum of squares overflows fp32 are outside the
 * domain.  The codes and scales are exactly those jetfp8_quantize_act
 * gives for the returned bf16 y.
 *   x     : bf16 [M][H]                    (input)
 *   gamma : bf16 [H]                       (input)
 *   eps   : finite, >= 0
 *   q, s  : uint8 [M][H], fp32 [H/128][M]  (as jetfp8_quantize_act), or both NULL
 *   y     : bf16 [M][H] or NULL            (the normalised values themselves)
 * At least one of (q, s) and y is given.  Requires H > 0, H % 256 == 0,
 * M * H < 2^40.
 */
JETFP8_API jetfp8_status jetfp8_rmsnorm_quantize_act(const void *x, const void *gamma, float eps, int64_t M,
                                                     int64_t H, uint8_t *q, float *s, void *y, void *stream);

/*
 * Fused SwiGLU producer: the 1x128 FP8 input of the down projection from
 * the gate_up output (Jet-RL, "Implémentation": fused activation kernels).
 * gu holds gate in columns 0..I-1 and up in columns I..2I-1 of each row;
 *   y = silu(g) * u = g / (1 + e^-g) * u,
 * returned as bf16 within one bf16 ulp of the exact value (fp32 in a fixed
 * order, e^-g and the reciprocal from the hardware's fp32 approximations,
 * whose error stays far inside that bound); for g < -87, where the fp32
 * sigmoid underflows, within 2^-119 |u| of it.  The codes and scales are
 * exactly those jetfp8_quantize_act gives for the returned bf16 y.
 *   gu   : bf16 [M][2I]                    (input)
 *   q, s : uint8 [M][I], fp32 [I/128][M], or both NULL
 *   y    : bf16 [M][I] or NULL
 * At least one of (q, s) and y is given.  Requires I > 0, I % 256 == 0,
 * M * 2I < 2^40.
 */
JETFP8_API jetfp8_status jetfp8_swiglu_quantize_act(const void *gu, int64_t M, int64_t I, uint8_t *q, float *s,
                                                    void *y, void *stream);

/*
 * Weight quantisation, 128x128 blocks (Jet-RL, "Schéma de Quantification":
 * weights 128x128 per block; master weights stay BF16, "Architecture
 * Centrale").
 *   w  : bf16 [N][K]                      (input, the BF16 master weight)
 *   q  : uint8 E4M3 codes [N][K]          (output)
 *   s  : fp32 [N/128][K/128] row-major    (output)
 *   qt : uint8 [K][N] or NULL             (optional output: the same codes
 *        transposed, the weight operand of jetfp8_gemm_dgrad; a 128x128
 *        block and its transpose share one scale, so no re-quantisation)
 * Requires N, K > 0, both multiples of 128, N * K < 2^40.
 */
JETFP8_API jetfp8_status jetfp8_quantize_weight(const void *w, int64_t N, int64_t K,
                                                uint8_t *q, float *s, uint8_t *qt,
                                                void *stream);

/*
 * Several weight tensors quantised in one launch, each exactly as
 * jetfp8_quantize_weight quantises it (same codes, scales and transposed
 * codes, bit for bit).  The pages quantise the BF16 master weights to FP8
 * each step ("Architecture Centrale", "Schéma de Quantification"); they
 * have no grouped call of their own: grouping only lets one launch cover
 * every weight of a step, so the small tensors share the start-up and the
 * last stores of the large ones.
 *   count : 0 .. JETFP8_WEIGHT_GROUP_MAX (0 does nothing)
 *   w, N, K, q, s, qt : host arrays of count entries, all six given (qt[t]
 *           may be NULL); entry t describes one tensor as the arguments of
 *           jetfp8_quantize_weight do.  The arrays are read during the call
 *           only; the device buffers they point to stay the caller's.
 * Every entry must satisfy jetfp8_quantize_weight's requirements, and no
 * output may overlap an input or output of any entry.  Nothing is launched
 * unless every entry passes.
 */
#define JETFP8_WEIGHT_GROUP_MAX 8
JETFP8_API jetfp8_status jetfp8_quantize_weight_group(int count, const void *const *w, const int64_t *N,
                                                      const int64_t *K, uint8_t *const *q, float *const *s,
                                                      uint8_t *const *qt, void *stream);

/*
 * Fprop: Y = X W^T (Jet-RL, "Schéma de Quantification": FP8 GEMMs of the
 * linear layers).
 *   y[m][n] = bf16( sum_g sx[g][m] * sw[n/128][g] * sum_{k in group g} e4m3(qx[m][k]) * e4m3(qw[n][k]) )
 *   qx : [M][K] codes,  sx : [K/128][M]   (from jetfp8_quantize_act)
 *   qw : [N][K] codes,  sw : [N/128][K/128] (from jetfp8_quantize_weight)
 *   y  : bf16 [M][N]                      (output)
 * Requires M >= 0, N, K > 0 and multiples of 128.
 */
JETFP8_API jetfp8_status jetfp8_gemm_fprop(const uint8_t *qx, const float *sx,
                                           const uint8_t *qw, const float *sw,
                                           void *y, int64_t M, int64_t N, int64_t K,
                                           void *stream);

/*
 * Dgrad: dX = dY W (Jet-RL, "Schéma de Quantification": DGrad in FP8; the
 * Portuguese page states FP8 where the French one says FP16 -- FP8 is the
 * reading taken, matching the unified-FP8 claim).
 *   dx[m][k] = bf16( sum_g sdy[g][m] * sw[g][k/128] * sum_{n in group g} e4m3(qdy[m][n]) * e4m3(qw[n][k]) )
 *   qdy : [M][N] codes, sdy : [N/128][M]  (jetfp8_quantize_act of dY)
 *   qwt : [K][N] codes                    (the transposed weight codes,
 *                                          jetfp8_quantize_weight's qt)
 *   sw  : [N/128][K/128]                  (the weight's block scales, untransposed)
 *   dx  : bf16 [M][K]                     (output)
 * Requires M >= 0, N, K > 0 and multiples of 128.
 */
JETFP8_API jetfp8_status jetfp8_gemm_dgrad(const uint8_t *qdy, const float *sdy,
                                           const uint8_t *qwt, const float *sw,
                                           void *dx, int64_t M, int64_t N, int64_t K,
                                           void *stream);

/*
 * Wgrad: dW = dY^T X, contraction over the M tokens (Jet-RL, "Schéma de
 * Quantification": WGrad in FP8 with 1x128 and 128x1 groups -- both
 * operands grouped along the token axis, as produced by
 * jetfp8_quantize_act_transposed).
 *   dw[n][k] = bf16( sum_g sdyt[g][n] * sxt[g][k] * sum_{m in group g} e4m3(qdyt[n][m]) * e4m3(qxt[k][m]) )
 *   qdyt : [N][M] codes, sdyt : [M/128][N]
 *   qxt  : [K][M] codes, sxt  : [M/128][K]
 *   dw   : bf16 [N][K]                    (output)
 * Requires M >= 0 and M % 128 == 0, N, K > 0 and multiples of 128.
 * M == 0 writes nothing (the empty sum is not materialised).
 */
JETFP8_API jetfp8_status jetfp8_gemm_wgrad(const uint8_t *qdyt, const float *sdyt,
                                           const uint8_t *qxt, const float *sxt,
                                           void *dw, int64_t M, int64_t N, int64_t K,
                                           void *stream);

/*
 * Test hook for the conversion every quantiser ends in: codes[i] = the
 * OCP E4M3 code (round to nearest even, saturating to +-448, every NaN ->
 * 0x7F, whatever its sign) that the GPU's E4M3 conversion gives for the fp32 value whose
 * bit pattern is first + i, i = 0 .. count-1.  Lets a test compare the
 * hardware conversion with a reference over all 2^32 fp32 patterns, in
 * chunks.
 *   codes : uint8 [count], device memory, 16-byte aligned (output)
 * Requires 0 <= count <= 2^32 - first.
 */
JETFP8_API jetfp8_status jetfp8_e4m3_encode_range(uint32_t first, int64_t count, uint8_t *codes, void *stream);

/* Number of fp32 scales of a [rows][cols] tensor quantised in 1x128 groups
 * along cols: (cols / 128) * rows.  Returns 0 for invalid sizes. */
JETFP8_API size_t jetfp8_act_scale_count(int64_t rows, int64_t cols);

/* Static, human-readable name of a status code (never NULL). */
JETFP8_API const char *jetfp8_status_string(jetfp8_status status);

/*
 * Debug / watchdog query.  Synchronises `stream`, then reads and clears the
 * current device's error word, which a kernel sets when one of its bounded
 * waits on an asynchronous-copy or tensor-core barrier gives up (the kernel
 * then releases its resources and exits instead of hanging).  Returns
 * JETFP8_ERR_TIMEOUT if the word was set, JETFP8_ERR_LAUNCH if the stream
 * reported a CUDA error, else JETFP8_OK.
 */
JETFP8_API jetfp8_status jetfp8_poll_device_error(void *stream);

/*
 * Watchdog self-test: launches one block whose only work is a bounded wait
 * on a shared-memory barrier that nothing ever completes, so the wait runs
 * out after about `timeout_us` microseconds (1..1000000) and sets the
 * device error word; jetfp8_poll_device_error then reports
 * JETFP8_ERR_TIMEOUT.  The same bounded-wait routine guards every wait in
 * the GEMM kernels.  Returns JETFP8_ERR_SHAPE for an out-of-range timeout.
 */
JETFP8_API jetfp8_status jetfp8_watchdog_selftest(int64_t timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* JETFP8_H */
