// Launchers shared between the C-ABI translation unit and the kernel
// translation units.  Arguments are already validated when these run.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace jetfp8 {

// Error-word bits set by bounded waits that gave up.
enum : uint32_t {
    ERRBIT_PRODUCER = 1u << 0,   // TMA producer: waiting for a free smem stage
    ERRBIT_MMA_SMEM = 1u << 1,   // MMA issuer: waiting for a filled smem stage
    ERRBIT_MMA_TMEM = 1u << 2,   // MMA issuer: waiting for a free TMEM buffer
    ERRBIT_PROMOTE = 1u << 3,    // promotion warps: waiting for a finished TMEM partial
    ERRBIT_DRAIN = 1u << 4,      // teardown: waiting for copies / MMAs in flight
    ERRBIT_SELFTEST = 1u << 5,   // the watchdog self-test kernel
    ERRBIT_QUANT = 1u << 6,      // dual / weight quantiser: waiting for its tile
};

// Quantisers (quantize.cu).  All return the cudaGetLastError() of the launch.
cudaError_t launch_quantize_act(const void *x, int64_t M, int64_t K, uint8_t *q, float *s,
                                cudaStream_t stream);
cudaError_t launch_quantize_act_transposed(const void *x, int64_t M, int64_t C, uint8_t *qt, float *st,
                                           cudaStream_t stream);
cudaError_t launch_quantize_act_dual(const void *x, int64_t M, int64_t K, uint8_t *q, float *s, uint8_t *qt,
                                     float *st, PFN_cuTensorMapEncodeTiled_v12000 encode, uint32_t *err,
                                     cudaStream_t stream);
cudaError_t launch_quantize_weight(const void *w, int64_t N, int64_t K, uint8_t *q, float *s, uint8_t *qt,
                                   PFN_cuTensorMapEncodeTiled_v12000 encode, uint32_t *err, int sm_count,
                                   cudaStream_t stream);
// 1 <= count <= 8 weight tensors in one launch (arrays of count host entries)
cudaError_t launch_quantize_weight_group(int count, const void *const *w, const int64_t *N, const int64_t *K,
                                         uint8_t *const *q, float *const *s, uint8_t *const *qt,
                                         PFN_cuTensorMapEncodeTiled_v12000 encode, uint32_t *err, int sm_count,
                                         cudaStream_t stream);
cudaError_t launch_e4m3_encode_range(uint32_t first, int64_t count, uint8_t *codes, int sm_count,
                                     cudaStream_t stream);

// Fused producers (producers.cu): RMSNorm / SwiGLU -> bf16 -> 1x128 FP8.
// q and s may be null (then only y is written); y may be null.
cudaError_t launch_rmsnorm_quantize(const void *x, const void *gamma, float eps, int64_t M, int64_t H, uint8_t *q,
                                    float *s, void *y, cudaStream_t stream);
cudaError_t launch_swiglu_quantize(const void *gu, int64_t M, int64_t I, uint8_t *q, float *s, void *y,
                                   int sm_count, cudaStream_t stream);

// One block-scaled GEMM D[rows][cols] = sum_g sa(g,row) sb(g,col) (A_g B_g^T),
// A: [rows][kdim] codes, B: [cols][kdim] codes, both K-major (gemm.cu).
enum class ScaleB { PerBlock128, PerColumn };

struct GemmProblem {
    const uint8_t *a;      // [rows][kdim]
    const uint8_t *b;      // [cols][kdim]
    const float *sa;       // sa(g,row) = sa[g*rows + row]
    const float *sb;       // PerBlock128: sb[g*sb_stride_g + (col/128)*sb_stride_c]
                           // PerColumn : sb[g*sb_stride_g + col]
    int64_t sb_stride_g;
    int64_t sb_stride_c;
    ScaleB sb_mode;
    void *d;               // bf16 [rows][cols]
    int64_t rows, cols, kdim;
};

struct DeviceInfo {
    int sm_count;
    uint32_t *err_word;    // device address of this device's error word
};

cudaError_t launch_gemm(const GemmProblem &p, const DeviceInfo &dev, PFN_cuTensorMapEncodeTiled_v12000 encode,
                        cudaStream_t stream);

cudaError_t launch_watchdog_selftest(uint32_t *err_word, uint64_t timeout_ns, cudaStream_t stream);

}  // namespace jetfp8
