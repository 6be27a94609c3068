// C-ABI entry points (include/jetfp8.h): host-side argument checks, the
// per-device cache, and dispatch to the kernels.  Every check runs before
// any CUDA call that could enqueue work, so a rejected call launches nothing.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "jetfp8.h"
#include "internal.cuh"

namespace {

using jetfp8::DeviceInfo;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;   // rows / columns
constexpr int64_t kMaxElems = int64_t{1} << 40;

// One error word per device, set by kernels whose bounded waits gave up.
__device__ uint32_t g_device_error;

struct DeviceSlot {
    std::once_flag once;
    bool ok = false;
    DeviceInfo info{};
};

DeviceSlot g_slots[kMaxDevices];
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

void init_encode()
{
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Immutable per-device facts, looked up once per device with it current.
jetfp8_status current_device(const DeviceInfo **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return JETFP8_ERR_UNSUPPORTED_DEVICE;
    }
    DeviceSlot &slot = g_slots[dev];
    std::call_once(slot.once, [&slot, dev]() {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        if (major != 10 || minor != 3)   // the kernels are built for sm_103a only
            return;
        void *err = nullptr;
        if (cudaGetSymbolAddress(&err, g_device_error) != cudaSuccess) {
            cudaGetLastError();
            return;
        }
        slot.info.sm_count = sms;
        slot.info.err_word = static_cast<uint32_t *>(err);
        slot.ok = true;
    });
    if (!slot.ok)
        return JETFP8_ERR_UNSUPPORTED_DEVICE;
    *out = &slot.info;
    return JETFP8_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;
};
Range range_of(const void *p, int64_t bytes)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, a + static_cast<uintptr_t>(bytes)};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

// outputs must not overlap inputs or each other
bool any_overlap(const Range *outs, int nout, const Range *ins, int nin)
{
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j)
            if (overlap(outs[i], ins[j]))
                return true;
        for (int j = i + 1; j < nout; ++j)
            if (overlap(outs[i], outs[j]))
                return true;
    }
    return false;
}

bool dims_ok(int64_t a, int64_t b) { return a <= kMaxDim && b <= kMaxDim && a * b < kMaxElems; }

jetfp8_status launch_status(cudaError_t e)
{
    if (e != cudaSuccess) {
        cudaGetLastError();
        return JETFP8_ERR_LAUNCH;
    }
    return JETFP8_OK;
}

jetfp8_status run_gemm(const jetfp8::GemmProblem &p, cudaStream_t stream)
{
    const DeviceInfo *dev = nullptr;
    jetfp8_status st = current_device(&dev);
    if (st != JETFP8_OK)
        return st;
    std::call_once(g_encode_once, init_encode);
    if (g_encode == nullptr)
        return JETFP8_ERR_UNSUPPORTED_DEVICE;
    return launch_status(jetfp8::launch_gemm(p, *dev, g_encode, stream));
}

// Common checks for the three GEMMs.  a: [ra][kd], b: [rb][kd] codes,
// scales given as byte ranges, d: bf16 [ra][rb].
jetfp8_status check_gemm(const void *a, const void *sa, const void *b, const void *sb, const void *d, int64_t ra,
                         int64_t rb, int64_t kd, int64_t sa_bytes, int64_t sb_bytes)
{
    if (!a || !sa || !b || !sb || !d)
        return JETFP8_ERR_INVALID_VALUE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || !aligned16(sa) || !aligned16(sb))
        return JETFP8_ERR_ALIGNMENT;
    const Range outs[1] = {range_of(d, ra * rb * 2)};
    const Range ins[4] = {range_of(a, ra * kd), range_of(b, rb * kd), range_of(sa, sa_bytes), range_of(sb, sb_bytes)};
    if (any_overlap(outs, 1, ins, 4))
        return JETFP8_ERR_INVALID_VALUE;
    return JETFP8_OK;
}

}  // namespace

extern "C" {

JETFP8_API size_t jetfp8_act_scale_count(int64_t rows, int64_t cols)
{
    if (rows < 0 || cols <= 0 || cols % 128 != 0 || !dims_ok(rows, cols))
        return 0;
    return static_cast<size_t>(cols / 128) * static_cast<size_t>(rows);
}

JETFP8_API const char *jetfp8_status_string(jetfp8_status status)
{
    switch (status) {
    case JETFP8_OK: return "JETFP8_OK";
    case JETFP8_ERR_INVALID_VALUE: return "JETFP8_ERR_INVALID_VALUE: null pointer or overlapping buffers";
    case JETFP8_ERR_SHAPE: return "JETFP8_ERR_SHAPE: unsupported or invalid size";
    case JETFP8_ERR_ALIGNMENT: return "JETFP8_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case JETFP8_ERR_UNSUPPORTED_DEVICE: return "JETFP8_ERR_UNSUPPORTED_DEVICE: needs a CUDA device of compute capability 10.3";
    case JETFP8_ERR_LAUNCH: return "JETFP8_ERR_LAUNCH: the CUDA runtime reported an error";
    case JETFP8_ERR_TIMEOUT: return "JETFP8_ERR_TIMEOUT: a kernel's bounded wait gave up";
    }
    return "JETFP8: unknown status";
}

JETFP8_API jetfp8_status jetfp8_quantize_act(const void *x, int64_t M, int64_t K, uint8_t *q, float *s, void *stream)
{
    if (M < 0 || K <= 0 || K % 128 != 0 || !dims_ok(M, K) || (K + 1023) / 1024 > 65535)   // grid y = ceil(K / 1024)
        return JETFP8_ERR_SHAPE;
    if (M == 0)
        return JETFP8_OK;
    if (!x || !q || !s)
        return JETFP8_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s))
        return JETFP8_ERR_ALIGNMENT;
    const Range outs[2] = {range_of(q, M * K), range_of(s, M * (K / 128) * 4)};
    const Range ins[1] = {range_of(x, M * K * 2)};
    if (any_overlap(outs, 2, ins, 1))
        return JETFP8_ERR_INVALID_VALUE;
    const DeviceInfo *dev = nullptr;
    jetfp8_status st = current_device(&dev);
    if (st != JETFP8_OK)
        return st;
    return launch_status(jetfp8::launch_quantize_act(x, M, K, q, s, static_cast<cudaStream_t>(stream)));
}

JETFP8_API jetfp8_status jetfp8_quantize_act_transposed(const void *x, int64_t M, int64_t C, uint8_t *qt, float *st,
                                                        void *stream)
{
    if (M < 0 || M % 128 != 0 || C <= 0 || C % 128 != 0 || !dims_ok(M, C) || C / 64 > 65535)
        return JETFP8_ERR_SHAPE;
    if (M == 0)
        return JETFP8_OK;
    if (!x || !qt || !st)
        return JETFP8_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(qt) || !aligned16(st))
        return JETFP8_ERR_ALIGNMENT;
    const Range outs[2] = {range_of(qt, M * C), range_of(st, (M / 128) * C * 4)};
    const Range ins[1] = {range_of(x, M * C * 2)};
    if (any_overlap(outs, 2, ins, 1))
        return JETFP8_ERR_INVALID_VALUE;
    const DeviceInfo *dev = nullptr;
    jetfp8_status status = current_device(&dev);
    if (status != JETFP8_OK)
        return status;
    return launch_status(
        jetfp8::launch_quantize_act_transposed(x, M, C, qt, st, static_cast<cudaStream_t>(stream)));
}

JETFP8_API jetfp8_status jetfp8_quantize_act_dual(const void *x, int64_t M, int64_t K, uint8_t *q, float *s,
                                                  uint8_t *qt, float *st, void *stream)
{
    if (M < 0 || M % 128 != 0 || K <= 0 || K % 128 != 0 || !dims_ok(M, K) || K / 128 > 65535)
        return JETFP8_ERR_SHAPE;
    if (M == 0)
        return JETFP8_OK;
    if (!x || !q || !s || !qt || !st)
        return JETFP8_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s) || !aligned16(qt) || !aligned16(st))
        return JETFP8_ERR_ALIGNMENT;
    const Range outs[4] = {range_of(q, M * K), range_of(s, M * (K / 128) * 4), range_of(qt, M * K),
                           range_of(st, (M / 128) * K * 4)};
    const Range ins[1] = {range_of(x, M * K * 2)};
    if (any_overlap(outs, 4, ins, 1))
        return JETFP8_ERR_INVALID_VALUE;
    const DeviceInfo *dev = nullptr;
    jetfp8_status status = current_device(&dev);
    if (status != JETFP8_OK)
        return status;
    std::call_once(g_encode_once, init_encode);
    if (g_encode == nullptr)
        return JETFP8_ERR_UNSUPPORTED_DEVICE;
    return launch_status(jetfp8::launch_quantize_act_dual(x, M, K, q, s, qt, st, g_encode, dev->err_word,
                                                          static_cast<cudaStream_t>(stream)));
}

JETFP8_API jetfp8_status jetfp8_e4m3_encode_range(uint32_t first, int64_t count, uint8_t *codes, void *stream)
{
    if (count < 0 || count > (int64_t{1} << 32) - static_cast<int64_t>(first))
        return JETFP8_ERR_SHAPE;
    if (count == 0)
        return JETFP8_OK;
    if (!codes)
        return JETFP8_ERR_INVALID_VALUE;
    if (!aligned16(codes))
        return JETFP8_ERR_ALIGNMENT;
    const DeviceInfo *dev = nullptr;
    jetfp8_status status = current_device(&dev);
    if (status != JETFP8_OK)
        return status;
    return launch_status(
        jetfp8::launch_e4m3_encode_range(first, count, codes, dev->sm_count, static_cast<cudaStream_t>(stream)));
}

namespace {
// One weight tensor's host-side checks (shared by the single and grouped calls).
jetfp8_status check_weight(const void *w, int64_t N, int64_t K, uint8_t *q, float *s, uint8_t *qt)
{
    if (N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0 || !dims_ok(N, K) || K / 128 > 65535 ||
        N / 128 > 65535)
        return JETFP8_ERR_SHAPE;
    if (!w || !q || !s)
        return JETFP8_ERR_INVALID_VALUE;
    if (!aligned16(w) || !aligned16(q) || !aligned16(s) || (qt && !aligned16(qt)))
        return JETFP8_ERR_ALIGNMENT;
    const Range outs[3] = {range_of(q, N * K), range_of(s, (N / 128) * (K / 128) * 4),
                           range_of(qt, qt ? N * K : 0)};
    const Range ins[1] = {range_of(w, N * K * 2)};
    if (any_overlap(outs, qt ? 3 : 2, ins, 1))
        return JETFP8_ERR_INVALID_VALUE;
    return JETFP8_OK;
}
}  // namespace

JETFP8_API jetfp8_status jetfp8_quantize_weight(const void *w, int64_t N, int64_t K, uint8_t *q, float *s,
                                                uint8_t *qt, void *stream)
{
    const jetfp8_status chk = check_weight(w, N, K, q, s, qt);
    if (chk != JETFP8_OK)
        return chk;
    const DeviceInfo *dev = nullptr;
    jetfp8_status st = current_device(&dev);
    if (st != JETFP8_OK)
        return st;
    std::call_once(g_encode_once, init_encode);
    if (g_encode == nullptr)
        return JETFP8_ERR_UNSUPPORTED_DEVICE;
    return launch_status(jetfp8::launch_quantize_weight(w, N, K, q, s, qt, g_encode, dev->err_word, dev->sm_count,
                                                        static_cast<cudaStream_t>(stream)));
}

JETFP8_API jetfp8_status jetfp8_quantize_weight_group(int count, const void *const *w, const int64_t *N,
                                                      const int64_t *K, uint8_t *const *q, float *const *s,
                                                      uint8_t *const *qt, void *stream)
{
    if (count < 0 || count > JETFP8_WEIGHT_GROUP_MAX)
        return JETFP8_ERR_SHAPE;
    if (count == 0)
        return JETFP8_OK;
    if (!w || !N || !K || !q || !s || !qt)
        return JETFP8_ERR_INVALID_VALUE;
    for (int t = 0; t < count; ++t) {
        const jetfp8_status chk = check_weight(w[t], N[t], K[t], q[t], s[t], qt[t]);
        if (chk != JETFP8_OK)
            return chk;
    }
    // no output of one entry may overlap an input or output of another
    for (int t = 0; t < count; ++t) {
        const Range outs[3] = {range_of(q[t], N[t] * K[t]), range_of(s[t], (N[t] / 128) * (K[t] / 128) * 4),
                               range_of(qt[t], qt[t] ? N[t] * K[t] : 0)};
        for (int u = 0; u < count; ++u) {
            if (u == t)
                continue;
            const Range others[4] = {range_of(w[u], N[u] * K[u] * 2), range_of(q[u], N[u] * K[u]),
                                     range_of(s[u], (N[u] / 128) * (K[u] / 128) * 4),
                                     range_of(qt[u], qt[u] ? N[u] * K[u] : 0)};
            if (any_overlap(outs, qt[t] ? 3 : 2, others, qt[u] ? 4 : 3))
                return JETFP8_ERR_INVALID_VALUE;
        }
    }
    const DeviceInfo *dev = nullptr;
    jetfp8_status st = current_device(&dev);
    if (st != JETFP8_OK)
        return st;
    std::call_once(g_encode_once, init_encode);
    if (g_encode == nullptr)
        return JETFP8_ERR_UNSUPPORTED_DEVICE;
    return launch_status(jetfp8::launch_quantize_weight_group(count, w, N, K, q, s, qt, g_encode, dev->err_word,
                                                              dev->sm_count, static_cast<cudaStream_t>(stream)));
}

JETFP8_API jetfp8_status jetfp8_rmsnorm_quantize_act(const void *x, const void *gamma, float eps, int64_t M,
                                                     int64_t H, uint8_t *q, float *s, void *y, void *stream)
{
    if (M < 0 || H <= 0 || H % 256 != 0 || !dims_ok(M, H) || (M + 7) / 8 > 0x7fffffff)
        return JETFP8_ERR_SHAPE;
    if (!(eps >= 0.0f) || eps > 3.4e38f)                 // NaN, negative and infinite eps rejected
        return JETFP8_ERR_INVALID_VALUE;
    if (M == 0)
        return JETFP8_OK;
    if (!x || !gamma || (q == nullptr) != (s == nullptr) || (!q && !y))
        return JETFP8_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(gamma) || (q && (!aligned16(q) || !aligned16(s))) || (y && !aligned16(y)))
        return JETFP8_ERR_ALIGNMENT;
    const Range outs[3] = {range_of(q, q ? M * H : 0), range_of(s, s ? M * (H / 128) * 4 : 0),
                           range_of(y, y ? M * H * 2 : 0)};
    const Range ins[2] = {range_of(x, M * H * 2), range_of(gamma, H * 2)};
    if (any_overlap(outs, 3, ins, 2))
        return JETFP8_ERR_INVALID_VALUE;
    const DeviceInfo *dev = nullptr;
    jetfp8_status st = current_device(&dev);
    if (st != JETFP8_OK)
        return st;
    return launch_status(
        jetfp8::launch_rmsnorm_quantize(x, gamma, eps, M, H, q, s, y, static_cast<cudaStream_t>(stream)));
}

JETFP8_API jetfp8_status jetfp8_swiglu_quantize_act(const void *gu, int64_t M, int64_t I, uint8_t *q, float *s,
                                                    void *y, void *stream)
{
    if (M < 0 || I <= 0 || I % 256 != 0 || !dims_ok(M, 2 * I))
        return JETFP8_ERR_SHAPE;
    if (M == 0)
        return JETFP8_OK;
    if (!gu || (q == nullptr) != (s == nullptr) || (!q && !y))
        return JETFP8_ERR_INVALID_VALUE;
    if (!aligned16(gu) || (q && (!aligned16(q) || !aligned16(s))) || (y && !aligned16(y)))
        return JETFP8_ERR_ALIGNMENT;
    const Range outs[3] = {range_of(q, q ? M * I : 0), range_of(s, s ? M * (I / 128) * 4 : 0),
                           range_of(y, y ? M * I * 2 : 0)};
    const Range ins[1] = {range_of(gu, M * I * 4)};
    if (any_overlap(outs, 3, ins, 1))
        return JETFP8_ERR_INVALID_VALUE;
    const DeviceInfo *dev = nullptr;
    jetfp8_status st = current_device(&dev);
    if (st != JETFP8_OK)
        return st;
    return launch_status(jetfp8::launch_swiglu_quantize(gu, M, I, q, s, y, dev->sm_count,
                                                        static_cast<cudaStream_t>(stream)));
}

JETFP8_API jetfp8_status jetfp8_gemm_fprop(const uint8_t *qx, const float *sx, const uint8_t *qw, const float *sw,
                                           void *y, int64_t M, int64_t N, int64_t K, void *stream)
{
    if (M < 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0 || !dims_ok(M, K) || !dims_ok(N, K) ||
        !dims_ok(M, N))
        return JETFP8_ERR_SHAPE;
    if (M == 0)
        return JETFP8_OK;
    jetfp8_status st = check_gemm(qx, sx, qw, sw, y, M, N, K, (K / 128) * M * 4, (N / 128) * (K / 128) * 4);
    if (st != JETFP8_OK)
        return st;
    jetfp8::GemmProblem p{};
    p.a = qx;
    p.b = qw;
    p.sa = sx;
    p.sb = sw;
    p.sb_mode = jetfp8::ScaleB::PerBlock128;
    p.sb_stride_g = 1;          // sw[n/128][g]
    p.sb_stride_c = K / 128;
    p.d = y;
    p.rows = M;
    p.cols = N;
    p.kdim = K;
    return run_gemm(p, static_cast<cudaStream_t>(stream));
}

JETFP8_API jetfp8_status jetfp8_gemm_dgrad(const uint8_t *qdy, const float *sdy, const uint8_t *qwt, const float *sw,
                                           void *dx, int64_t M, int64_t N, int64_t K, void *stream)
{
    if (M < 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0 || !dims_ok(M, K) || !dims_ok(N, K) ||
        !dims_ok(M, N))
        return JETFP8_ERR_SHAPE;
    if (M == 0)
        return JETFP8_OK;
    jetfp8_status st = check_gemm(qdy, sdy, qwt, sw, dx, M, K, N, (N / 128) * M * 4, (N / 128) * (K / 128) * 4);
    if (st != JETFP8_OK)
        return st;
    jetfp8::GemmProblem p{};
    p.a = qdy;                  // [M][N], contraction over N
    p.b = qwt;                  // [K][N]
    p.sa = sdy;                 // [N/128][M]
    p.sb = sw;                  // sw[g][k/128]
    p.sb_mode = jetfp8::ScaleB::PerBlock128;
    p.sb_stride_g = K / 128;
    p.sb_stride_c = 1;
    p.d = dx;
    p.rows = M;
    p.cols = K;
    p.kdim = N;
    return run_gemm(p, static_cast<cudaStream_t>(stream));
}

JETFP8_API jetfp8_status jetfp8_gemm_wgrad(const uint8_t *qdyt, const float *sdyt, const uint8_t *qxt,
                                           const float *sxt, void *dw, int64_t M, int64_t N, int64_t K,
                                           void *stream)
{
    if (M < 0 || M % 128 != 0 || N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0 || !dims_ok(M, K) ||
        !dims_ok(N, K) || !dims_ok(M, N))
        return JETFP8_ERR_SHAPE;
    if (M == 0)
        return JETFP8_OK;
    jetfp8_status st = check_gemm(qdyt, sdyt, qxt, sxt, dw, N, K, M, (M / 128) * N * 4, (M / 128) * K * 4);
    if (st != JETFP8_OK)
        return st;
    jetfp8::GemmProblem p{};
    p.a = qdyt;                 // [N][M]
    p.b = qxt;                  // [K][M]
    p.sa = sdyt;                // [M/128][N]
    p.sb = sxt;                 // [M/128][K]
    p.sb_mode = jetfp8::ScaleB::PerColumn;
    p.sb_stride_g = K;
    p.sb_stride_c = 1;
    p.d = dw;
    p.rows = N;
    p.cols = K;
    p.kdim = M;
    return run_gemm(p, static_cast<cudaStream_t>(stream));
}

JETFP8_API jetfp8_status jetfp8_poll_device_error(void *stream)
{
    const DeviceInfo *dev = nullptr;
    jetfp8_status st = current_device(&dev);
    if (st != JETFP8_OK)
        return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return JETFP8_ERR_LAUNCH;
    }
    uint32_t word = 0;
    if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof word) != cudaSuccess) {
        cudaGetLastError();
        return JETFP8_ERR_LAUNCH;
    }
    if (word != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) {
            cudaGetLastError();
            return JETFP8_ERR_LAUNCH;
        }
        return JETFP8_ERR_TIMEOUT;
    }
    return JETFP8_OK;
}

JETFP8_API jetfp8_status jetfp8_watchdog_selftest(int64_t timeout_us, void *stream)
{
    if (timeout_us < 1 || timeout_us > 1000000)
        return JETFP8_ERR_SHAPE;
    const DeviceInfo *dev = nullptr;
    jetfp8_status st = current_device(&dev);
    if (st != JETFP8_OK)
        return st;
    return launch_status(jetfp8::launch_watchdog_selftest(dev->err_word, static_cast<uint64_t>(timeout_us) * 1000u,
                                                          static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
