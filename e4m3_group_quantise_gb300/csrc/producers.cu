// Producers fused in front of the FP8 linear layers: RMSNorm and SwiGLU that
// emit the next GEMM's 1x128 FP8 input directly (Jet-RL technical summaries,
// "Implémentation": fused activation / RMSNorm kernels feeding the FP8
// GEMMs), so the bf16 intermediate need not make a round trip through HBM.
//
// The pages give no arithmetic for these operators, so their textbook
// definitions are the contract: RMSNorm y = x / sqrt(mean(x^2) + eps) * gamma
// and SwiGLU y = silu(g) * u, each bf16 result within one bf16 ulp of the
// exact value (for gates below -87, where the fp32 sigmoid underflows, within
// 2^-119 |u|; rows whose sum of squares overflows fp32 are outside the
// domain).  The kernels evaluate them in fp32 in a fixed order (every
// operation one IEEE fp32 operation, written with the _rn intrinsics and
// fmaf so that nothing is contracted), so a row's result never depends on
// the launch or on the other rows; the bf16 value (nearest even) is then
// quantised exactly as jetfp8_quantize_act quantises it, and the optional
// bf16 output is that same value.
//
// Layout of the work: a warp takes a 256-column chunk of one row, lane l the
// eight values 8l .. 8l+7, loaded and stored as 16-byte vectors.  A 1x128
// group is then one half-warp: its amax takes four shuffles and its codes
// leave as one contiguous 128-byte store.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "e4m3.cuh"
#include "internal.cuh"

namespace jetfp8 {
namespace {

constexpr int PR_THREADS = 256;
constexpr int PR_WARPS = PR_THREADS / 32;

// 2^k for -126 <= k <= 127 (unsigned arithmetic: other k, from lanes whose
// result is discarded, give some bit pattern without overflow)
__device__ __forceinline__ float pow2_normal(int k)
{
    return __uint_as_float((static_cast<uint32_t>(k) + 127u) << 23);
}

// e^x in fp32 for two values at once: Cody-Waite range reduction
// x = n ln2 + r with n = rint(x / ln2), |r| <= ln2 / 2; e^r from its degree-7
// Taylor polynomial in Horner form with fused multiply-adds; then the scaling
// by 2^n in two exact steps.  ln2 is split into a head with 16 significant
// bits (45426 / 2^16, so n * head is exact) and the rounded remainder.
// x >= 89 gives +inf, x < -87 gives +0, NaN stays NaN.  Every multiply and
// fused multiply-add is one packed fp32x2 operation, whose lanes round
// exactly as the scalar operation would (fma(-n, c, x) is written
// fma(n, -c, x): the same product, the same rounding); lanes outside the
// range are replaced at the end.
__device__ __forceinline__ void exp_f32x2(float x0, float x1, float &e0, float &e1)
{
    using namespace ptx;
    auto dup = [](float c) { return pack_f32x2(c, c); };
    const uint64_t x = pack_f32x2(x0, x1);
    const uint64_t t = mul_f32x2(x, dup(1.44269502f));
    const float n0 = rintf(lo_f32(t)), n1 = rintf(hi_f32(t));
    const uint64_t n = pack_f32x2(n0, n1);
    uint64_t r = fma2_f32x2(n, dup(-0.693145751953125f), x);
    r = fma2_f32x2(n, dup(-1.42860677e-06f), r);
    uint64_t p = fma2_f32x2(dup(0.000198412701f), r, dup(0.00138888892f));
    p = fma2_f32x2(p, r, dup(0.00833333377f));
    p = fma2_f32x2(p, r, dup(0.0416666679f));
    p = fma2_f32x2(p, r, dup(0.166666672f));
    p = fma2_f32x2(p, r, dup(0.5f));
    p = fma2_f32x2(p, r, dup(1.0f));
    p = fma2_f32x2(p, r, dup(1.0f));
    const int i0 = __float2int_rz(n0), i1 = __float2int_rz(n1);   // exact in range, saturating outside
    const int h0 = i0 / 2, h1 = i1 / 2;
    const uint64_t s1 = pack_f32x2(pow2_normal(h0), pow2_normal(h1));
    const uint64_t s2 = pack_f32x2(pow2_normal(i0 - h0), pow2_normal(i1 - h1));
    const uint64_t e = mul_f32x2(mul_f32x2(p, s1), s2);
    auto fix = [](float xv, float ev) {
        if (xv != xv)
            return xv;
        if (xv >= 89.0f)
            return __int_as_float(0x7f800000);
        if (xv < -87.0f)
            return 0.0f;
        return ev;
    };
    e0 = fix(x0, lo_f32(e));
    e1 = fix(x1, hi_f32(e));
}

// Round eight fp32 values to bf16 (nearest even), two per conversion: the
// bf16 words (value 2k in the low half of word k) and their fp32 values.
__device__ __forceinline__ void round_bf16x8(const float (&v)[8], uint32_t (&w)[4], float (&r)[8])
{
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t *>(&h);
        r[2 * k] = bf16_lo(w[k]);
        r[2 * k + 1] = bf16_hi(w[k]);
    }
}

// ---------------------------------------------------------------------------
// RMSNorm: one warp per row.  Pass 1 sums the squares: lane l adds, in order,
// the squares of its chunks' values (chunk 32 j + l, j = 0, 1, ...), then the
// lanes combine by butterfly (partner distance 16, 8, 4, 2, 1).  Pass 2
// re-reads the row (from cache), forms y = bf16((x * rstd) * gamma) and
// quantises it.  Both passes are unrolled four chunks deep so that each warp
// keeps several loads in flight; the additions stay in chunk order.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float sum_squares8(float acc, const uint4 &c)
{
    float f[8];
    unpack8(c, f);
    // x^2 of a bf16 value is exact in fp32, so the fused multiply-add rounds
    // exactly as the separate multiply and add would
#pragma unroll
    for (int e = 0; e < 8; ++e)
        acc = fmaf(f[e], f[e], acc);
    return acc;
}

__global__ void __launch_bounds__(PR_THREADS)
rmsnorm_quantize_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ gamma, float eps, int64_t M,
                        int64_t H, uint8_t *__restrict__ q, float *__restrict__ s, uint4 *__restrict__ y)
{
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * PR_WARPS + (threadIdx.x >> 5);
    if (row >= M)
        return;                                   // whole warps only
    const int64_t H8 = H >> 3;
    const uint4 *xr = x + row * H8;
    const int nj = static_cast<int>(H >> 8);

    float acc = 0.0f;
#pragma unroll 4
    for (int j = 0; j < nj; ++j)
        acc = sum_squares8(acc, __ldg(xr + 32 * j + lane));
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1)
        acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, d));
    const float ms = __fdiv_rn(acc, static_cast<float>(H));
    const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));

#pragma unroll 4
    for (int j = 0; j < nj; ++j) {
        const int64_t c = 32 * j + lane;
        float f[8], g[8], u[8], v[8];
        unpack8(__ldg(xr + c), f);
        unpack8(__ldg(gamma + c), g);
        // (x * rstd) * gamma, two values per packed multiply (each lane
        // rounded as the scalar multiply)
        const uint64_t r2 = ptx::pack_f32x2(rstd, rstd);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const uint64_t xr2 = ptx::mul_f32x2(ptx::pack_f32x2(f[e], f[e + 1]), r2);
            const uint64_t y2 = ptx::mul_f32x2(xr2, ptx::pack_f32x2(g[e], g[e + 1]));
            u[e] = ptx::lo_f32(y2);
            u[e + 1] = ptx::hi_f32(y2);
        }
        uint32_t w[4];
        round_bf16x8(u, w, v);
        if (y)
            y[row * H8 + c] = make_uint4(w[0], w[1], w[2], w[3]);
        if (q)
            quantize8_halfwarp(v, q + row * H + 8 * c, s + (c >> 4) * M + row, lane);
    }
}

// ---------------------------------------------------------------------------
// SwiGLU of a gate_up output [M][2I] (gate = columns 0..I-1, up = I..2I-1):
// y = bf16( (g * (1 / (1 + e^-g))) * u ).  A warp handles one 256-column
// chunk of one row per iteration (grid-stride over all chunks).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(PR_THREADS)
swiglu_quantize_kernel(const uint4 *__restrict__ gu, int64_t M, int64_t I, uint8_t *__restrict__ q,
                       float *__restrict__ s, uint4 *__restrict__ y)
{
    const int lane = threadIdx.x & 31;
    const int64_t chunks = I >> 8;
    const int64_t items = M * chunks;
    const int64_t in_row = I >> 2;                // uint4 per gate_up row (2I bf16)
    const int64_t out_row = I >> 3;               // uint4 per output row
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * PR_WARPS + (threadIdx.x >> 5); it < items;
         it += static_cast<int64_t>(gridDim.x) * PR_WARPS) {
        const int64_t row = it / chunks;
        const int64_t c = (it - row * chunks) * 32 + lane;   // output uint4 index within the row
        float g[8], u[8], t[8], v[8];
        unpack8(__ldg(gu + row * in_row + c), g);
        unpack8(__ldg(gu + row * in_row + out_row + c), u);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            // 1 / (1 + e^-g): the correctly rounded reciprocal is the IEEE quotient
            float x0, x1;
            exp_f32x2(-g[e], -g[e + 1], x0, x1);
            const float s0 = __frcp_rn(__fadd_rn(1.0f, x0)), s1 = __frcp_rn(__fadd_rn(1.0f, x1));
            const uint64_t gs = ptx::mul_f32x2(ptx::pack_f32x2(g[e], g[e + 1]), ptx::pack_f32x2(s0, s1));
            const uint64_t tu = ptx::mul_f32x2(gs, ptx::pack_f32x2(u[e], u[e + 1]));
            t[e] = ptx::lo_f32(tu);
            t[e + 1] = ptx::hi_f32(tu);
        }
        uint32_t w[4];
        round_bf16x8(t, w, v);
        if (y)
            y[row * out_row + c] = make_uint4(w[0], w[1], w[2], w[3]);
        if (q)
            quantize8_halfwarp(v, q + row * I + 8 * c, s + (c >> 4) * M + row, lane);
    }
}

}  // namespace

cudaError_t launch_rmsnorm_quantize(const void *x, const void *gamma, float eps, int64_t M, int64_t H, uint8_t *q,
                                    float *s, void *y, cudaStream_t stream)
{
    const int64_t blocks = (M + PR_WARPS - 1) / PR_WARPS;
    rmsnorm_quantize_kernel<<<static_cast<unsigned>(blocks), PR_THREADS, 0, stream>>>(
        static_cast<const uint4 *>(x), static_cast<const uint4 *>(gamma), eps, M, H, q, s, static_cast<uint4 *>(y));
    return cudaGetLastError();
}

cudaError_t launch_swiglu_quantize(const void *gu, int64_t M, int64_t I, uint8_t *q, float *s, void *y,
                                   int sm_count, cudaStream_t stream)
{
    const int64_t items = M * (I >> 8);
    const int64_t want = (items + PR_WARPS - 1) / PR_WARPS;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;    // 8 resident blocks per SM
    const int64_t blocks = want < cap ? want : cap;
    swiglu_quantize_kernel<<<static_cast<unsigned>(blocks), PR_THREADS, 0, stream>>>(
        static_cast<const uint4 *>(gu), M, I, q, s, static_cast<uint4 *>(y));
    return cudaGetLastError();
}

}  // namespace jetfp8
