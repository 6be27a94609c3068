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
// domain).  The kernels evaluate them in fp32 in a fixed order, so a
// row's result never depends on the launch or on the other rows; the bf16
// value (nearest even) is then quantised exactly as jetfp8_quantize_act
// quantises it, and the optional bf16 output is that same value.
//
// Layout of the work: a 1x128 group (sixteen 16-byte pieces) is held by four
// neighbouring lanes, lane l of the four holding pieces l, l + 4, l + 8 and
// l + 12 (its "quad", 32 values): the group's amax takes two shuffles, its
// scale is computed once per 32 values, and each load or store instruction
// of a warp touches eight 64-byte runs (eight cache lines) instead of
// sixteen lines for a lane holding four consecutive pieces -- the cache's
// request throughput, not DRAM, was the tighter limit.  (Rows wider than
// 32768 columns fall back to eight values per lane, a group per half-warp.)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "e4m3.cuh"
#include "internal.cuh"

namespace jetfp8 {
namespace {

constexpr int PR_THREADS = 256;
constexpr int PR_WARPS = PR_THREADS / 32;

// Hardware approximations of 2^x and 1/x (deterministic; the relative
// error of each is a few fp32 ulps), in their flush-to-zero forms, which need
// no extra instructions around the hardware unit.  In the sigmoid
// 1 / (1 + 2^a) that changes nothing above gates of about -87.3: a subnormal
// a gives 2^a = 1 either way, a subnormal 2^a vanishes next to the 1 it is
// added to, and the reciprocal's argument is at least 1.  Below, the
// sigmoid itself would be subnormal and is 0 instead -- within the bound
// stated for gates below -87.
__device__ __forceinline__ float ex2_approx(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
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

// The same for 32 values (four 16-byte vectors' worth).
__device__ __forceinline__ void round_bf16x32(const float (&v)[32], uint32_t (&w)[16], float (&r)[32])
{
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t *>(&h);
        r[2 * k] = bf16_lo(w[k]);
        r[2 * k + 1] = bf16_hi(w[k]);
    }
}

// ---------------------------------------------------------------------------
// RMSNorm.  The sum of squares of a row: each thread adds, in order, the
// squares of its values (even and odd values in two chains, added at the
// end; with one warp per row, a single chain); the lanes of a warp combine by
// butterfly (partner distance 16, 8, 4, 2, 1); the warps of the row then add
// up in warp order.  y = bf16((x * rstd) * gamma) is then quantised per 1x128
// group.  Rows of up to RN_REG_MAX_H columns: up to sixteen warps per row,
// each thread's quads held in registers between the two steps, so the row is
// read from memory once.  Wider rows: one warp per row, the row read a
// second time (from cache).
// ---------------------------------------------------------------------------
constexpr int RN_MAX_THREADS = 512;           // up to sixteen warps per row
constexpr int64_t RN_REG_MAX_H = 32768;      // sixteen warps of two quads (32 values each) per row

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

__device__ __forceinline__ uint64_t sum_squares8x2(uint64_t acc2, const uint4 &c)
{
    float f[8];
    unpack8(c, f);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const uint64_t x2 = ptx::pack_f32x2(f[e], f[e + 1]);
        ptx::fma_f32x2(acc2, x2, x2);
    }
    return acc2;
}

// 1 / sqrt(sum_sq / H + eps) from the hardware reciprocal and reciprocal square
// root (each within about an fp32 ulp): a few instructions instead of two
// correctly rounded divisions and a square root per row and thread, and an
// error near 2^-21 relative, far inside the one-bf16-ulp (2^-8) bound on y.
__device__ __forceinline__ float rms_rstd(float sum_sq, int64_t H, float eps)
{
    float inv_h, r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(inv_h) : "f"(static_cast<float>(H)));
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__fadd_rn(__fmul_rn(sum_sq, inv_h), eps)));
    return r;
}

// y = bf16((x * rstd) * gamma) of one 16-byte chunk c (eight values) of a
// row: stored to y and / or quantised (the chunk's half-warp is its group)
__device__ __forceinline__ void rms_chunk_out(const uint4 &xc, const uint4 &gc, float rstd, int64_t row, int64_t c,
                                              int64_t M, int64_t H, uint8_t *__restrict__ q, float *__restrict__ s,
                                              uint4 *__restrict__ y, int lane)
{
    float f[8], g[8], u[8], v[8];
    unpack8(xc, f);
    unpack8(gc, g);
    // (x * rstd) * gamma, two values per packed multiply (each lane rounded
    // as the scalar multiply)
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
        y[row * (H >> 3) + c] = make_uint4(w[0], w[1], w[2], w[3]);
    if (q)
        quantize8_halfwarp(v, w, q + row * H + 8 * c, s + (c >> 4) * M + row, lane);
}

// y = bf16((x * rstd) * gamma) of one quad of a row: the pieces p0 + 4k
// (k = 0..3, xq and gq) of the group p0 >> 4, stored to y and / or quantised
// (the group's four lanes are neighbours in the warp).  Every lane of the
// warp takes part; a lane whose quad is past the row's end (`live` false)
// stores nothing.
__device__ __forceinline__ void rms_quad_out(const uint4 (&xq)[4], const uint4 (&gq)[4], bool live,
                                             float rstd, int64_t row, int64_t p0, int64_t M, int64_t H,
                                             uint8_t *__restrict__ q, float *__restrict__ s,
                                             uint4 *__restrict__ y, int lane)
{
    const uint64_t r2 = ptx::pack_f32x2(rstd, rstd);
    float u[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float f[8], g[8];
        unpack8(xq[k], f);
        unpack8(gq[k], g);
        // (x * rstd) * gamma, two values per packed multiply (each lane
        // rounded as the scalar multiply)
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const uint64_t xr2 = ptx::mul_f32x2(ptx::pack_f32x2(f[e], f[e + 1]), r2);
            const uint64_t y2 = ptx::mul_f32x2(xr2, ptx::pack_f32x2(g[e], g[e + 1]));
            u[8 * k + e] = ptx::lo_f32(y2);
            u[8 * k + e + 1] = ptx::hi_f32(y2);
        }
    }
    uint32_t w[16];
    float v[32];
    round_bf16x32(u, w, v);
    if (y && live) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            y[row * (H >> 3) + p0 + 4 * k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
    if (q)
        quantize32_quad<32>(v, w, live, q + row * H + 8 * p0, s + (p0 >> 4) * M + row, lane);
}

// first piece of quad qd: group qd >> 2, lane qd & 3 of the group's four
__device__ __forceinline__ int64_t quad_first_piece(int64_t qd)
{
    return 16 * (qd >> 2) + (qd & 3);
}

// A row is taken by `rw` warps (32 rw threads: thread t holds quads t,
// t + 32 rw, ...), 8 / rw rows per block (integer division; one when rw > 4);
// each thread holds at most JQ quads, so the row is read from memory once.
// (With one quad per thread, capped at 64 registers: more resident warps hide
// the loads better than a larger register budget; measured.)
template <int JQ>
__global__ void __launch_bounds__(RN_MAX_THREADS, JQ == 1 ? 2 : 1)
rmsnorm_quantize_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ gamma, float eps, int64_t M,
                        int64_t H, int rw, uint8_t *__restrict__ q, float *__restrict__ s, uint4 *__restrict__ y)
{
    __shared__ float part[RN_MAX_THREADS / 32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int row_threads = 32 * rw;
    const int t = threadIdx.x % row_threads;
    const int r_in_block = threadIdx.x / row_threads;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / row_threads) + r_in_block;
    const bool live = row < M;                    // no early exit: the block meets at a barrier
    const int64_t NQ = H >> 5;                    // quads per row (a multiple of 4: groups are whole)
    const uint4 *xr = x + (live ? row : 0) * (H >> 3);

    uint4 v[JQ][4];
#pragma unroll
    for (int j = 0; j < JQ; ++j) {
        const int64_t qd = t + static_cast<int64_t>(row_threads) * j;
        const int64_t p0 = quad_first_piece(qd);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            v[j][k] = live && qd < NQ ? __ldg(xr + p0 + 4 * k) : make_uint4(0u, 0u, 0u, 0u);
    }
    // squares summed as two interleaved fp32 chains (even and odd values,
    // one packed fused multiply-add per pair; zero-filled quads add +0),
    // then added
    uint64_t acc2 = 0ull;
#pragma unroll
    for (int j = 0; j < JQ; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            acc2 = sum_squares8x2(acc2, v[j][k]);
    float acc = __fadd_rn(ptx::lo_f32(acc2), ptx::hi_f32(acc2));
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1)
        acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, d));
    if (lane == 0)
        part[warp] = acc;
    __syncthreads();
    const int w0 = r_in_block * rw;               // the row's first warp
    float sum_sq = part[w0];
    for (int w = 1; w < rw; ++w)
        sum_sq = __fadd_rn(sum_sq, part[w0 + w]);
    if (!live)
        return;                                   // whole rows, so whole groups
    const float rstd = rms_rstd(sum_sq, H, eps);
#pragma unroll
    for (int j = 0; j < JQ; ++j) {
        const int64_t qd = t + static_cast<int64_t>(row_threads) * j;
        if ((t & ~31) + static_cast<int64_t>(row_threads) * j < NQ) {   // some lane of the warp is in the row
            const int64_t p0 = quad_first_piece(qd);
            uint4 g[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                g[k] = qd < NQ ? __ldg(gamma + p0 + 4 * k) : make_uint4(0u, 0u, 0u, 0u);
            rms_quad_out(v[j], g, qd < NQ, rstd, row, p0, M, H, q, s, y, lane);
        }
    }
}

__global__ void __launch_bounds__(PR_THREADS)
rmsnorm_quantize_wide_kernel(const uint4 *__restrict__ x, const uint4 *__restrict__ gamma, float eps, int64_t M,
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
    const float rstd = rms_rstd(acc, H, eps);
#pragma unroll 4
    for (int j = 0; j < nj; ++j) {
        const int64_t c = 32 * j + lane;
        rms_chunk_out(__ldg(xr + c), __ldg(gamma + c), rstd, row, c, M, H, q, s, y, lane);
    }
}

// ---------------------------------------------------------------------------
// SwiGLU of a gate_up output [M][2I] (gate = columns 0..I-1, up = I..2I-1):
// y = bf16( (g * (1 / (1 + e^-g))) * u ).  A warp handles four 256-column
// chunks per iteration, eight lanes (one quad each) per chunk, grid-stride
// over all chunks.
//
// Accuracy: -g log2 e is rounded once, which moves the exponent by at most
// 2^-24 |g log2 e| <= 2^-17 where 2^(-g log2 e) is finite and normal, i.e. a
// relative error below 2^-17.5 in e^-g; the hardware 2^x and 1/x add a few
// fp32 ulps each and the three roundings (1 + e^-g, g * sigmoid, * u) one
// ulp each.  The fp32 result is within 2^-16 of silu(g) u relative, well
// inside half a bf16 ulp (2^-9), so its bf16 rounding is within one bf16 ulp
// of the exact value.  Below g = -87 the reciprocal's result leaves fp32's
// normal range and ends at 0 (e^-g overflowing); there the exact value is
// below 2^-119 |u|.
// ---------------------------------------------------------------------------
constexpr float LOG2E = 1.44269502f;              // log2(e) rounded to fp32
__global__ void __launch_bounds__(PR_THREADS)
swiglu_quantize_kernel(const uint4 *__restrict__ gu, int64_t M, int64_t I, uint8_t *__restrict__ q,
                       float *__restrict__ s, uint4 *__restrict__ y)
{
    // A warp takes four 256-column chunks (items) per iteration, eight lanes
    // per chunk (its two 1x128 groups), each lane a quad: pieces c0 + 4j of
    // the output row (32 outputs).
    const int lane = threadIdx.x & 31;
    const int sub = lane & 7;                     // lane within its chunk's eight
    const int64_t chunks = I >> 8;                // 256-column chunks per row
    const int64_t items = M * chunks;
    const int64_t in_row = I >> 2;                // uint4 per gate_up row (2I bf16)
    const int64_t out_row = I >> 3;               // uint4 per output row
    const int64_t step = static_cast<int64_t>(gridDim.x) * PR_WARPS * 4;
    for (int64_t base = (static_cast<int64_t>(blockIdx.x) * PR_WARPS + (threadIdx.x >> 5)) * 4; base < items;
         base += step) {
        const int64_t it = base + (lane >> 3);
        const bool live = it < items;             // (a lane past the end still joins the group's shuffles)
        const int64_t row = live ? it / chunks : 0;
        const int64_t c0 = (live ? it - row * chunks : 0) * 32 + 16 * (sub >> 2) + (sub & 3);   // first piece
        float t[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float g[8], u[8];
            unpack8(__ldg(gu + row * in_row + c0 + 4 * j), g);
            unpack8(__ldg(gu + row * in_row + out_row + c0 + 4 * j), u);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                // sigmoid(g) = 1 / (1 + 2^(-g log2 e))
                const uint64_t a =
                    ptx::mul_f32x2(ptx::pack_f32x2(g[e], g[e + 1]), ptx::pack_f32x2(-LOG2E, -LOG2E));
                const float s0 = rcp_approx(__fadd_rn(1.0f, ex2_approx(ptx::lo_f32(a))));
                const float s1 = rcp_approx(__fadd_rn(1.0f, ex2_approx(ptx::hi_f32(a))));
                const uint64_t gs = ptx::mul_f32x2(ptx::pack_f32x2(g[e], g[e + 1]), ptx::pack_f32x2(s0, s1));
                const uint64_t tu = ptx::mul_f32x2(gs, ptx::pack_f32x2(u[e], u[e + 1]));
                t[8 * j + e] = ptx::lo_f32(tu);
                t[8 * j + e + 1] = ptx::hi_f32(tu);
            }
        }
        uint32_t w[16];
        float v[32];
        round_bf16x32(t, w, v);
        if (y && live) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                y[row * out_row + c0 + 4 * j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
        if (q)
            quantize32_quad<32>(v, w, live, q + row * I + 8 * c0, s + (c0 >> 4) * M + row, lane);
    }
}

}  // namespace

cudaError_t launch_rmsnorm_quantize(const void *x, const void *gamma, float eps, int64_t M, int64_t H, uint8_t *q,
                                    float *s, void *y, cudaStream_t stream)
{
    const uint4 *xv = static_cast<const uint4 *>(x);
    const uint4 *gv = static_cast<const uint4 *>(gamma);
    uint4 *yv = static_cast<uint4 *>(y);
    if (H > RN_REG_MAX_H) {
        const int64_t blocks = (M + PR_WARPS - 1) / PR_WARPS;
        rmsnorm_quantize_wide_kernel<<<static_cast<unsigned>(blocks), PR_THREADS, 0, stream>>>(xv, gv, eps, M, H, q,
                                                                                               s, yv);
        return cudaGetLastError();
    }
    // one quad per thread up to eight warps per row (8192 columns), else two
    // (sixteen warps of one quad measured slower at 16384 columns: 3.20
    // against 3.31 TB/s)
    const int64_t NQ = H >> 5;
    const int jq = NQ <= 256 ? 1 : 2;
    const int rw = static_cast<int>((NQ + 32 * jq - 1) / (32 * jq));
    const int rows = rw <= 4 ? PR_WARPS / rw : 1;
    const unsigned blocks = static_cast<unsigned>((M + rows - 1) / rows);
    const unsigned threads = static_cast<unsigned>(rows * rw * 32);
    if (jq == 1)
        rmsnorm_quantize_kernel<1><<<blocks, threads, 0, stream>>>(xv, gv, eps, M, H, rw, q, s, yv);
    else
        rmsnorm_quantize_kernel<2><<<blocks, threads, 0, stream>>>(xv, gv, eps, M, H, rw, q, s, yv);
    return cudaGetLastError();
}

cudaError_t launch_swiglu_quantize(const void *gu, int64_t M, int64_t I, uint8_t *q, float *s, void *y,
                                   int sm_count, cudaStream_t stream)
{
    const int64_t items = M * (I >> 8);
    const int64_t want = (items + 4 * PR_WARPS - 1) / (4 * PR_WARPS);   // four chunks per warp and iteration
    // one block per resident slot: a grid-stride loop over more blocks than
    // fit at once leaves a partial last round (measured: 6.23 -> 6.52 TB/s at
    // 16384 x 14336, 4.81 -> 5.15 at 2048 x 14336)
    static const int resident = [] {
        int bps = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, swiglu_quantize_kernel, PR_THREADS, 0) != cudaSuccess) {
            (void)cudaGetLastError();            // not a launch error: fall back to one block per SM
            bps = 1;
        }
        return bps < 1 ? 1 : bps;
    }();
    const int64_t cap = static_cast<int64_t>(sm_count) * resident;
    const int64_t blocks = want < cap ? want : cap;
    swiglu_quantize_kernel<<<static_cast<unsigned>(blocks), PR_THREADS, 0, stream>>>(
        static_cast<const uint4 *>(gu), M, I, q, s, static_cast<uint4 *>(y));
    return cudaGetLastError();
}

}  // namespace jetfp8
