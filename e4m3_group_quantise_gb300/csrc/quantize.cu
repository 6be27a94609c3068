// Group-wise FP8 (E4M3) quantisers for sm_103a.
//
// Jet-RL (technical summaries on gist.science, "Schéma de Quantification"):
// activations and gradients use 1x128 groups, weights 128x128 blocks, and the
// WGrad operands 1x128 / 128x1 groups, read here as groups of 128 tokens
// along the token axis, which the transposed quantiser writes out as 1x128
// groups of the transposed tensor.  Per group: amax = max |x|, s = amax / 448 (IEEE fp32
// division), code = E4M3(RNE, saturating)(x / s) (IEEE fp32 division); a
// zero group stores s = 0 and codes 0x00.
//
// All three kernels are HBM-streaming: 16-byte vector loads, warp-shuffle
// amax reductions, and stores arranged so that every written sector is full.
// Compiled without fast-math so that `/` is the correctly rounded IEEE
// division and subnormals are kept; the per-element division itself is
// replaced by a once-corrected quotient whose codes are exact on the inputs
// met here (e4m3.cuh), with the division for the rest (tiny or infinite
// scales, -0 inputs).
#include <cuda_runtime.h>
#include <cstdint>

#include "e4m3.cuh"
#include "internal.cuh"
#include "ptx.cuh"

namespace jetfp8 {
namespace {

// ---------------------------------------------------------------------------
// 1x128 groups along rows.  CTA tile: 16 rows x 8 groups (1024 columns).
// Warp w owns group g0 + w of 8 rows at a time; four lanes share a group
// (lane = 4 * row + sub), each holding 32 values: 16-byte chunks sub, sub+4,
// sub+8, sub+12 of the group's 256 bytes.  Every load instruction reads 64
// contiguous bytes per row, every code store writes 32 (one full sector),
// and the 8 rows' scales of one group are contiguous (group-major), so
// lanes with sub == 0 store them as one 32-byte sector -- no shared memory.
// The amax needs two shuffles; the scale arithmetic is shared by 32 values.
// ---------------------------------------------------------------------------
// Four bf16 values (word k, k = 0..7) of a lane's 32 held as four 16-byte
// chunks: chunk k / 2, half k % 2; picked by selects, so the rare exact path
// needs neither a memory access nor an indexed register array.
__device__ __forceinline__ uint2 pick_word(const uint4 (&v)[4], int k)
{
    uint2 r = make_uint2(v[0].x, v[0].y);
#pragma unroll
    for (int i = 1; i < 8; ++i) {
        const uint4 &c = v[i >> 1];
        const uint2 cand = (i & 1) ? make_uint2(c.z, c.w) : make_uint2(c.x, c.y);
        r = (k == i) ? cand : r;
    }
    return r;
}

constexpr int Q1_ROWS = 16;
constexpr int Q1_GROUPS = 8;
constexpr int Q1_THREADS = 256;

__global__ void __launch_bounds__(Q1_THREADS)
quantize_act_kernel(const uint4 *__restrict__ x, int64_t M, int64_t K, uint2 *__restrict__ q,
                    float *__restrict__ s)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, sub = lane & 3;
    const int64_t G = K >> 7;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * Q1_ROWS;
    const int64_t g = static_cast<int64_t>(blockIdx.y) * Q1_GROUPS + warp;
    const int64_t K8 = K >> 3;   // 16-byte bf16 chunks per row (= 8-byte code chunks per row)
    if (g >= G)
        return;

    uint4 v[2][4];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int64_t m = m0 + 8 * b + r;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[b][j] = (m < M) ? __ldcs(x + m * K8 + g * 16 + 4 * j + sub) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const int64_t m = m0 + 8 * b + r;
        float f[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float t[8];
            unpack8(v[b][j], t);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                f[8 * j + e] = t[e];
        }
        uint32_t am2 = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            am2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(am2, v[b][j].x), v[b][j].y), v[b][j].z),
                                v[b][j].w);
        float amax = absmax_value(am2);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const GroupScale gs = group_scale(amax);
        uint32_t m2 = 0x7FFF7FFFu;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m2 = min_s16x2(min_s16x2(min_s16x2(min_s16x2(m2, v[b][j].x), v[b][j].y), v[b][j].z), v[b][j].w);
        uint32_t w[8];
        uint32_t redo = encode_words<8>(f, gs, has_neg_zero(m2), w);
        if (m < M) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                __stcs(q + m * K8 + g * 16 + 4 * j + sub, make_uint2(w[2 * j], w[2 * j + 1]));
            if (sub == 0)
                s[g * M + m] = gs.s;
            // rare: words that need the correctly rounded quotient
            while (redo != 0u) {
                const int k = __ffs(redo) - 1;
                redo &= redo - 1u;
                const int64_t e = m * K + g * 128 + (4 * (k >> 1) + sub) * 8 + 4 * (k & 1);
                const uint2 in = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(x) + e);
                *reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(q) + e) = encode4_exact(in, gs.s);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 128x1 groups along rows (tokens) of each column, written transposed.
// CTA tile: 128 rows x 64 columns of bf16 staged in shared memory (128 bytes
// per row).  Warp q takes rows 32q .. 32q+31; lane l takes the column pair
// 2l, 2l+1, reading one 4-byte word per row (a warp reads one contiguous
// 128-byte row per step: no bank conflicts).  The four row quarters combine
// their amax through shared memory; each column's 32 codes of a quarter
// (one 32-byte sector of an output row) then leave whole, two lanes per
// sector per store instruction.
// ---------------------------------------------------------------------------
constexpr int Q2_ROWS = 128;
constexpr int Q2_COLS = 64;
constexpr int Q2_THREADS = 128;

__global__ void __launch_bounds__(Q2_THREADS)
quantize_act_t_kernel(const uint4 *__restrict__ x, int64_t M, int64_t C, uint8_t *__restrict__ qt,
                      float *__restrict__ st)
{
    __shared__ uint4 tile[Q2_ROWS][Q2_COLS / 8];
    __shared__ float2 s_amax[4][Q2_COLS / 2];
    const int t = threadIdx.x, q = t >> 5, lane = t & 31;
    const int64_t m0 = static_cast<int64_t>(blockIdx.x) * Q2_ROWS;
    const int64_t c0 = static_cast<int64_t>(blockIdx.y) * Q2_COLS;
    const int64_t C8 = C >> 3;

    uint4 v[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const int idx = p * Q2_THREADS + t;
        v[p] = __ldcs(x + (m0 + (idx >> 3)) * C8 + (c0 >> 3) + (idx & 7));
    }
#pragma unroll
    for (int p = 0; p < 8; ++p) {
        const int idx = p * Q2_THREADS + t;
        tile[idx >> 3][idx & 7] = v[p];
    }
    __syncthreads();

    float f0[32], f1[32];
    // per-half running maxima and minima: low halves column 0, high halves column 1
    uint32_t am2 = 0u, m2 = 0x7FFF7FFFu;   // (m2: a -0 among this thread's values)
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t w = reinterpret_cast<const uint32_t *>(&tile[32 * q + i][0])[lane];
        f0[i] = bf16_lo(w);
        f1[i] = bf16_hi(w);
        am2 = absmax_bf16x2(am2, w);
        m2 = min_s16x2(m2, w);
    }
    am2 &= 0x7FFF7FFFu;
    float a0 = bf16_lo(am2), a1 = bf16_hi(am2);
    s_amax[q][lane] = make_float2(a0, a1);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 o = s_amax[k][lane];
        a0 = fmaxf(a0, o.x);
        a1 = fmaxf(a1, o.y);
    }
    const GroupScale g0 = group_scale(a0), g1 = group_scale(a1);
    uint32_t w0[8], w1[8];
    uint32_t redo = encode_words<8>(f0, g0, (m2 & 0xFFFFu) == 0x8000u, w0) |
                    (encode_words<8>(f1, g1, (m2 >> 16) == 0x8000u, w1) << 8);
    const int64_t col = c0 + 2 * lane;
    if (q == 0)
        *reinterpret_cast<float2 *>(st + (m0 >> 7) * C + col) = make_float2(g0.s, g1.s);
    // rare: words that need the correctly rounded quotient (inputs re-read
    // from the shared-memory tile: 4 rows of this thread's column), patched in
    // the registers before anything is stored
    while (redo != 0u) {
        const int b = __ffs(redo) - 1;
        redo &= redo - 1u;
        const int hi = b >> 3, k = b & 7;
        float v4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t wv = reinterpret_cast<const uint32_t *>(&tile[32 * q + 4 * k + e][0])[lane];
            v4[e] = hi ? bf16_hi(wv) : bf16_lo(wv);
        }
        const uint32_t fixed = encode4_exact(v4[0], v4[1], v4[2], v4[3], hi ? g1.s : g0.s);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w0[i] = (!hi && k == i) ? fixed : w0[i];
            w1[i] = (hi && k == i) ? fixed : w1[i];
        }
    }
    // Each column's 32 codes of this row quarter form one 32-byte sector.  Lane
    // pairs (2i, 2i+1) exchange halves so that every store instruction writes
    // whole sectors: the even lane writes bytes 0-15 and the odd lane bytes
    // 16-31 of the same column (a sector written in two halves by two
    // instructions costs DRAM bandwidth).  The even lane holds columns
    // c, c+1 and the odd lane c+2, c+3 (c = c0 + 4i).
    const bool odd = lane & 1;
    uint32_t x0[4], x1[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        x0[k] = __shfl_xor_sync(0xffffffffu, odd ? w0[k] : w0[4 + k], 1);
        x1[k] = __shfl_xor_sync(0xffffffffu, odd ? w1[k] : w1[4 + k], 1);
    }
    const int64_t cp = c0 + 2 * (lane & ~1);          // the pair's first column
    uint8_t *base = qt + m0 + 32 * q + (odd ? 16 : 0);
    // column cp (the even lane's first): even its own bytes 0-15, odd the received 16-31
    __stcs(reinterpret_cast<uint4 *>(base + cp * M),
           odd ? make_uint4(x0[0], x0[1], x0[2], x0[3]) : make_uint4(w0[0], w0[1], w0[2], w0[3]));
    // column cp + 2 (the odd lane's first)
    __stcs(reinterpret_cast<uint4 *>(base + (cp + 2) * M),
           odd ? make_uint4(w0[4], w0[5], w0[6], w0[7]) : make_uint4(x0[0], x0[1], x0[2], x0[3]));
    // columns cp + 1 and cp + 3 (the lanes' second columns)
    __stcs(reinterpret_cast<uint4 *>(base + (cp + 1) * M),
           odd ? make_uint4(x1[0], x1[1], x1[2], x1[3]) : make_uint4(w1[0], w1[1], w1[2], w1[3]));
    __stcs(reinterpret_cast<uint4 *>(base + (cp + 3) * M),
           odd ? make_uint4(w1[4], w1[5], w1[6], w1[7]) : make_uint4(x1[0], x1[1], x1[2], x1[3]));
}

// ---------------------------------------------------------------------------
// 128x128 weight blocks of one or several weight tensors (a group: every
// master weight of a step in one launch).  The tensors' blocks are numbered
// one after the other, each tensor's in row-major order.  Persistent CTAs (two
// per SM) walk them, block b, b + gridDim.x, ...; each block arrives by two
// bulk tensor copies (TMA, 128-byte swizzle, as in the dual quantiser) into
// one of two shared-memory stages, so the next block is in flight while this
// one is encoded.  Per block (8 warps):
//   read:      warp w takes rows 16w .. 16w+15, eight rows per step, four
//              lanes per row holding 32 values each (16-byte chunks sub,
//              sub+4, sub+8, sub+12), kept in registers as bf16 words;
//   amax:      lane maxima, warp shuffles, one value per warp in shared
//              memory, one barrier -- after which the stage is free and the
//              block two ahead is requested into it;
//   encode:    the codes of the lane's 32 values with the block's scale,
//              written to q (32 contiguous bytes per row quarter) and to a
//              shared code tile;
//   transpose: after a barrier, each lane reads four code columns of 16 rows
//              from the tile and writes them, transposed by byte permutes,
//              as 16-byte runs of qt's rows; the two lanes of a pair take
//              adjacent 16-row ranges, so each store instruction writes whole
//              32-byte sectors.
// The next block's first barrier orders this block's tile reads before the
// next block's tile writes.
// ---------------------------------------------------------------------------
constexpr int QW_THREADS = 256;
constexpr int QW_STAGES = 2;
constexpr int QW_CODE_PITCH = 160;           // bytes per code-tile row: row-pass writes in two wavefronts
constexpr int QW_GROUP_MAX = 8;              // weight tensors per launch (JETFP8_WEIGHT_GROUP_MAX)

struct WeightSmem {
    uint8_t tile[QW_STAGES][2][128][128];    // per stage: two 64-column halves, 128-byte swizzle
    uint8_t codes[128][QW_CODE_PITCH];
    uint64_t full[QW_STAGES];
    float red[QW_THREADS / 32];
};
constexpr uint32_t QW_SMEM_BYTES = sizeof(WeightSmem) + 1024;   // + alignment slack

__device__ __forceinline__ const uint8_t *weight_chunk(const WeightSmem &sm, int stage, int r, int c)
{
    return &sm.tile[stage][c >> 3][r][((c & 7) ^ (r & 7)) << 4];
}

// The tensors of one launch: tensor t's blocks are first_block[t] ..
// first_block[t + 1] - 1 of the launch's numbering.
struct WeightGroup {
    CUtensorMap map[QW_GROUP_MAX];           // W_t [N_t][K_t] bf16 as 128-row x 64-column boxes, 128-byte swizzle
    int64_t N[QW_GROUP_MAX], K[QW_GROUP_MAX];
    uint8_t *q[QW_GROUP_MAX];
    float *s[QW_GROUP_MAX];
    uint8_t *qt[QW_GROUP_MAX];               // may be null per tensor
    int64_t first_block[QW_GROUP_MAX + 1];
    int count;
};

// Block blk of the launch: its tensor, and its block row and column there.
struct WeightBlock {
    int t;
    int64_t bn, bk;
};

__device__ __forceinline__ WeightBlock locate_block(const WeightGroup &grp, int64_t blk)
{
    int t = 0;
    while (t + 1 < grp.count && blk >= grp.first_block[t + 1])
        ++t;
    const int64_t local = blk - grp.first_block[t], bk_count = grp.K[t] >> 7;
    return WeightBlock{t, local / bk_count, local % bk_count};
}

__global__ void __launch_bounds__(QW_THREADS, 2)
quantize_weight_kernel(const __grid_constant__ WeightGroup grp, uint32_t *__restrict__ err)
{
    extern __shared__ uint8_t weight_smem_raw[];
    WeightSmem &sm = *reinterpret_cast<WeightSmem *>((reinterpret_cast<uintptr_t>(weight_smem_raw) + 1023) &
                                                     ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t blocks = grp.first_block[grp.count];
    const int64_t first = blockIdx.x, stride = gridDim.x;
    constexpr uint32_t TILE_BYTES = 128 * 128 * 2;

    auto request = [&](int64_t blk, int stage) {   // one thread: bring block blk into stage
        const WeightBlock b = locate_block(grp, blk);
        const int32_t n0 = static_cast<int32_t>(b.bn << 7), k0 = static_cast<int32_t>(b.bk << 7);
        ptx::mbar_arrive_expect_tx(&sm.full[stage], TILE_BYTES);
        ptx::tma_load_2d(&sm.tile[stage][0][0][0], &grp.map[b.t], &sm.full[stage], k0, n0);
        ptx::tma_load_2d(&sm.tile[stage][1][0][0], &grp.map[b.t], &sm.full[stage], k0 + 64, n0);
    };
    if (threadIdx.x == 0) {
        for (int st = 0; st < QW_STAGES; ++st)
            ptx::mbar_init(&sm.full[st], 1);
        ptx::fence_mbar_init();
        for (int t = 0; t < grp.count; ++t)
            ptx::tma_prefetch_desc(&grp.map[t]);
        for (int st = 0; st < QW_STAGES; ++st)
            if (first + st * stride < blocks)
                request(first + st * stride, st);
    }
    __syncthreads();

    const int rr = lane >> 2, sub = lane & 3;
    int it = 0;
    for (int64_t blk = first; blk < blocks; blk += stride, ++it) {
        const int stage = it % QW_STAGES;
        const uint32_t phase = static_cast<uint32_t>(it / QW_STAGES) & 1u;
        const bool landed = ptx::mbar_wait(&sm.full[stage], phase, nullptr, err, ERRBIT_QUANT, 2000000000ull);
        if (__syncthreads_or(!landed)) {
            // give up together; the copies still requested must land before exit
            if (threadIdx.x == 0)
                for (int k = 0; k < QW_STAGES; ++k) {
                    const int64_t b2 = blk + k * stride;
                    if (b2 < blocks)
                        ptx::mbar_wait(&sm.full[(it + k) % QW_STAGES], static_cast<uint32_t>((it + k) / QW_STAGES) & 1u,
                                       nullptr, err, ERRBIT_DRAIN, 2000000000ull);
                }
            return;
        }
        const WeightBlock wb = locate_block(grp, blk);
        const int64_t N = grp.N[wb.t], K = grp.K[wb.t], bk_count = K >> 7;
        uint8_t *__restrict__ q = grp.q[wb.t];
        uint8_t *__restrict__ qt = grp.qt[wb.t];
        const int64_t n_base = wb.bn << 7, k_base = wb.bk << 7;

        // ---- read this lane's 64 values and their amax
        uint4 v[2][4];
        uint32_t am2 = 0u;
#pragma unroll
        for (int step = 0; step < 2; ++step) {
            const int r = 16 * warp + 8 * step + rr;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[step][j] = *reinterpret_cast<const uint4 *>(weight_chunk(sm, stage, r, sub + 4 * j));
                am2 = absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(am2, v[step][j].x), v[step][j].y),
                                                  v[step][j].z),
                                    v[step][j].w);
            }
        }
        float amax = absmax_value(am2);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0)
            sm.red[warp] = amax;
        __syncthreads();   // every read of this stage is done; the block's warp maxima are visible
        if (threadIdx.x == 0 && blk + QW_STAGES * stride < blocks)
            request(blk + QW_STAGES * stride, stage);
        amax = sm.red[0];
#pragma unroll
        for (int i = 1; i < QW_THREADS / 32; ++i)
            amax = fmaxf(amax, sm.red[i]);
        const GroupScale gs = group_scale(amax);
        if (threadIdx.x == 0)
            grp.s[wb.t][wb.bn * bk_count + wb.bk] = gs.s;

        // ---- encode: codes to q and to the shared code tile
#pragma unroll
        for (int step = 0; step < 2; ++step) {
            const int r = 16 * warp + 8 * step + rr;
            float f[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float u[8];
                unpack8(v[step][j], u);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    f[8 * j + e] = u[e];
            }
            uint32_t m2 = 0x7FFF7FFFu;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                m2 = min_s16x2(min_s16x2(min_s16x2(min_s16x2(m2, v[step][j].x), v[step][j].y), v[step][j].z),
                               v[step][j].w);
            uint32_t wd[8];
            uint32_t redo = encode_words<8>(f, gs, has_neg_zero(m2), wd);
            uint8_t *row_q = q + (n_base + r) * K + k_base;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint2 c = make_uint2(wd[2 * j], wd[2 * j + 1]);
                __stcs(reinterpret_cast<uint2 *>(row_q + 8 * (sub + 4 * j)), c);
                if (qt != nullptr)
                    *reinterpret_cast<uint2 *>(&sm.codes[r][8 * (sub + 4 * j)]) = c;
            }
            // rare: a word that needs the correctly rounded quotient gets it, its
            // four inputs taken from the lane's registers (word k: chunk
            // sub + 4(k/2), half k%2)
            while (redo != 0u) {
                const int k = __ffs(redo) - 1;
                redo &= redo - 1u;
                const int col = 8 * (sub + 4 * (k >> 1)) + 4 * (k & 1);
                const uint32_t code = encode4_exact(pick_word(v[step], k), gs.s);
                *reinterpret_cast<uint32_t *>(row_q + col) = code;
                if (qt != nullptr)
                    *reinterpret_cast<uint32_t *>(&sm.codes[r][col]) = code;
            }
        }
        if (qt == nullptr)
            continue;
        __syncthreads();   // the code tile is complete

        // ---- transposed write: lane l of warp w takes output rows kq .. kq+3
        // (columns of the block, kq = 64 (w / 4) + 4 (l / 2)) and their codes
        // for block rows n0 .. n0+15 (n0 = 32 (w % 4) + 16 (l % 2)): sixteen
        // 4-byte reads (one block row each), a 4 x 4 byte transpose per four
        // rows, one 16-byte store per output row, lanes 2i and 2i+1 filling
        // the two halves of one 32-byte sector
        const int kq = 64 * (warp >> 2) + 4 * (lane >> 1), n0 = 32 * (warp & 3) + 16 * (lane & 1);
        uint32_t rw[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            rw[i] = *reinterpret_cast<const uint32_t *>(&sm.codes[n0 + i][kq]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t o[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                // byte j of block rows 4b .. 4b+3: the codes of column kq + j
                const uint32_t lo = __byte_perm(rw[4 * b], rw[4 * b + 1], j | ((4 + j) << 4));
                const uint32_t hi = __byte_perm(rw[4 * b + 2], rw[4 * b + 3], j | ((4 + j) << 4));
                o[b] = __byte_perm(lo, hi, 0x5410);
            }
            __stcs(reinterpret_cast<uint4 *>(qt + (k_base + kq + j) * N + n_base + n0),
                   make_uint4(o[0], o[1], o[2], o[3]));
        }
    }
}

// ---------------------------------------------------------------------------
// Dual output: one read of X [M][K] yields both the 1x128 row-group codes and
// scales (as quantize_act_kernel) and the 128x1 column-group codes and scales
// written transposed (as quantize_act_t_kernel).  One CTA (8 warps) per 128 x
// 128 tile:
//   load:    two bulk tensor copies (tensor memory accelerator) bring the tile
//            into shared memory as two 64-column halves with the 128-byte
//            swizzle (16-byte chunk c of row r at position c ^ (r & 7)); every
//            thread waits on one mbarrier, bounded, and the block gives up
//            together if the copies never land.
//   rows:    warp w takes rows 16w .. 16w+15, eight rows per step, four lanes
//            per row holding 32 values each (16-byte chunks sub, sub + 4,
//            sub + 8, sub + 12), and encodes them: one scale per 32 values per
//            lane, amax in two shuffles, codes in 32-byte runs.
//   columns: warp w then takes 8-column chunk w (then w + 8) and reads it with
//            four transposing matrix loads (ldmatrix .trans, 32 rows each,
//            conflict-free thanks to the swizzle): lane 4c + q then holds
//            column c, rows 8j + 2q and 8j + 2q + 1 for j = 0..15, so a 128x1
//            group is four lanes of one warp (amax: two shuffles).  The tile is
//            read-only once it has landed, so no barrier separates the passes.
//            The interleaved codes are put back in row order through a small
//            per-warp staging buffer and leave as two 16-byte stores per lane,
//            arranged so that each store instruction writes whole 32-byte
//            sectors.
// ---------------------------------------------------------------------------
constexpr int QD_TILE = 128;
constexpr int QD_THREADS = 256;
constexpr int QD_STAGE_PITCH = 140;          // bytes per staged column (35 words: writes and reads bank-conflict free)

struct DualSmem {
    // the 128 x 128 bf16 tile as two 64-column halves written by the tensor
    // memory accelerator with its 128-byte swizzle: 16-byte chunk c of row r
    // of a half sits at position c ^ (r & 7) of the row (1024-byte aligned)
    uint8_t tile[2][QD_TILE][128];                             // 32 KB
    uint8_t stage[QD_THREADS / 32][8][QD_STAGE_PITCH];        // codes of 8 columns per warp
    uint64_t bar;
};
constexpr uint32_t QD_SMEM_BYTES = sizeof(DualSmem) + 1024;    // + alignment slack

// Address of 16-byte chunk c (0..15) of tile row r.
__device__ __forceinline__ const uint8_t *dual_chunk(const DualSmem &sm, int r, int c)
{
    return &sm.tile[c >> 3][r][((c & 7) ^ (r & 7)) << 4];
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], const void *row_addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(ptx::smem_u32(row_addr))
                 : "memory");
}

// (five blocks per SM: 48 registers, which the packed bf16 amax makes room
// for without spills; +2 % against four on the 8B-class gradient shapes)
__global__ void __launch_bounds__(QD_THREADS, 5)
quantize_act_dual_kernel(const __grid_constant__ CUtensorMap tmap_x, int64_t M, int64_t K, uint8_t *__restrict__ q,
                         float *__restrict__ s, uint8_t *__restrict__ qt, float *__restrict__ st,
                         uint32_t *__restrict__ err)
{
    extern __shared__ uint8_t dual_smem_raw[];
    DualSmem &sm = *reinterpret_cast<DualSmem *>((reinterpret_cast<uintptr_t>(dual_smem_raw) + 1023) &
                                                 ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles_k = K / QD_TILE;
    const int64_t m0 = (static_cast<int64_t>(blockIdx.x) / tiles_k) * QD_TILE;
    const int64_t k0 = (static_cast<int64_t>(blockIdx.x) % tiles_k) * QD_TILE;

    // the whole tile arrives by two bulk tensor copies; every thread waits
    // (bounded) for them, and the block gives up together if they never land
    if (threadIdx.x == 0) {
        ptx::mbar_init(&sm.bar, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ptx::mbar_arrive_expect_tx(&sm.bar, 2 * QD_TILE * 128);
        ptx::tma_load_2d(&sm.tile[0][0][0], &tmap_x, &sm.bar, static_cast<int32_t>(k0), static_cast<int32_t>(m0));
        ptx::tma_load_2d(&sm.tile[1][0][0], &tmap_x, &sm.bar, static_cast<int32_t>(k0 + 64),
                         static_cast<int32_t>(m0));
    }
    const bool landed = ptx::mbar_wait(&sm.bar, 0, nullptr, err, ERRBIT_QUANT, 2000000000ull);
    if (__syncthreads_or(!landed)) {
        // the block gives up, but the copies it started must not land in
        // shared memory after it has gone: one more bounded wait for them
        if (threadIdx.x == 0)
            ptx::mbar_wait(&sm.bar, 0, nullptr, err, ERRBIT_DRAIN, 2000000000ull);
        return;
    }

    // ---- rows: 16 per warp, 8 per step; four lanes per row, 32 values each
    //      (16-byte chunks sub, sub+4, sub+8, sub+12 of the row's 256 bytes)
    {
        const int rr = lane >> 2, sub = lane & 3;
#pragma unroll
        for (int step = 0; step < 2; ++step) {
            const int r = 16 * warp + 8 * step + rr;
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                v[j] = *reinterpret_cast<const uint4 *>(dual_chunk(sm, r, sub + 4 * j));
            float f[32];
            uint32_t am2 = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float u[8];
                unpack8(v[j], u);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    f[8 * j + e] = u[e];
                am2 = absmax_bf16x2(absmax_bf16x2(am2, v[j].x), v[j].y);
                am2 = absmax_bf16x2(absmax_bf16x2(am2, v[j].z), v[j].w);
            }
            float amax = absmax_value(am2);
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const GroupScale gs = group_scale(amax);
            uint32_t m2 = 0x7FFF7FFFu;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                m2 = min_s16x2(min_s16x2(min_s16x2(min_s16x2(m2, v[j].x), v[j].y), v[j].z), v[j].w);
            uint32_t w[8];
            uint32_t redo = encode_words<8>(f, gs, has_neg_zero(m2), w);
            uint8_t *row_q = q + (m0 + r) * K + k0;
#pragma unroll
            for (int j = 0; j < 4; ++j)      // the row's four lanes write 32 contiguous bytes per j
                *reinterpret_cast<uint2 *>(row_q + 8 * (sub + 4 * j)) = make_uint2(w[2 * j], w[2 * j + 1]);
            if (sub == 0)
                s[(k0 >> 7) * M + m0 + r] = gs.s;
            // rare: a word that needs the correctly rounded quotient gets it, its
            // four inputs re-read from the shared tile (word k: chunk sub + 4(k/2),
            // half k%2)
            while (redo != 0u) {
                const int k = __ffs(redo) - 1;
                redo &= redo - 1u;
                const int c = sub + 4 * (k >> 1);
                const uint2 in = reinterpret_cast<const uint2 *>(dual_chunk(sm, r, c))[k & 1];
                *reinterpret_cast<uint32_t *>(row_q + 8 * c + 4 * (k & 1)) = encode4_exact(in, gs.s);
            }
        }
    }
    // ---- columns: chunk w, then w + 8 (the tile is read-only from here on:
    //      no barrier between the passes) -----------------------------------
    const int cq = lane & 3;                         // q: which row pairs of each 8-row block
    const int cc = lane >> 2;                        // column within the 8-column chunk
    uint8_t *stg = &sm.stage[warp][0][0];
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const int chunk = warp + 8 * pass;
        uint32_t wv[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int r = 32 * j + lane;              // this lane's row address for the x4 load
            uint32_t t4[4];
            ldmatrix_x4_trans(t4, dual_chunk(sm, r, chunk));
#pragma unroll
            for (int m = 0; m < 4; ++m)
                wv[4 * j + m] = t4[m];               // rows 8(4j+m) + 2cq, +1 of column cc
        }
        float f[32];
        uint32_t am2 = 0u;
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            f[2 * b] = bf16_lo(wv[b]);
            f[2 * b + 1] = bf16_hi(wv[b]);
            am2 = absmax_bf16x2(am2, wv[b]);
        }
        float amax = absmax_value(am2);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const GroupScale gs = group_scale(amax);
        uint32_t m2 = 0x7FFF7FFFu;
#pragma unroll
        for (int b = 0; b < 16; ++b)
            m2 = min_s16x2(m2, wv[b]);
        uint32_t w[8];
        uint32_t redo = encode_words<8>(f, gs, has_neg_zero(m2), w);
        // word k holds rows 8(2k) + 2cq, +1 (low half) and 8(2k+1) + 2cq, +1 (high
        // half): put each 2-byte unit at its row in the staged column
        uint8_t *col = stg + cc * QD_STAGE_PITCH;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            *reinterpret_cast<uint16_t *>(col + 8 * (2 * k) + 2 * cq) = static_cast<uint16_t>(w[k]);
            *reinterpret_cast<uint16_t *>(col + 8 * (2 * k + 1) + 2 * cq) = static_cast<uint16_t>(w[k] >> 16);
        }
        // rare: a word that needs the correctly rounded quotient gets it, its four
        // inputs (rows 16k + 2cq, +1, 16k + 8 + 2cq, +1 of the column) re-read
        // from the shared tile; the fixed units overwrite the staged ones
        {
            const int colw = 8 * chunk + cc;          // column within the tile
            while (redo != 0u) {
                const int k = __ffs(redo) - 1;
                redo &= redo - 1u;
                float v4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int rr = 16 * k + 8 * (e >> 1) + 2 * cq + (e & 1);
                    const uint16_t h =
                        reinterpret_cast<const uint16_t *>(dual_chunk(sm, rr, chunk))[colw & 7];
                    v4[e] = __uint_as_float(static_cast<uint32_t>(h) << 16);
                }
                const uint32_t fixed = encode4_exact(v4[0], v4[1], v4[2], v4[3], gs.s);
                *reinterpret_cast<uint16_t *>(col + 16 * k + 2 * cq) = static_cast<uint16_t>(fixed);
                *reinterpret_cast<uint16_t *>(col + 16 * k + 8 + 2 * cq) = static_cast<uint16_t>(fixed >> 16);
            }
        }
        __syncwarp();
        // Column c's 128 codes leave as four 32-byte sectors (rows 32t .. 32t+31,
        // t = 0..3), each written whole by one store instruction: lanes 4c + q
        // with q = 2p and 2p+1 write the two 16-byte halves of sector 2p, then of
        // sector 2p+1 (a sector written in two halves by two instructions costs
        // DRAM bandwidth)
        const int64_t colg = k0 + 8 * chunk + cc;
        const int pair = cq >> 1, half = cq & 1;
#pragma unroll
        for (int t2 = 0; t2 < 2; ++t2) {
            const int sector = 2 * pair + t2;
            const uint32_t *s32 = reinterpret_cast<const uint32_t *>(stg + cc * QD_STAGE_PITCH + 32 * sector + 16 * half);
            __stcs(reinterpret_cast<uint4 *>(qt + colg * M + m0 + 32 * sector + 16 * half),
                   make_uint4(s32[0], s32[1], s32[2], s32[3]));
        }
        if (cq == 0)
            st[(m0 >> 7) * K + colg] = gs.s;
        __syncwarp();                                 // the staging buffer is reused next pass
    }
}

}  // namespace

cudaError_t launch_quantize_act(const void *x, int64_t M, int64_t K, uint8_t *q, float *s, cudaStream_t stream)
{
    const int64_t G = K / 128;
    dim3 grid(static_cast<unsigned>((M + Q1_ROWS - 1) / Q1_ROWS),
              static_cast<unsigned>((G + Q1_GROUPS - 1) / Q1_GROUPS));
    quantize_act_kernel<<<grid, Q1_THREADS, 0, stream>>>(static_cast<const uint4 *>(x), M, K,
                                                         reinterpret_cast<uint2 *>(q), s);
    return cudaGetLastError();
}

cudaError_t launch_quantize_act_transposed(const void *x, int64_t M, int64_t C, uint8_t *qt, float *st,
                                           cudaStream_t stream)
{
    dim3 grid(static_cast<unsigned>(M / Q2_ROWS), static_cast<unsigned>(C / Q2_COLS));
    quantize_act_t_kernel<<<grid, Q2_THREADS, 0, stream>>>(static_cast<const uint4 *>(x), M, C, qt, st);
    return cudaGetLastError();
}


namespace {
// codes[i] = E4M3 code of the fp32 pattern first + i, through the same
// conversion instruction the quantisers use; eight patterns per thread.
__global__ void __launch_bounds__(256) e4m3_encode_range_kernel(uint32_t first, int64_t count,
                                                                 uint8_t *__restrict__ codes)
{
    const int64_t words = (count + 7) >> 3;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < words;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t base = 8 * i;
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)   // patterns past the end wrap around; they are not stored
                v[e] = __uint_as_float(first + static_cast<uint32_t>(base + 4 * h + e));
            w[h] = ptx::cvt_e4m3x2(v[0], v[1]) | (ptx::cvt_e4m3x2(v[2], v[3]) << 16);
        }
        if (base + 8 <= count) {
            *reinterpret_cast<uint2 *>(codes + base) = make_uint2(w[0], w[1]);
        } else {
            for (int e = 0; base + e < count; ++e)
                codes[base + e] = static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)));
        }
    }
}
}  // namespace

cudaError_t launch_e4m3_encode_range(uint32_t first, int64_t count, uint8_t *codes, int sm_count,
                                     cudaStream_t stream)
{
    const int64_t words = (count + 7) / 8;
    const int64_t want = (words + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    e4m3_encode_range_kernel<<<static_cast<unsigned>(want < cap ? want : cap), 256, 0, stream>>>(first, count,
                                                                                                 codes);
    return cudaGetLastError();
}

}  // namespace jetfp8

namespace jetfp8 {
cudaError_t launch_quantize_weight_group(int count, const void *const *w, const int64_t *N, const int64_t *K,
                                         uint8_t *const *q, float *const *s, uint8_t *const *qt,
                                         PFN_cuTensorMapEncodeTiled_v12000 encode, uint32_t *err, int sm_count,
                                         cudaStream_t stream)
{
    if (count < 1 || count > QW_GROUP_MAX)
        return cudaErrorInvalidValue;
    WeightGroup grp = {};
    grp.count = count;
    grp.first_block[0] = 0;
    for (int t = 0; t < count; ++t) {
        // W_t [N][K] bf16 seen as 128-row x 64-column boxes with the 128-byte swizzle
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K[t]), static_cast<cuuint64_t>(N[t])};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K[t]) * 2};
        cuuint32_t box[2] = {64, 128};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&grp.map[t], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w[t]), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        grp.N[t] = N[t];
        grp.K[t] = K[t];
        grp.q[t] = q[t];
        grp.s[t] = s[t];
        grp.qt[t] = qt[t];
        grp.first_block[t + 1] = grp.first_block[t] + (N[t] / 128) * (K[t] / 128);
    }
    cudaError_t e = cudaFuncSetAttribute(quantize_weight_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(QW_SMEM_BYTES));
    if (e != cudaSuccess)
        return e;
    const int64_t blocks = grp.first_block[count];
    const int64_t cap = static_cast<int64_t>(sm_count) * 2;   // two resident CTAs per SM
    const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
    quantize_weight_kernel<<<grid, QW_THREADS, QW_SMEM_BYTES, stream>>>(grp, err);
    return cudaGetLastError();
}

cudaError_t launch_quantize_weight(const void *w, int64_t N, int64_t K, uint8_t *q, float *s, uint8_t *qt,
                                   PFN_cuTensorMapEncodeTiled_v12000 encode, uint32_t *err, int sm_count,
                                   cudaStream_t stream)
{
    return launch_quantize_weight_group(1, &w, &N, &K, &q, &s, &qt, encode, err, sm_count, stream);
}

cudaError_t launch_quantize_act_dual(const void *x, int64_t M, int64_t K, uint8_t *q, float *s, uint8_t *qt,
                                     float *st, PFN_cuTensorMapEncodeTiled_v12000 encode, uint32_t *err,
                                     cudaStream_t stream)
{
    // X [M][K] bf16 seen as 128-row x 64-column boxes with the 128-byte swizzle
    CUtensorMap tmap;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(QD_TILE)};
    cuuint32_t estr[2] = {1, 1};
    if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(quantize_act_dual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(QD_SMEM_BYTES));
    if (e != cudaSuccess)
        return e;
    const int64_t tiles = (M / QD_TILE) * (K / QD_TILE);
    quantize_act_dual_kernel<<<static_cast<unsigned>(tiles), QD_THREADS, QD_SMEM_BYTES, stream>>>(tmap, M, K, q, s,
                                                                                                  qt, st, err);
    return cudaGetLastError();
}
}  // namespace jetfp8
