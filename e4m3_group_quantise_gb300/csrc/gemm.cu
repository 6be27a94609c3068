// Block-scaled FP8 (E4M3) GEMM on the 5th-generation tensor cores (sm_103a).
//
//   D[r][c] = bf16( sum_g  sa(g,r) * sb(g,c) * P_g[r][c] ),
//   P_g = A[:, 128g:128g+128] * B[:, 128g:128g+128]^T   (exact FP8 products,
//                                                         fp32 sums, tensor cores)
//
// One kernel serves the three products of a linear layer (Jet-RL, technical
// summaries on gist.science, "Schéma de Quantification": FP8 GEMMs for the
// forward pass and for DGrad / WGrad, 1x128 activation groups, 128x128
// weight blocks, 1x128 and 128x1 groups for WGrad):
//   Fprop  A = X codes [M][K],    sa = X's 1x128 scales,   B = W codes [N][K],
//          sb = one scale per 128x128 weight block;
//   Dgrad  A = dY codes [M][N],   sa = dY's 1x128 scales,  B = W^T codes [K][N],
//          sb = one scale per 128x128 weight block;
//   Wgrad  A = dY^T codes [N][M], sa = dY's 128x1 scales,  B = X^T codes [K][M],
//          sb = X's 128x1 scales (one per output column and token group).
// The scales are arbitrary fp32 values (amax / 448), not powers of two, so the
// tensor core's own block scaling cannot apply them: each 128-wide group is
// multiplied into a fresh TMEM partial and CUDA-core warps fold it into an
// fp32 register accumulator with the group's scales ("promotion").
//
// Structure: persistent, one CTA per SM, 384 threads (3 warpgroups).
//   warp 0, lane 0 : TMA producer   -- A and B tiles of one group per smem stage
//   warps 1 and 3,  : MMA issuers   -- even and odd groups: 4 x tcgen05.mma
//   lane 0                             (K = 32 each) per group into one of the
//                                      TMEM partial buffers
//   warp 2         : scale loader   -- cp.async of the group's row scales (128)
//                                      and block scales into a smem ring (with
//                                      per-column scales, both contiguous, the
//                                      TMA producer fetches them instead, two
//                                      bulk copies per group)
//   warps 4..11    : promotion      -- two warpgroups, each 128 rows x BN/2
//                                      columns (narrow tiles: the first alone);
//                                      tcgen05.ld the partial, free the buffer,
//                                      acc += partial * sa * sb (packed fp32x2
//                                      operations); bf16 epilogue: each warp
//                                      stages 32 rows x 16 columns in shared
//                                      memory and TMA-stores them (double-
//                                      buffered, asynchronous)
// Registers are rebalanced with setmaxnreg (RegSplit): with 128 x 256 tiles
// the control warpgroup drops to 40 per thread and the promotion warpgroups
// rise to 232 (128*40 + 256*232 = 64512 = 384 threads * 168, the launch
// allocation).  Tile BM = 128 rows x BN (256; 128, 64 or 32 for problems with
// few tiles) columns; one pipeline stage per 128-wide K group (the scale
// granularity).  Every wait is bounded: a wait that runs out sets the device
// error word, the CTA drains its copies and MMAs in flight, frees its tensor
// memory and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "internal.cuh"
#include "ptx.cuh"

namespace jetfp8 {
namespace {

constexpr int BM = 128;
constexpr int BK = 128;                  // one scale group
constexpr int NUM_THREADS = 384;
constexpr int PRODUCER_WARP = 0;
constexpr int MMA_WARP = 1;
constexpr int SCALE_WARP = 2;
constexpr int FIRST_PROMO_WARP = 4;
constexpr int SCALE_STAGES_ALL = 4;      // scale ring slots
constexpr int SCALE_RAW_AHEAD = 2;       // block scales: groups the loader stages ahead
constexpr int MAX_TBUF = 8;              // TMEM partial buffers at most (narrow tiles)
// setmaxnreg split per tile width: wide tiles keep 128 accumulator registers
// per promotion thread, 128-wide tiles 64 (which leaves the control warps room).
template <int BN> struct RegSplit;
template <> struct RegSplit<256> { static constexpr uint32_t CTRL = 40, PROMO = 232; };
template <> struct RegSplit<128> { static constexpr uint32_t CTRL = 88, PROMO = 200; };
template <> struct RegSplit<64> { static constexpr uint32_t CTRL = 88, PROMO = 200; };
template <> struct RegSplit<32> { static constexpr uint32_t CTRL = 88, PROMO = 200; };
static_assert(128 * RegSplit<256>::CTRL + 256 * RegSplit<256>::PROMO <= NUM_THREADS * 168, "register split");
static_assert(128 * RegSplit<128>::CTRL + 256 * RegSplit<128>::PROMO <= NUM_THREADS * 168, "register split");
// Tile rasterisation: the part of an operand that a band of tiles reuses
// across waves is kept to this many bytes.  Measured on GB300 (one launch per
// ncu capture): a 25 MB operand reused by every wave is read from DRAM once,
// a 59-67 MB one 10 to 30 times -- lines that every SM reads are held in both
// halves of the L2, so reuse across waves holds only for about a quarter of
// the L2's nominal size.
constexpr int64_t L2_BAND_BYTES = int64_t{30} << 20;
constexpr int BALANCED_BAND_M = 16;      // bands of 16 m-tiles when no operand slice can stay in L2
constexpr uint64_t WAIT_TIMEOUT_NS = 2000000000ull;   // 2 s

struct KernelArgs {
    const float *sa;
    const float *sb;
    int64_t sb_stride_g;
    int64_t sb_stride_c;
    __nv_bfloat16 *d;
    uint32_t *err;
    int32_t rows, cols, groups;
    int32_t tiles_m, tiles_n;
    int32_t band;         // tile rasterisation: tiles per band along the banded axis (see launch_gemm)
    int32_t band_n;       // 0: bands of m-tiles, 1: bands of n-tiles
    int32_t stream_a;     // 1: A's tiles are read once, load them with the evict-first L2 priority
    int32_t stream_b;     // 1: the same for B
    int32_t stream_d;     // 1: the output is larger than L2 can keep: store it with evict-first
    uint32_t stage_bytes; // bytes one pipeline stage's two copies bring (A's box may be short)
};

// HALF_A (problems of at most 64 rows, i.e. decode): A arrives as a 64-row box
// (no out-of-bounds fill for the missing rows) and consecutive stages' A
// tiles are packed 64 rows (8 KB) apart.  The MMA still reads a 128-row
// window: its rows 64..127 are the next stage's rows 0..63 (or the padding
// after the last stage), which only feed output rows 64..127 -- rows past the
// problem, never stored.  Halving A's footprint buys more stages, i.e. more of
// W in flight, which is what bounds decode.
template <int BN, int STAGES, bool HALF_A = false, bool SB_PER_COLUMN = false>
struct Smem {
    static constexpr uint32_t A_BYTES = HALF_A ? (BM / 2) * BK : BM * BK;   // A stride between stages
    static constexpr uint32_t A_LOAD_BYTES = A_BYTES;                       // bytes one stage's A copy brings
    static constexpr uint32_t A_PAD = HALF_A ? (BM / 2) * BK : 0;          // the last stage's window tail
    static constexpr uint32_t B_BYTES = BN * BK;
    static constexpr uint32_t STAGE_BYTES = A_LOAD_BYTES + B_BYTES;
    static constexpr uint32_t B_OFF = STAGES * A_BYTES + A_PAD;
    static constexpr uint32_t TILES = B_OFF + STAGES * B_BYTES;
    // scale ring.  Per slot 128 row scales, then BN column scales (per-column
    // scales) or the tile's block scale (narrow tiles, padded to 16 bytes).
    // 256-wide block-scale tiles (READY): per slot the ready products sa * sb
    // of the tile's 128 rows, one row of 128 per 128-column block.
    static constexpr bool READY = !SB_PER_COLUMN && BN >= 256;
    static constexpr int NBLK = BN >= 256 ? 2 : 1;
    static constexpr uint32_t SCALE_FLOATS = SB_PER_COLUMN ? BM + BN : (READY ? NBLK * BM : BM + 4);
    static constexpr uint32_t SCALE_OFF = TILES;
    // TMEM partial buffers: two 256-wide ones; four 128-wide ones; eight for
    // narrower (decode) tiles.  Block scales have one slot per buffer (the
    // TMEM-full barrier also covers the slot); per-column scales their own ring.
    static constexpr uint32_t NBUF = BN >= 256 ? 2 : (BN == 128 ? 4 : MAX_TBUF);
    static constexpr int SCALE_STAGES = SB_PER_COLUMN ? SCALE_STAGES_ALL : static_cast<int>(NBUF);
    static constexpr uint32_t SCALE_BYTES = SCALE_STAGES * SCALE_FLOATS * 4;
    // block scales: the loader's staging ring of raw scales (128 row scales,
    // then the tile's block scales, padded to 16 bytes)
    static constexpr int RAW_SLOTS = READY ? SCALE_RAW_AHEAD + 1 : 0;
    static constexpr uint32_t RAW_FLOATS = BM + 4;
    static constexpr uint32_t RAW_OFF = SCALE_OFF + SCALE_BYTES;
    static constexpr uint32_t RAW_BYTES = (RAW_SLOTS * RAW_FLOATS * 4 + 127) / 128 * 128;
    // epilogue staging: per promotion warp two 32-row x 16-column bf16 chunks,
    // the sources of TMA stores (which need an aligned shared-memory address)
    static constexpr uint32_t OUT_OFF = (RAW_OFF + RAW_BYTES + 1023) / 1024 * 1024;
    static constexpr uint32_t OUT_CHUNK_BYTES = 32 * 16 * 2;
    static constexpr uint32_t OUT_BYTES = 8 * 2 * OUT_CHUNK_BYTES;
    static constexpr uint32_t BAR_OFF = OUT_OFF + OUT_BYTES;
    // full[S], empty[S], sfull[SS], sempty[SS], tfull[MAX_TBUF], tempty[MAX_TBUF], mma_done,
    // tmem holder, abort flag
    static constexpr uint32_t CTRL_BYTES = (2 * STAGES + 2 * SCALE_STAGES + 2 * MAX_TBUF + 1) * 8 + 16;
    static constexpr uint32_t TOTAL = 1024 /* alignment slack */ + BAR_OFF + CTRL_BYTES;
    static_assert(B_OFF % 1024 == 0 && TILES % 1024 == 0, "operand tiles on 1024-byte boundaries (128-byte swizzle)");
    static_assert(SCALE_OFF % 16 == 0 && RAW_OFF % 16 == 0 && (SCALE_FLOATS * 4) % 16 == 0 &&
                      (RAW_FLOATS * 4) % 16 == 0,
                  "16-byte copies into the scale slots");
    static_assert(OUT_OFF % 1024 == 0 && OUT_CHUNK_BYTES % 128 == 0, "TMA store sources aligned");
    static_assert(BAR_OFF % 8 == 0, "barriers 8-byte aligned");
};

// Tile order: bands of `band` tiles along one axis, the banded axis varying
// fastest inside a band, which then sweeps the whole other axis.  The
// band's slice of its operand (band x 128 rows of A, or band x BN rows of B,
// each over the whole contraction) is what consecutive waves reuse; the
// other operand is read once per band.
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int band, int band_n, int &tm,
                                            int &tn)
{
    const int banded = band_n ? tiles_n : tiles_m;
    const int other = band_n ? tiles_m : tiles_n;
    const int per_band = band * other;
    const int b = tile / per_band;
    const int first = b * band;
    const int width = min(banded - first, band);
    const int in_band = tile - b * per_band;
    const int u = first + in_band % width, v = in_band / width;
    tm = band_n ? v : u;
    tn = band_n ? u : v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// 16x256b TMEM loads of 64 or 32 columns, chosen by the register array

template <int BN, int STAGES, bool SB_PER_COLUMN, bool HALF_A>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
            const __grid_constant__ CUtensorMap tmap_d, const KernelArgs args)
{
    using L = Smem<BN, STAGES, HALF_A, SB_PER_COLUMN>;
    constexpr int SCALE_STAGES = L::SCALE_STAGES;
    // Tiles 128 or 256 wide: two promotion warpgroups, one per column half.
    // Narrow tiles (decode-sized problems): the first warpgroup alone.
    constexpr int NWG = BN >= 128 ? 2 : 1;
    constexpr int COLS_PER_WG = BN / NWG;        // columns per promotion warpgroup
    constexpr int CHUNKS = COLS_PER_WG / 32;     // tcgen05.ld x32 per group
    constexpr int LPW = CHUNKS >= 2 ? 2 : 1;     // 32-column chunks per load and wait
    static_assert(CHUNKS % LPW == 0, "loads are issued in pairs");
    // Per-column scales (Wgrad) read the partial as 16x256b quads instead:
    // a thread then holds four rows x a quarter of the columns, so each
    // column-scale pair it fetches from shared memory serves four rows.
    // The range is read in slabs of 32 columns (4 blocks of 8), both 16-lane
    // halves of the warp's quarter per slab, the next slab's load in flight
    // while this one is scaled (Wgrad +3 % against two unpipelined 64-column
    // slabs; the same pipelining of the 32x32b loads measured 19 % slower for
    // Fprop, whose arithmetic per slab is too short to hide a load).
    constexpr int CB = COLS_PER_WG / 8;          // 8-column blocks per warpgroup
    constexpr int PS = 4;                        // blocks per slab
    constexpr int NPS = CB / PS;                 // slabs per group
    static_assert(CB % PS == 0, "32-column slabs");
    // TMEM partial buffers (two 256-wide ones; four 128-wide ones; eight for
    // narrower, decode, tiles), so that the MMAs can run several groups ahead
    // of the read-back instead of waiting on every hand-off.
    constexpr uint32_t NBUF = L::NBUF;
    // The MMA issuers commit only the TMEM-full barrier: its completion also
    // means the group's MMAs have read their shared-memory stage, and the
    // first promotion warp, seeing it, releases the stage to the producer.
    // One commit per group shortens the issue loop, which sits in the chain
    // of hand-offs (measured: decode tiles 5-9 % faster, 256-wide tiles about
    // even).
    // A second MMA issuer (the otherwise idle fourth control warp): even
    // groups from the MMA warp, odd groups from warp 3, into different TMEM
    // buffers, so one group's MMAs are issued as soon as its buffer is free
    // rather than after the previous group's issue loop (the issue of a
    // group's four MMAs and commits takes a few hundred cycles).
    constexpr int SECOND_MMA_WARP = 3;
    constexpr uint32_t TMEM_COLS = NBUF * BN;
    static_assert(TMEM_COLS <= 512, "TMEM holds 512 columns");
    static_assert(TMEM_COLS >= 32 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "an allocation is a power of two >= 32 columns");
    constexpr uint32_t IDESC = ptx::idesc_e4m3_f32(BM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + L::B_OFF;
    float *scl = reinterpret_cast<float *>(smem + L::SCALE_OFF);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint64_t *empty = full + STAGES;
    uint64_t *sfull = empty + STAGES;
    uint64_t *sempty = sfull + SCALE_STAGES;
    uint64_t *tfull = sempty + SCALE_STAGES;
    uint64_t *tempty = tfull + MAX_TBUF;
    uint64_t *mma_done = tempty + MAX_TBUF;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(mma_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = args.groups;
    const int num_work = args.tiles_m * args.tiles_n;
    const int work_first = static_cast<int>(blockIdx.x);
    const int work_stride = static_cast<int>(gridDim.x);
    auto coords = [&](int w, int &tm, int &tn) {
        tile_coords(w, args.tiles_m, args.tiles_n, args.band, args.band_n, tm, tn);
    };

    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            for (int s = 0; s < STAGES; ++s) {
                ptx::mbar_init(&full[s], 1);
                ptx::mbar_init(&empty[s], 1);   // the first promotion warp
            }
            for (int s = 0; s < SCALE_STAGES; ++s) {
                // (the scale slots' fill is counted on the TMEM-full barriers)
                ptx::mbar_init(&sfull[s], 1);
                ptx::mbar_init(&sempty[s], 4 * NWG);   // one arrival per promotion warp
            }
            for (uint32_t b = 0; b < NBUF; ++b) {
                // the group's commit, and the scale loader: its expect-tx arrival
                // (per-column scales) or every one of its lanes (block scales)
                ptx::mbar_init(&tfull[b], SB_PER_COLUMN ? 2 : 33);
                ptx::mbar_init(&tempty[b], 4 * NWG);   // one arrival per promotion warp
            }
            ptx::mbar_init(mma_done, 2);   // one final commit per MMA issuer
            *abort_flag = 0;
            ptx::fence_mbar_init();
            ptx::tma_prefetch_desc(&tmap_a);
            ptx::tma_prefetch_desc(&tmap_b);
        }
        __syncwarp();
        ptx::tmem_alloc(tmem_holder, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    // Programmatic dependent launch: the set-up above (barriers, TMEM, tensor
    // map prefetch) may overlap the previous kernel of the stream; no global
    // memory is read or written before that kernel has completed and its
    // writes are visible.  Then the next kernel may begin its own set-up.
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
    const uint32_t tmem_base = *tmem_holder;

    if (warp < FIRST_PROMO_WARP) {
        ptx::setmaxnreg_dec<RegSplit<BN>::CTRL>();
        if (warp == PRODUCER_WARP) {
            // -------------------------------------------------- TMA producer
            if (lane == 0) {
                int stage = 0;
                uint32_t phase = 0;
                uint32_t issued_mask = 0, issued_parity = 0;
                const uint64_t pol_a = args.stream_a ? ptx::l2_policy_evict_first() : ptx::l2_policy_evict_normal();
                const uint64_t pol_b = args.stream_b ? ptx::l2_policy_evict_first() : ptx::l2_policy_evict_normal();
                bool ok = true;
                for (int tile = work_first; ok && tile < num_work; tile += work_stride) {
                    int tm, tn;
                    coords(tile, tm, tn);
                    for (int g = 0; g < G; ++g) {
                        if (!ptx::mbar_wait(&empty[stage], phase ^ 1u, abort_flag, args.err, ERRBIT_PRODUCER,
                                            WAIT_TIMEOUT_NS)) {
                            ok = false;
                            break;
                        }
                        ptx::mbar_arrive_expect_tx(&full[stage], args.stage_bytes);
                        ptx::tma_load_2d_hint(sA + stage * L::A_BYTES, &tmap_a, &full[stage], g * BK, tm * BM, pol_a);
                        ptx::tma_load_2d_hint(sB + stage * L::B_BYTES, &tmap_b, &full[stage], g * BK, tn * BN, pol_b);
                        issued_mask |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
                if (!ok) {
                    // drain: every copy this thread started must land before exit
                    for (int s = 0; s < STAGES; ++s)
                        if (issued_mask & (1u << s))
                            ptx::mbar_wait(&full[s], (issued_parity >> s) & 1u, nullptr, args.err, ERRBIT_DRAIN,
                                           WAIT_TIMEOUT_NS);
                }
            }
            __syncwarp();
        } else if (warp == MMA_WARP || warp == SECOND_MMA_WARP) {
            // -------------------------------------------------- MMA issuer(s)
            if (lane == 0) {
                const uint32_t parity = warp == MMA_WARP ? 0u : 1u;   // groups this issuer takes
                uint32_t it = 0;   // global group counter -> smem stage, TMEM buffer, phases
                bool ok = true;
                const uint32_t a_base = ptx::smem_u32(sA);
                const uint32_t b_base = ptx::smem_u32(sB);
                for (int tile = work_first; ok && tile < num_work; tile += work_stride) {
                    for (int g = 0; g < G; ++g, ++it) {
                        if ((it & 1u) != parity)
                            continue;
                        const int stage = static_cast<int>(it % STAGES);
                        const uint32_t phase = (it / STAGES) & 1u;
                        const uint32_t buf = it % NBUF;
                        const uint32_t bphase = (it / NBUF) & 1u;
                        // the stage's data first: it is almost always there already, so
                        // once the TMEM buffer comes back the MMAs go out at once (+2.5 %
                        // Fprop and Dgrad against the other order)
                        if (!ptx::mbar_wait(&full[stage], phase, abort_flag, args.err, ERRBIT_MMA_SMEM,
                                            WAIT_TIMEOUT_NS) ||
                            !ptx::mbar_wait(&tempty[buf], bphase ^ 1u, abort_flag, args.err, ERRBIT_MMA_TMEM,
                                            WAIT_TIMEOUT_NS)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint64_t adesc = ptx::smem_desc_sw128_kmajor(a_base + stage * L::A_BYTES);
                        const uint64_t bdesc = ptx::smem_desc_sw128_kmajor(b_base + stage * L::B_BYTES);
                        const uint32_t d_tmem = tmem_base + buf * BN;
#pragma unroll
                        for (int j = 0; j < BK / 32; ++j)   // 32 bytes of K per instruction: +2 in the >>4 field
                            ptx::mma_f8(d_tmem, adesc + 2 * j, bdesc + 2 * j, IDESC, j > 0 ? 1u : 0u);
                        ptx::mma_commit(&tfull[buf]);
                    }
                }
                // all MMAs issued by this thread complete before teardown
                ptx::mma_commit(mma_done);
                ptx::mbar_wait(mma_done, 0, nullptr, args.err, ERRBIT_DRAIN, WAIT_TIMEOUT_NS);
            }
            __syncwarp();
        } else if (warp == SCALE_WARP && SB_PER_COLUMN) {
            // -------------------------------------------------- scale loader
            // Per-column scales: the group's 128 row scales and the tile's
            // column scales, both contiguous, by two bulk copies into the next
            // slot of a 4-slot ring, completing on the TMEM-full barrier of the
            // group's buffer (which therefore waits for the MMAs and the scales
            // together).  A slot is free once every promotion warp has handed
            // back the group that last used it; the copies may only be counted
            // on the buffer's barrier once its previous group has completed
            // there.
            if (lane == 0) {
                int ss = 0;
                uint32_t sphase = 0;
                uint32_t it = 0;   // global group counter -> TMEM buffer and phase
                bool ok = true;
                for (int tile = work_first; ok && tile < num_work; tile += work_stride) {
                    int tm, tn;
                    coords(tile, tm, tn);
                    const uint32_t col_bytes = static_cast<uint32_t>(min(BN, args.cols - tn * BN)) * 4u;
                    const float *sa_g = args.sa + tm * BM;     // group g's row scales, advanced per group
                    const float *sb_g = args.sb + tn * BN;     // and its column scales
                    for (int g = 0; g < G; ++g, ++it, sa_g += args.rows, sb_g += args.sb_stride_g) {
                        const uint32_t buf = it % NBUF;
                        if (!ptx::mbar_wait(&sempty[ss], sphase ^ 1u, abort_flag, args.err, ERRBIT_PROMOTE,
                                            WAIT_TIMEOUT_NS) ||
                            !ptx::mbar_wait(&tfull[buf], ((it / NBUF) & 1u) ^ 1u, abort_flag, args.err,
                                            ERRBIT_PROMOTE, WAIT_TIMEOUT_NS)) {
                            ok = false;
                            break;
                        }
                        float *dst = scl + ss * L::SCALE_FLOATS;
                        ptx::mbar_arrive_expect_tx(&tfull[buf], BM * 4 + col_bytes);
                        ptx::bulk_load_1d(dst, sa_g, BM * 4, &tfull[buf]);
                        ptx::bulk_load_1d(dst + BM, sb_g, col_bytes, &tfull[buf]);
                        if (++ss == SCALE_STAGES) {
                            ss = 0;
                            sphase ^= 1u;
                        }
                    }
                }
                if (!ok) {
                    // drain: the copies of the last groups must land before exit
                    // (their barriers complete only with the MMAs' commits too, so
                    // a wait may also run out: the copies have landed by then)
                    for (uint32_t k = 0; k < NBUF && k < it; ++k) {
                        const uint32_t j = it - 1 - k;
                        ptx::mbar_wait(&tfull[j % NBUF], (j / NBUF) & 1u, nullptr, args.err, ERRBIT_DRAIN,
                                       WAIT_TIMEOUT_NS);
                    }
                }
            }
            __syncwarp();
        } else if (warp == SCALE_WARP && L::READY) {
            // -------------------------------------------------- scale loader
            // Block scales.  Per group the slot receives the ready products
            // sa[row] * sb[block] for the tile's 128 rows and its one or two
            // 128-column blocks, so that a promotion thread reads one value per
            // group: a group's scale reads sit on its chain between the MMA's
            // completion and the TMEM load (measured: one read instead of two
            // reads and a product, +5.8 % on Fprop).  The raw scales come by
            // cp.async SCALE_RAW_AHEAD groups ahead into a small staging ring;
            // lane l takes rows 4l .. 4l+3 (one 16-byte copy when the row count
            // keeps them aligned, i.e. is a multiple of 4, else four 4-byte
            // copies).
            int rs = 0;
            uint32_t it = 0;   // global group counter -> TMEM buffer and phase, as the MMA issuers
            bool ok = true;
            float *raw = reinterpret_cast<float *>(smem + L::RAW_OFF);
            const int r = 4 * lane;
            for (int tile = work_first; ok && tile < num_work; tile += work_stride) {
                int tm, tn;
                coords(tile, tm, tn);
                const int row = tm * BM + r;
                auto stage_raw = [&](int gg, int slot) {
                    float *dst = raw + slot * L::RAW_FLOATS;
                    const float *sa_g = args.sa + static_cast<int64_t>(gg) * args.rows;
                    if ((args.rows & 3) == 0) {
                        const bool in = row < args.rows;
                        ptx::cp_async_16z(dst + r, in ? sa_g + row : args.sa, in ? 16u : 0u);
                    } else {
#pragma unroll 1
                        for (int e = 0; e < 4; ++e) {
                            const bool in = row + e < args.rows;
                            ptx::cp_async_4(dst + r + e, in ? sa_g + row + e : args.sa, in ? 4u : 0u);
                        }
                    }
                    if (lane < L::NBLK) {
                        const int col = tn * BN + lane * 128;
                        const bool in = col < args.cols;
                        const float *sb_g = args.sb + static_cast<int64_t>(gg) * args.sb_stride_g;
                        ptx::cp_async_4(dst + BM + lane,
                                        in ? sb_g + static_cast<int64_t>(col >> 7) * args.sb_stride_c : args.sb,
                                        in ? 4u : 0u);
                    }
                };
                // the tile's first groups (one commit group each, empty past G)
#pragma unroll
                for (int k = 0; k < SCALE_RAW_AHEAD; ++k) {
                    if (k < G)
                        stage_raw(k, (rs + k) % L::RAW_SLOTS);
                    ptx::cp_async_commit();
                }
                for (int g = 0; g < G; ++g, ++it) {
                    __syncwarp();                // every lane is done with the slot refilled next
                    if (g + SCALE_RAW_AHEAD < G)
                        stage_raw(g + SCALE_RAW_AHEAD, (rs + SCALE_RAW_AHEAD) % L::RAW_SLOTS);
                    ptx::cp_async_commit();
                    ptx::cp_async_wait<SCALE_RAW_AHEAD>();   // this lane's copies of group g have landed
                    __syncwarp();                            // and every lane's
                    // the group's slot belongs to its TMEM buffer: free when the
                    // promotion warps have handed that buffer back
                    const uint32_t buf = it % NBUF;
                    if (!ptx::mbar_wait(&tempty[buf], ((it / NBUF) & 1u) ^ 1u, abort_flag, args.err, ERRBIT_PROMOTE,
                                        WAIT_TIMEOUT_NS)) {
                        ok = false;
                        break;
                    }
                    const float *src = raw + rs * L::RAW_FLOATS;
                    const float4 a = *reinterpret_cast<const float4 *>(src + r);
                    float *dst = scl + buf * L::SCALE_FLOATS;
#pragma unroll
                    for (int b = 0; b < L::NBLK; ++b) {
                        const float sb = src[BM + b];
                        *reinterpret_cast<float4 *>(dst + b * BM + r) =
                            make_float4(a.x * sb, a.y * sb, a.z * sb, a.w * sb);
                    }
                    ptx::mbar_arrive(&tfull[buf]);   // every lane, after its own stores
                    if (++rs == L::RAW_SLOTS)
                        rs = 0;
                }
            }
            ptx::cp_async_wait_all();
        } else if (warp == SCALE_WARP && !SB_PER_COLUMN) {
            // -------------------------------------------------- scale loader
            // Narrow block-scale tiles: the group's 128 row scales and the
            // tile's block scale, by cp.async, straight into the slot of the
            // group's TMEM buffer; their completion is counted on that buffer's
            // TMEM-full barrier.
            uint32_t it = 0;   // global group counter -> TMEM buffer and phase, as the MMA issuers
            bool ok = true;
            for (int tile = work_first; ok && tile < num_work; tile += work_stride) {
                int tm, tn;
                coords(tile, tm, tn);
                for (int g = 0; g < G; ++g, ++it) {
                    const uint32_t buf = it % NBUF;
                    if (!ptx::mbar_wait(&tempty[buf], ((it / NBUF) & 1u) ^ 1u, abort_flag, args.err, ERRBIT_PROMOTE,
                                        WAIT_TIMEOUT_NS)) {
                        ok = false;
                        break;
                    }
                    float *dst = scl + buf * L::SCALE_FLOATS;
                    const float *sa_g = args.sa + static_cast<int64_t>(g) * args.rows;
                    // lane l: rows 4l .. 4l+3 of the tile, one 16-byte copy when
                    // the row count keeps them 16-byte aligned (every row count
                    // that is a multiple of 4), else four 4-byte copies (one
                    // 16-byte copy instead of four measured +2 % on Fprop / Dgrad:
                    // fewer copies queue in front of the promotion warps' shared
                    // memory traffic)
                    const int r = 4 * lane;
                    const int row = tm * BM + r;
                    if ((args.rows & 3) == 0) {
                        const bool in = row < args.rows;
                        ptx::cp_async_16z(dst + r, in ? sa_g + row : args.sa, in ? 16u : 0u);
                    } else {
#pragma unroll 1
                        for (int e = 0; e < 4; ++e) {
                            const bool in = row + e < args.rows;
                            ptx::cp_async_4(dst + r + e, in ? sa_g + row + e : args.sa, in ? 4u : 0u);
                        }
                    }
                    const float *sb_g = args.sb + static_cast<int64_t>(g) * args.sb_stride_g;
                    if (lane == 0) {
                        const int col = tn * BN;
                        const bool in = col < args.cols;
                        ptx::cp_async_4(dst + BM, in ? sb_g + static_cast<int64_t>(col >> 7) * args.sb_stride_c : args.sb,
                                        in ? 4u : 0u);
                    }
                    ptx::cp_async_mbar_arrive_noinc(&tfull[buf]);
                }
            }
            ptx::cp_async_wait_all();
        }
    } else {
        ptx::setmaxnreg_inc<RegSplit<BN>::PROMO>();
        // ------------------------------------------------------ promotion
        const int wg = (warp - FIRST_PROMO_WARP) >> 2;   // 0 or 1: column half of the tile
        // (with narrow tiles the second warpgroup has no columns and skips the loop)
        const int quarter = warp & 3;                    // TMEM lanes 32*quarter .. +31
        const int row_in_tile = quarter * 32 + lane;
        uint8_t *out_stage = smem + L::OUT_OFF + (warp - FIRST_PROMO_WARP) * 2 * L::OUT_CHUNK_BYTES;
        const uint64_t pol_d = args.stream_d ? ptx::l2_policy_evict_first() : ptx::l2_policy_evict_normal();
        uint32_t it = 0;
        int ss = 0;
        uint32_t sphase = 0;
        bool ok = true;
        for (int tile = work_first; ok && wg < NWG && tile < num_work; tile += work_stride) {
            int tm, tn;
            coords(tile, tm, tn);
            const int col0 = tn * BN + wg * COLS_PER_WG;
            // fp32 accumulators as packed pairs of adjacent columns: with one
            // scale per 128-column block, this thread's row (pair i = columns
            // 2i, 2i+1); with a scale per column, four rows r = 8k + lane/4 of
            // the warp's 32 (k = 0..3) at columns 8b + 2(lane%4) + {0, 1} of
            // each 8-column block b (pair k * CB + b)
            uint64_t acc2[SB_PER_COLUMN ? 1 : COLS_PER_WG / 2];
            uint64_t accp[SB_PER_COLUMN ? COLS_PER_WG / 2 : 1];
#pragma unroll
            for (int i = 0; i < (SB_PER_COLUMN ? 1 : COLS_PER_WG / 2); ++i)
                acc2[i] = 0ull;
#pragma unroll
            for (int i = 0; i < (SB_PER_COLUMN ? COLS_PER_WG / 2 : 1); ++i)
                accp[i] = 0ull;

            for (int g = 0; g < G; ++g, ++it) {
                const uint32_t buf = it % NBUF;
                const uint32_t bphase = (it / NBUF) & 1u;
                // The TMEM-full barrier also means that the group's scales have
                // landed (one wait per group instead of two: +8 % on the 256-wide
                // Fprop and Dgrad tiles).  Block scales sit in the slot of the
                // buffer, free again with it; per-column scales, read until the
                // last multiply-add, in a ring of their own, handed back at the
                // end of the group.
                const float *scur = scl + (SB_PER_COLUMN ? static_cast<uint32_t>(ss) : buf) * L::SCALE_FLOATS;
                const float *sbcol = scur + BM + wg * COLS_PER_WG;
                if (!ptx::mbar_wait(&tfull[buf], bphase, abort_flag, args.err, ERRBIT_PROMOTE, WAIT_TIMEOUT_NS)) {
                    ok = false;
                    break;
                }
                float w_blk = 0.0f;
                if constexpr (L::READY)
                    w_blk = scur[((wg * COLS_PER_WG) / 128) * BM + row_in_tile];   // the loader's sa * sb
                else if constexpr (!SB_PER_COLUMN)
                    w_blk = scur[row_in_tile] * scur[BM];
                ptx::tc_fence_after();
                if (warp == FIRST_PROMO_WARP) {                  // the group's MMAs are done with it
                    if (SB_PER_COLUMN) {
                        if (lane == 0)
                            ptx::mbar_arrive(&empty[it % STAGES]);
                    } else {
                        ptx::mbar_arrive_elected(&empty[it % STAGES]);
                    }
                }
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + buf * BN +
                                       wg * COLS_PER_WG;
                if (SB_PER_COLUMN) {
                    // acc += p * (sa[row] * sb[col]), two columns at a time
                    // (packed fp32 multiply and fused multiply-add, each lane
                    // rounded as the scalar operation would be)
                    const int cq = 2 * (lane & 3);
                    uint64_t sa2[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float v = scur[quarter * 32 + 8 * k + (lane >> 2)];
                        sa2[k] = ptx::pack_f32x2(v, v);
                    }
#pragma unroll
                    for (int j = 0; j < NPS; ++j) {
                        // the slab's partials (lanes 0-15 and 16-31 of the
                        // quarter), loaded and waited for as packed column pairs:
                        // +7 % against loads into loose 32-bit registers issued a
                        // slab ahead, whose pairs had to be moved together before
                        // every packed multiply-add (and a wait drains every
                        // pending load anyway)
                        uint64_t p0[8], p1[8];
                        ptx::tmem_ld_16x256b_x4_pair_packed(taddr + j * 8 * PS, p0, p1);
                        // this slab's column-scale pairs (read with no TMEM load
                        // pending: a shared load queued behind one waits for it)
                        uint64_t sb2[PS];
#pragma unroll
                        for (int i = 0; i < PS; ++i)
                            sb2[i] = *reinterpret_cast<const uint64_t *>(sbcol + 8 * (j * PS + i) + cq);
                        if (j + 1 == NPS) {
                            // the whole partial is in registers: hand the buffer back
                            ptx::tc_fence_before();
                            __syncwarp();
                            ptx::mbar_arrive_elected(&tempty[buf]);
                        }
#pragma unroll
                        for (int i = 0; i < PS; ++i) {
                            const int b = j * PS + i;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint64_t pp = (k < 2 ? p0 : p1)[2 * i + (k & 1)];
                                const uint64_t w = ptx::mul_f32x2(sa2[k], sb2[i]);
                                ptx::fma_f32x2(accp[k * CB + b], pp, w);
                            }
                        }
                    }
                } else {
                    // acc += partial * (sa * sb) for 32 columns starting at
                    // column c0 of this warpgroup's range; one 64-column load
                    // per wait where the range allows (against two 32-column
                    // loads: +1.5 %), so each group pays the TMEM load latency
                    // only COLS_PER_WG / 64 times
                    auto apply32 = [&](const uint64_t *p, const int c0) {
                        const uint64_t w2 = ptx::pack_f32x2(w_blk, w_blk);
                        uint64_t *a0 = acc2 + c0 / 2;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            ptx::fma_f32x2(a0[i], p[i], w2);
                    };
                    // partials loaded and waited for as packed column pairs
                    // (no moves to pair loose registers before each multiply-add)
                    if (LPW == 2) {
#pragma unroll
                        for (int h = 0; h < CHUNKS / 2; ++h) {
                            uint64_t pp[32];
                            ptx::tmem_ld_32x32b_x64_packed(taddr + h * 64, pp);
                            if (h + 1 == CHUNKS / 2) {
                                // the whole partial is in registers: hand the buffer back
                                ptx::tc_fence_before();
                                __syncwarp();
                                ptx::mbar_arrive_elected(&tempty[buf]);
                            }
                            apply32(pp, h * 64);
                            apply32(pp + 16, h * 64 + 32);
                        }
                    } else {
                        uint64_t p0[16];
                        ptx::tmem_ld_32x32b_x32_packed(taddr, p0);
                        ptx::tc_fence_before();
                        __syncwarp();
                        ptx::mbar_arrive_elected(&tempty[buf]);
                        apply32(p0, 0);
                    }
                }
                if (SB_PER_COLUMN) {
                    __syncwarp();
                    ptx::mbar_arrive_elected(&sempty[ss]);
                }
                if (++ss == SCALE_STAGES) {
                    ss = 0;
                    sphase ^= 1u;
                }
            }
            if (!ok)
                break;
            // Epilogue: bf16 rows of this warp (32 rows x COLS_PER_WG) leave through
            // shared memory in 16-column chunks, each written by one TMA store
            // (rows or columns past the tensor are clipped by the copy engine).
            if (col0 < args.cols) {
#pragma unroll
                for (int c = 0; c < COLS_PER_WG / 16; ++c) {
                    uint8_t *chunk = out_stage + (c & 1) * L::OUT_CHUNK_BYTES;
                    if (lane == 0)
                        ptx::bulk_wait_read<1>();          // the store that last used this buffer has read it
                    __syncwarp();
                    if (SB_PER_COLUMN) {
                        // chunk c is blocks 2c and 2c+1; a row of the chunk is 32 bytes
#pragma unroll
                        for (int k = 0; k < 4; ++k)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const uint64_t a = accp[k * CB + 2 * c + e];
                                *reinterpret_cast<uint32_t *>(chunk + (8 * k + (lane >> 2)) * 32 + e * 16 +
                                                              (lane & 3) * 4) = pack_bf16x2(ptx::lo_f32(a), ptx::hi_f32(a));
                            }
                    } else {
                        uint4 *dst = reinterpret_cast<uint4 *>(chunk + lane * 32);
                        uint4 o0, o1;
                        float v[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            v[k] = (k & 1) ? ptx::hi_f32(acc2[8 * c + k / 2]) : ptx::lo_f32(acc2[8 * c + k / 2]);
                        o0.x = pack_bf16x2(v[0], v[1]);
                        o0.y = pack_bf16x2(v[2], v[3]);
                        o0.z = pack_bf16x2(v[4], v[5]);
                        o0.w = pack_bf16x2(v[6], v[7]);
                        o1.x = pack_bf16x2(v[8], v[9]);
                        o1.y = pack_bf16x2(v[10], v[11]);
                        o1.z = pack_bf16x2(v[12], v[13]);
                        o1.w = pack_bf16x2(v[14], v[15]);
                        dst[0] = o0;
                        dst[1] = o1;
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d_hint(&tmap_d, chunk, col0 + 16 * c, tm * BM + quarter * 32, pol_d);
                        ptx::bulk_commit();
                    }
                }
            }
        }
        if (lane == 0)
            ptx::bulk_wait_all();                          // stores complete before the CTA exits
        __syncwarp();
    }

    // ---------------------------------------------------------- teardown
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == PRODUCER_WARP)
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
}

// A's box height: a whole 128-row tile, or for a problem of fewer rows only the
// rows present (rounded up to the 8-row swizzle atom), so that no copy is spent
// on out-of-bounds fill.  The tile's rows beyond the box are never written by
// the copy; they only feed output rows past the problem, which are not stored.
int64_t a_box_rows(int64_t rows)
{
    return rows >= BM ? BM : ((rows + 7) / 8) * 8;
}

template <int BN, int STAGES, bool SB_PER_COLUMN, bool HALF_A = false>
cudaError_t launch_variant(const GemmProblem &p, const DeviceInfo &dev, const CUtensorMap &ta, const CUtensorMap &tb,
                           const CUtensorMap &td, cudaStream_t stream)
{
    using L = Smem<BN, STAGES, HALF_A, SB_PER_COLUMN>;
    static_assert(L::TOTAL <= 227 * 1024, "shared memory per CTA");
    static_assert(!HALF_A || !SB_PER_COLUMN, "the packed A tiles serve block-scale problems of <= 64 rows");
    auto kern = gemm_kernel<BN, STAGES, SB_PER_COLUMN, HALF_A>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(L::TOTAL));
    if (e != cudaSuccess)
        return e;
    KernelArgs a;
    a.sa = p.sa;
    a.sb = p.sb;
    a.sb_stride_g = p.sb_stride_g;
    a.sb_stride_c = p.sb_stride_c;
    a.d = static_cast<__nv_bfloat16 *>(p.d);
    a.err = dev.err_word;
    a.rows = static_cast<int32_t>(p.rows);
    a.cols = static_cast<int32_t>(p.cols);
    a.groups = static_cast<int32_t>(p.kdim / BK);
    a.tiles_m = static_cast<int32_t>((p.rows + BM - 1) / BM);
    a.tiles_n = static_cast<int32_t>((p.cols + BN - 1) / BN);
    // Tile order and L2 priorities.  Every CTA of a wave walks the whole
    // contraction, so an operand is fetched from DRAM once per wave that
    // uses it unless it stays in L2 between waves.  Bands along m keep a
    // band of A in L2 and read B once per band; bands along n the reverse.
    // Each band's reused slice is at most L2_BAND_BYTES; the cheaper axis
    // (reused operand once + the other once per band) is compared with the
    // balanced order (bands of 16 m-tiles, every wave reading its own
    // operand slices), and a band is used only when it promises under 0.8
    // of the balanced order's bytes: with long contractions the slices that
    // one wave streams are as large as the L2 and the reuse does not
    // materialise (measured).  With a band, the operand read once per band
    // is loaded with the evict-first priority so that it does not push the
    // reused slice out.  The order never changes how an output element is
    // reduced.
    const int64_t a_bytes = p.rows * p.kdim, b_bytes = p.cols * p.kdim;
    const int64_t a_tile = int64_t{BM} * p.kdim, b_tile = int64_t{BN} * p.kdim;
    auto clamp_band = [](int64_t v, int64_t hi) { return v < 1 ? int64_t{1} : (v > hi ? hi : v); };
    const int64_t band_m = clamp_band(L2_BAND_BYTES / a_tile, a.tiles_m);
    const int64_t band_n = clamp_band(L2_BAND_BYTES / b_tile, a.tiles_n);
    const int64_t cost_m = a_bytes + b_bytes * ((a.tiles_m + band_m - 1) / band_m);
    const int64_t cost_n = b_bytes + a_bytes * ((a.tiles_n + band_n - 1) / band_n);
    const int64_t bal_m = a.tiles_m < BALANCED_BAND_M ? a.tiles_m : BALANCED_BAND_M;
    const int64_t bal_n_per_wave = (dev.sm_count + bal_m - 1) / bal_m;
    const int64_t bal_n = bal_n_per_wave < a.tiles_n ? bal_n_per_wave : a.tiles_n;
    const int64_t waves = (int64_t{a.tiles_m} * a.tiles_n + dev.sm_count - 1) / dev.sm_count;
    const int64_t cost_bal = waves * (bal_m * a_tile + bal_n * b_tile);
    const int64_t cost_band = cost_n < cost_m ? cost_n : cost_m;
    a.stream_a = a.stream_b = 0;
    if (5 * cost_band < 4 * cost_bal) {
        a.band_n = cost_n < cost_m ? 1 : 0;
        a.band = static_cast<int32_t>(a.band_n ? band_n : band_m);
        a.stream_a = a.band_n ? 1 : 0;
        a.stream_b = a.band_n ? 0 : 1;
    } else {
        a.band_n = 0;
        a.band = static_cast<int32_t>(bal_m);
    }
    a.stream_d = p.rows * p.cols * 2 > 2 * L2_BAND_BYTES ? 1 : 0;
    a.stage_bytes = static_cast<uint32_t>(a_box_rows(p.rows)) * BK + L::B_BYTES;
    const int work = a.tiles_m * a.tiles_n;
    const int grid = work < dev.sm_count ? work : dev.sm_count;
    // launched as a programmatic dependent of the stream's previous kernel
    // (the kernel itself waits for it before touching global memory)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = L::TOTAL;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, td, a);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

CUresult encode_operand(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *map, const uint8_t *ptr,
                        int64_t rows, int64_t kdim, int box_rows)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kdim), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kdim)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// bf16 output [rows][cols]: boxes of 32 rows x 16 columns (32-byte rows), no swizzle.
CUresult encode_output(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap *map, void *ptr, int64_t rows,
                       int64_t cols)
{
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

cudaError_t launch_gemm(const GemmProblem &p, const DeviceInfo &dev, PFN_cuTensorMapEncodeTiled_v12000 encode,
                        cudaStream_t stream)
{
    // Tile width: the fewest waves of tiles over the SMs, and among widths
    // with that many waves the narrowest (more CTAs streaming B).  A tile's
    // time is set mostly by its number of K groups, not its width, so extra
    // waves cost more than idle SMs (measured on the 8B-class decode shapes:
    // this rule picks the fastest width on every one).  Training-sized
    // problems get 128 x 256 tiles.  The width never changes how an output
    // element is reduced.
    const int64_t tm_count = (p.rows + BM - 1) / BM;
    int bn = 256;
    int64_t best_waves = -1;
    for (int w : {256, 128, 64, 32}) {
        const int64_t tiles = tm_count * ((p.cols + w - 1) / w);
        const int64_t waves = (tiles + dev.sm_count - 1) / dev.sm_count;
        if (best_waves < 0 || waves <= best_waves) {   // ties: the narrower width (later in the list)
            best_waves = waves;
            bn = w;
        }
    }
    const bool per_col = p.sb_mode == ScaleB::PerColumn;
    const bool half_a = !per_col && p.rows <= BM / 2;   // decode: A fits a 64-row box
    CUtensorMap ta, tb, td;
    if (encode_operand(encode, &ta, p.a, p.rows, p.kdim, static_cast<int>(a_box_rows(p.rows))) != CUDA_SUCCESS ||
        encode_operand(encode, &tb, p.b, p.cols, p.kdim, bn) != CUDA_SUCCESS ||
        encode_output(encode, &td, p.d, p.rows, p.cols) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (half_a) {
        switch (bn) {
        case 256: return launch_variant<256, 4, false, true>(p, dev, ta, tb, td, stream);
        case 128: return launch_variant<128, 8, false, true>(p, dev, ta, tb, td, stream);
        case 64: return launch_variant<64, 12, false, true>(p, dev, ta, tb, td, stream);
        default: return launch_variant<32, 16, false, true>(p, dev, ta, tb, td, stream);
        }
    }
    switch (bn) {
    case 256:
        return per_col ? launch_variant<256, 4, true>(p, dev, ta, tb, td, stream)
                       : launch_variant<256, 4, false>(p, dev, ta, tb, td, stream);
    case 128:
        return per_col ? launch_variant<128, 6, true>(p, dev, ta, tb, td, stream)
                       : launch_variant<128, 6, false>(p, dev, ta, tb, td, stream);
    case 64:
        return per_col ? launch_variant<64, 8, true>(p, dev, ta, tb, td, stream)
                       : launch_variant<64, 8, false>(p, dev, ta, tb, td, stream);
    default:
        return per_col ? launch_variant<32, 9, true>(p, dev, ta, tb, td, stream)
                       : launch_variant<32, 9, false>(p, dev, ta, tb, td, stream);
    }
}

// ---------------------------------------------------------------------------
// Watchdog self-test: one warp waits, bounded, on a barrier that nothing
// completes, using the same routine as the GEMM's waits.
// ---------------------------------------------------------------------------
namespace {
__global__ void watchdog_selftest_kernel(uint32_t *err, uint64_t timeout_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        ptx::mbar_wait(&bar, 0, &abort_flag, err, ERRBIT_SELFTEST, timeout_ns);
    __syncthreads();
}
}  // namespace

cudaError_t launch_watchdog_selftest(uint32_t *err_word, uint64_t timeout_ns, cudaStream_t stream)
{
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>(err_word, timeout_ns);
    return cudaGetLastError();
}

}  // namespace jetfp8
