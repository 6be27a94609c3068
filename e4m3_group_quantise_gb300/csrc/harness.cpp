// jetfp8_bench: a native timing harness for the jetfp8 C-ABI on one GPU.
//
// It runs the FP8 training step of a linear layer (Jet-RL, technical
// summaries on gist.science, "Schéma de Quantification": 128x128 weight
// blocks, 1x128 activation and gradient groups, 1x128 / 128x1 groups for
// WGrad) over the four projections of an 8B- or 32B-class decoder layer:
// per projection quantise W (codes + transposed codes), quantise X and dY
// into both layouts (jetfp8_quantize_act_dual), then Fprop, Dgrad and Wgrad.
// Everything goes through the public C functions of include/jetfp8.h; this
// program only allocates memory, creates streams and events, and times.
//
//   jetfp8_bench [--workload train-8b|train-32b] [--steps K] [--warmup W]
//                [--streams 1|2] [--seed S] [--no-e2e] [--e2e-steps E]
//                [--device D]
//
// Timed quantities (CUDA events on the launching streams, after warm-up):
//   value    the step with every input already in device memory: GEMM
//            TFLOP/s = (Fprop + Dgrad + Wgrad flops) / step time;
//   kernels  each launch between events in a serial pass after the timed
//            region (per-kernel milliseconds per step);
//   e2e      the same step from pinned host memory: every step copies X, W
//            and dY of each projection in and Y, dX, dW back out, the next
//            projection's inputs travelling while this one computes.
// The device error word is read after every synchronisation; a kernel whose
// bounded wait gave up fails the run.  Inputs are seeded synthetic bf16:
// X ~ N(0,1) (8B: 1% of channels x20) or Student-t(3) (32B: 1% of channels
// x100), W ~ N(0,0.02), dY ~ N(0,1e-2) (8B) or N(0,1e-3) (32B), drawn on the
// host from a counter-based generator (splitmix64, Box-Muller).
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "jetfp8.h"

namespace {

void fail(const char *what, const char *detail)
{
    std::fprintf(stderr, "jetfp8_bench: %s: %s\n", what, detail);
    std::exit(1);
}

void cuda_ok(cudaError_t e, const char *what)
{
    if (e != cudaSuccess)
        fail(what, cudaGetErrorString(e));
}

void lib_ok(jetfp8_status st, const char *what)
{
    if (st != JETFP8_OK)
        fail(what, jetfp8_status_string(st));
}

// ------------------------------------------------------------ inputs
uint64_t splitmix64(uint64_t x)
{
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

// Uniform in (0, 1] from the top 53 bits.
double uniform(uint64_t key) { return (static_cast<double>(splitmix64(key) >> 11) + 1.0) * 0x1.0p-53; }

// Standard normal number `i` of stream `stream` (Box-Muller on two uniforms).
double normal(uint64_t stream, uint64_t i)
{
    const uint64_t base = splitmix64(stream ^ 0x5851F42D4C957F2Dull) + 2 * i;
    const double u1 = uniform(base), u2 = uniform(base + 1);
    return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586 * u2);
}

uint16_t to_bf16(float f)   // round to nearest even (finite inputs)
{
    uint32_t b;
    std::memcpy(&b, &f, 4);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return static_cast<uint16_t>(b >> 16);
}

enum class Dist { Normal, StudentT3 };

// rows x cols bf16 values, sigma * N(0,1) or Student-t(3) = N / sqrt(chi2_3 / 3);
// `outlier_cols` columns scaled by `outlier_scale` before rounding.
void fill(uint16_t *dst, int64_t rows, int64_t cols, Dist dist, double sigma, uint64_t stream,
          const std::vector<int64_t> &outlier_cols, double outlier_scale)
{
    std::vector<float> colscale(static_cast<size_t>(cols), 1.0f);
    for (int64_t c : outlier_cols)
        colscale[static_cast<size_t>(c)] = static_cast<float>(outlier_scale);
    const unsigned nt = std::max(1u, std::thread::hardware_concurrency());
    std::vector<std::thread> pool;
    for (unsigned t = 0; t < nt; ++t) {
        pool.emplace_back([=, &colscale]() {
            for (int64_t r = t; r < rows; r += nt) {
                for (int64_t c = 0; c < cols; ++c) {
                    const uint64_t i = static_cast<uint64_t>(r * cols + c);
                    double v = normal(stream, i);
                    if (dist == Dist::StudentT3) {
                        double chi = 0.0;
                        for (int d = 0; d < 3; ++d) {
                            const double z = normal(stream + 1000003ull * (d + 1), i);
                            chi += z * z;
                        }
                        v /= std::sqrt(chi / 3.0);
                    }
                    dst[r * cols + c] = to_bf16(static_cast<float>(v * sigma) * colscale[static_cast<size_t>(c)]);
                }
            }
        });
    }
    for (auto &th : pool)
        th.join();
}

std::vector<int64_t> pick_outliers(int64_t cols, uint64_t seed)
{
    const int64_t n = static_cast<int64_t>(std::llround(0.01 * static_cast<double>(cols)));
    std::vector<int64_t> perm(static_cast<size_t>(cols));
    for (int64_t i = 0; i < cols; ++i)
        perm[static_cast<size_t>(i)] = i;
    for (int64_t i = cols - 1; i > 0; --i) {   // Fisher-Yates with the counter-based generator
        const int64_t j = static_cast<int64_t>(splitmix64(seed * 7919ull + static_cast<uint64_t>(i)) %
                                               static_cast<uint64_t>(i + 1));
        std::swap(perm[static_cast<size_t>(i)], perm[static_cast<size_t>(j)]);
    }
    perm.resize(static_cast<size_t>(n));
    return perm;
}

// ------------------------------------------------------------ workload
struct Workload {
    const char *name;
    int64_t tokens;
    Dist xdist;
    double outlier_scale, dy_sigma;
    struct {
        const char *name;
        int64_t n, k;
    } proj[4];
};

const Workload kWorkloads[] = {
    {"train-8b", 16384, Dist::Normal, 20.0, 1e-2,
     {{"qkv", 6144, 4096}, {"o", 4096, 4096}, {"gate_up", 28672, 4096}, {"down", 4096, 14336}}},
    {"train-32b", 32768, Dist::StudentT3, 100.0, 1e-3,
     {{"qkv", 7168, 5120}, {"o", 5120, 5120}, {"gate_up", 55296, 5120}, {"down", 5120, 27648}}},
};

template <typename T>
T *dev_alloc(size_t count)
{
    void *p = nullptr;
    cuda_ok(cudaMalloc(&p, count * sizeof(T)), "cudaMalloc");
    return static_cast<T *>(p);
}

template <typename T>
T *host_alloc(size_t count)
{
    void *p = nullptr;
    cuda_ok(cudaMallocHost(&p, count * sizeof(T)), "cudaMallocHost");
    return static_cast<T *>(p);
}

struct Proj {
    std::string name;
    int64_t m, n, k;
    // device
    uint16_t *x, *w, *dy, *y, *dx, *dw;
    uint8_t *qw, *qwt, *qx, *qxt, *qdy, *qdyt;
    float *sw, *sx, *sxt, *sdy, *sdyt;
    // pinned host copies of the inputs and room for the outputs
    uint16_t *hx, *hw, *hdy, *hy, *hdx, *hdw;
};

enum Kind { QUANT_W, QUANT_X_DUAL, QUANT_DY_DUAL, FPROP, DGRAD, WGRAD, NKIND };
const char *kKindName[NKIND] = {"quant_w", "quant_x_dual", "quant_dy_dual", "fprop", "dgrad", "wgrad"};

jetfp8_status launch(Proj &p, Kind kind, cudaStream_t s)
{
    switch (kind) {
    case QUANT_W: return jetfp8_quantize_weight(p.w, p.n, p.k, p.qw, p.sw, p.qwt, s);
    case QUANT_X_DUAL: return jetfp8_quantize_act_dual(p.x, p.m, p.k, p.qx, p.sx, p.qxt, p.sxt, s);
    case QUANT_DY_DUAL: return jetfp8_quantize_act_dual(p.dy, p.m, p.n, p.qdy, p.sdy, p.qdyt, p.sdyt, s);
    case FPROP: return jetfp8_gemm_fprop(p.qx, p.sx, p.qw, p.sw, p.y, p.m, p.n, p.k, s);
    case DGRAD: return jetfp8_gemm_dgrad(p.qdy, p.sdy, p.qwt, p.sw, p.dx, p.m, p.n, p.k, s);
    default: return jetfp8_gemm_wgrad(p.qdyt, p.sdyt, p.qxt, p.sxt, p.dw, p.m, p.n, p.k, s);
    }
}

struct Streams {
    cudaStream_t main = nullptr, side = nullptr;
    std::vector<cudaEvent_t> pool;
    size_t next = 0;
    cudaEvent_t event()
    {
        if (next == pool.size()) {
            cudaEvent_t e;
            cuda_ok(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreate");
            pool.push_back(e);
        }
        return pool[next++];
    }
};

// Every projection's weight (codes + transposed codes) in one grouped launch.
jetfp8_status quantize_all_weights(std::vector<Proj> &projs, cudaStream_t s)
{
    const void *w[JETFP8_WEIGHT_GROUP_MAX];
    int64_t n[JETFP8_WEIGHT_GROUP_MAX], k[JETFP8_WEIGHT_GROUP_MAX];
    uint8_t *q[JETFP8_WEIGHT_GROUP_MAX], *qt[JETFP8_WEIGHT_GROUP_MAX];
    float *sc[JETFP8_WEIGHT_GROUP_MAX];
    const int count = static_cast<int>(projs.size());
    if (count > JETFP8_WEIGHT_GROUP_MAX)
        return JETFP8_ERR_SHAPE;
    for (int i = 0; i < count; ++i) {
        w[i] = projs[i].w;
        n[i] = projs[i].n;
        k[i] = projs[i].k;
        q[i] = projs[i].qw;
        sc[i] = projs[i].sw;
        qt[i] = projs[i].qwt;
    }
    return jetfp8_quantize_weight_group(count, w, n, k, q, sc, qt, s);
}

// One step on device-resident inputs.  It starts with one grouped launch that
// quantises every projection's weight (the master weights are all resident,
// so they share one launch's start-up and last stores); then per projection
// the X and dY quantisations and the three GEMMs.  With a side stream, each
// projection's dY quantisation and Wgrad run there (Wgrad after X's
// transposed codes exist; Dgrad on the main stream after dY's codes exist),
// so one GEMM's last partial wave is filled by the other's tiles.  With
// `timing`, every launch is bracketed by timing events recorded into
// timing[kind] (serial pass: main stream only).
void step(std::vector<Proj> &projs, Streams &st, bool two_streams,
          std::vector<std::pair<Kind, std::pair<cudaEvent_t, cudaEvent_t>>> *timing)
{
    st.next = 0;
    if (two_streams) {
        cudaEvent_t e = st.event();
        cuda_ok(cudaEventRecord(e, st.main), "record");
        cuda_ok(cudaStreamWaitEvent(st.side, e, 0), "wait");
    }
    {
        cudaEvent_t t0 = nullptr, t1 = nullptr;
        if (timing) {
            cuda_ok(cudaEventCreate(&t0), "cudaEventCreate");
            cuda_ok(cudaEventCreate(&t1), "cudaEventCreate");
            cuda_ok(cudaEventRecord(t0, st.main), "record");
        }
        lib_ok(quantize_all_weights(projs, st.main), "quant_w (grouped)");
        if (timing) {
            cuda_ok(cudaEventRecord(t1, st.main), "record");
            timing->push_back({QUANT_W, {t0, t1}});
        }
    }
    for (Proj &p : projs) {
        cudaEvent_t x_ready = nullptr, dy_ready = nullptr;
        for (int k = QUANT_X_DUAL; k < NKIND; ++k) {
            const Kind kind = static_cast<Kind>(k);
            cudaStream_t s = (two_streams && (kind == QUANT_DY_DUAL || kind == WGRAD)) ? st.side : st.main;
            if (two_streams && kind == DGRAD)
                cuda_ok(cudaStreamWaitEvent(s, dy_ready, 0), "wait");
            if (two_streams && kind == WGRAD)
                cuda_ok(cudaStreamWaitEvent(s, x_ready, 0), "wait");
            cudaEvent_t t0 = nullptr, t1 = nullptr;
            if (timing) {
                cuda_ok(cudaEventCreate(&t0), "cudaEventCreate");
                cuda_ok(cudaEventCreate(&t1), "cudaEventCreate");
                cuda_ok(cudaEventRecord(t0, s), "record");
            }
            lib_ok(launch(p, kind, s), kKindName[k]);
            if (timing) {
                cuda_ok(cudaEventRecord(t1, s), "record");
                timing->push_back({kind, {t0, t1}});
            }
            if (two_streams && kind == QUANT_X_DUAL) {
                x_ready = st.event();
                cuda_ok(cudaEventRecord(x_ready, s), "record");
            }
            if (two_streams && kind == QUANT_DY_DUAL) {
                dy_ready = st.event();
                cuda_ok(cudaEventRecord(dy_ready, s), "record");
            }
        }
    }
    if (two_streams) {
        cudaEvent_t e = st.event();
        cuda_ok(cudaEventRecord(e, st.side), "record");
        cuda_ok(cudaStreamWaitEvent(st.main, e, 0), "wait");
    }
}

void sync_and_check(const char *where)
{
    cuda_ok(cudaDeviceSynchronize(), where);
    lib_ok(jetfp8_poll_device_error(nullptr), where);
}

}  // namespace

int main(int argc, char **argv)
{
    const Workload *wl = &kWorkloads[0];
    int steps = 20, warmup = 5, streams = 2, e2e_steps = 10, device = 0;
    uint64_t seed = 1000;
    bool e2e = true;
    for (int i = 1; i < argc; ++i) {
        const std::string a = argv[i];
        auto next = [&]() -> const char * {
            if (i + 1 >= argc)
                fail("missing value for", a.c_str());
            return argv[++i];
        };
        if (a == "--workload") {
            const std::string w = next();
            wl = nullptr;
            for (const Workload &c : kWorkloads)
                if (w == c.name)
                    wl = &c;
            if (!wl)
                fail("unknown workload", w.c_str());
        } else if (a == "--steps") {
            steps = std::atoi(next());
        } else if (a == "--warmup") {
            warmup = std::atoi(next());
        } else if (a == "--streams") {
            streams = std::atoi(next());
        } else if (a == "--seed") {
            seed = std::strtoull(next(), nullptr, 10);
        } else if (a == "--e2e-steps") {
            e2e_steps = std::atoi(next());
        } else if (a == "--device") {
            device = std::atoi(next());
        } else if (a == "--no-e2e") {
            e2e = false;
        } else {
            fail("unknown argument", a.c_str());
        }
    }
    if (steps < 1 || warmup < 0 || e2e_steps < 1 || (streams != 1 && streams != 2))
        fail("arguments", "need --steps >= 1, --warmup >= 0, --e2e-steps >= 1, --streams 1 or 2");

    cuda_ok(cudaSetDevice(device), "cudaSetDevice");
    const auto t_gen = std::chrono::steady_clock::now();
    std::vector<Proj> projs;
    double flops = 0.0;
    uint64_t h2d = 0, d2h = 0;
    for (int i = 0; i < 4; ++i) {
        Proj p{};
        p.name = wl->proj[i].name;
        p.m = wl->tokens;
        p.n = wl->proj[i].n;
        p.k = wl->proj[i].k;
        const size_t mk = static_cast<size_t>(p.m * p.k), nk = static_cast<size_t>(p.n * p.k),
                     mn = static_cast<size_t>(p.m * p.n);
        p.hx = host_alloc<uint16_t>(mk);
        p.hw = host_alloc<uint16_t>(nk);
        p.hdy = host_alloc<uint16_t>(mn);
        p.hy = host_alloc<uint16_t>(mn);
        p.hdx = host_alloc<uint16_t>(mk);
        p.hdw = host_alloc<uint16_t>(nk);
        const uint64_t s0 = seed * 1000003ull + static_cast<uint64_t>(i) * 101ull;
        fill(p.hx, p.m, p.k, wl->xdist, 1.0, s0 + 1, pick_outliers(p.k, s0 + 4), wl->outlier_scale);
        fill(p.hw, p.n, p.k, Dist::Normal, 0.02, s0 + 2, {}, 1.0);
        fill(p.hdy, p.m, p.n, Dist::Normal, wl->dy_sigma, s0 + 3, {}, 1.0);
        p.x = dev_alloc<uint16_t>(mk);
        p.w = dev_alloc<uint16_t>(nk);
        p.dy = dev_alloc<uint16_t>(mn);
        p.y = dev_alloc<uint16_t>(mn);
        p.dx = dev_alloc<uint16_t>(mk);
        p.dw = dev_alloc<uint16_t>(nk);
        p.qw = dev_alloc<uint8_t>(nk);
        p.qwt = dev_alloc<uint8_t>(nk);
        p.sw = dev_alloc<float>(nk / 16384);
        p.qx = dev_alloc<uint8_t>(mk);
        p.sx = dev_alloc<float>(mk / 128);
        p.qxt = dev_alloc<uint8_t>(mk);
        p.sxt = dev_alloc<float>(mk / 128);
        p.qdy = dev_alloc<uint8_t>(mn);
        p.sdy = dev_alloc<float>(mn / 128);
        p.qdyt = dev_alloc<uint8_t>(mn);
        p.sdyt = dev_alloc<float>(mn / 128);
        cuda_ok(cudaMemcpy(p.x, p.hx, mk * 2, cudaMemcpyHostToDevice), "copy x");
        cuda_ok(cudaMemcpy(p.w, p.hw, nk * 2, cudaMemcpyHostToDevice), "copy w");
        cuda_ok(cudaMemcpy(p.dy, p.hdy, mn * 2, cudaMemcpyHostToDevice), "copy dy");
        flops += 3.0 * 2.0 * static_cast<double>(p.m) * static_cast<double>(p.n) * static_cast<double>(p.k);
        h2d += 2 * (mk + nk + mn);
        d2h += 2 * (mn + mk + nk);
        projs.push_back(p);
    }
    const double gen_s = std::chrono::duration<double>(std::chrono::steady_clock::now() - t_gen).count();

    Streams st;
    cuda_ok(cudaStreamCreateWithFlags(&st.main, cudaStreamNonBlocking), "cudaStreamCreate");
    cuda_ok(cudaStreamCreateWithFlags(&st.side, cudaStreamNonBlocking), "cudaStreamCreate");
    const bool two = streams == 2;

    // ---- device-resident step
    for (int i = 0; i < warmup; ++i)
        step(projs, st, two, nullptr);
    sync_and_check("warm-up");
    cudaEvent_t a, b;
    cuda_ok(cudaEventCreate(&a), "cudaEventCreate");
    cuda_ok(cudaEventCreate(&b), "cudaEventCreate");
    cuda_ok(cudaEventRecord(a, st.main), "record");
    for (int i = 0; i < steps; ++i)
        step(projs, st, two, nullptr);
    cuda_ok(cudaEventRecord(b, st.main), "record");
    sync_and_check("timed steps");
    float total_ms = 0.0f;
    cuda_ok(cudaEventElapsedTime(&total_ms, a, b), "elapsed");
    const double ms_step = total_ms / steps;

    // ---- per-kernel serial pass
    const int serial = 3;
    std::vector<std::pair<Kind, std::pair<cudaEvent_t, cudaEvent_t>>> timing;
    for (int i = 0; i < serial; ++i)
        step(projs, st, false, &timing);
    sync_and_check("serial pass");
    double kind_ms[NKIND] = {0};
    for (auto &t : timing) {
        float ms = 0.0f;
        cuda_ok(cudaEventElapsedTime(&ms, t.second.first, t.second.second), "elapsed");
        kind_ms[t.first] += ms / serial;
        cudaEventDestroy(t.second.first);
        cudaEventDestroy(t.second.second);
    }
    // device-resident steps: one grouped weight launch + five per projection;
    // end-to-end steps (below): six per projection
    int launches = (warmup + steps + serial) * (1 + static_cast<int>(projs.size()) * (NKIND - 1));

    // ---- end to end from pinned host memory
    double e2e_ms = 0.0;
    if (e2e) {
        cudaStream_t s_in, s_out;
        cuda_ok(cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking), "cudaStreamCreate");
        cuda_ok(cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking), "cudaStreamCreate");
        const size_t np = projs.size();
        std::vector<cudaEvent_t> landed(np), computed(np), copied(np);
        for (size_t i = 0; i < np; ++i) {
            cuda_ok(cudaEventCreateWithFlags(&landed[i], cudaEventDisableTiming), "cudaEventCreate");
            cuda_ok(cudaEventCreateWithFlags(&computed[i], cudaEventDisableTiming), "cudaEventCreate");
            cuda_ok(cudaEventCreateWithFlags(&copied[i], cudaEventDisableTiming), "cudaEventCreate");
        }
        std::vector<bool> first(np, true);
        // Per projection: inputs in on s_in (after the previous step's kernels
        // have read them), compute on the main stream once they have landed
        // (and the previous step's results have left), results out on s_out.
        // The weights arrive one projection at a time, so each is quantised
        // on its own as it lands (no grouped launch here).
        auto one = [&]() {
            for (size_t i = 0; i < np; ++i) {
                Proj &p = projs[i];
                const size_t mk = static_cast<size_t>(p.m * p.k), nk = static_cast<size_t>(p.n * p.k),
                             mn = static_cast<size_t>(p.m * p.n);
                if (!first[i])
                    cuda_ok(cudaStreamWaitEvent(s_in, computed[i], 0), "wait");
                cuda_ok(cudaMemcpyAsync(p.x, p.hx, mk * 2, cudaMemcpyHostToDevice, s_in), "h2d");
                cuda_ok(cudaMemcpyAsync(p.w, p.hw, nk * 2, cudaMemcpyHostToDevice, s_in), "h2d");
                cuda_ok(cudaMemcpyAsync(p.dy, p.hdy, mn * 2, cudaMemcpyHostToDevice, s_in), "h2d");
                cuda_ok(cudaEventRecord(landed[i], s_in), "record");
                cuda_ok(cudaStreamWaitEvent(st.main, landed[i], 0), "wait");
                if (!first[i])
                    cuda_ok(cudaStreamWaitEvent(st.main, copied[i], 0), "wait");
                for (int k = 0; k < NKIND; ++k)
                    lib_ok(launch(p, static_cast<Kind>(k), st.main), kKindName[k]);
                cuda_ok(cudaEventRecord(computed[i], st.main), "record");
                cuda_ok(cudaStreamWaitEvent(s_out, computed[i], 0), "wait");
                cuda_ok(cudaMemcpyAsync(p.hy, p.y, mn * 2, cudaMemcpyDeviceToHost, s_out), "d2h");
                cuda_ok(cudaMemcpyAsync(p.hdx, p.dx, mk * 2, cudaMemcpyDeviceToHost, s_out), "d2h");
                cuda_ok(cudaMemcpyAsync(p.hdw, p.dw, nk * 2, cudaMemcpyDeviceToHost, s_out), "d2h");
                cuda_ok(cudaEventRecord(copied[i], s_out), "record");
                first[i] = false;
            }
        };
        one();
        sync_and_check("e2e warm-up");
        cuda_ok(cudaEventRecord(a, st.main), "record");
        for (int i = 0; i < e2e_steps; ++i)
            one();
        for (size_t i = 0; i < np; ++i)   // the last results are on the host
            cuda_ok(cudaStreamWaitEvent(st.main, copied[i], 0), "wait");
        cuda_ok(cudaEventRecord(b, st.main), "record");
        sync_and_check("e2e");
        float ms = 0.0f;
        cuda_ok(cudaEventElapsedTime(&ms, a, b), "elapsed");
        e2e_ms = ms / e2e_steps;
        launches += (1 + e2e_steps) * static_cast<int>(projs.size()) * NKIND;
    }

    // ---- one JSON line
    std::printf("{\"harness\": \"jetfp8_bench (C++, CUDA events, C-ABI)\", \"workload\": \"%s\", "
                "\"tokens\": %lld, \"steps\": %d, \"warmup\": %d, \"streams\": %d, "
                "\"value\": %.2f, \"unit\": \"TFLOP/s\", \"ms_per_step\": %.4f, \"kernels\": {",
                wl->name, static_cast<long long>(wl->tokens), steps, warmup, streams,
                flops / (ms_step * 1e-3) / 1e12, ms_step);
    for (int k = 0; k < NKIND; ++k)
        std::printf("%s\"%s\": {\"ms_per_step\": %.4f}", k ? ", " : "", kKindName[k], kind_ms[k]);
    std::printf("}");
    if (e2e)
        std::printf(", \"e2e\": {\"value\": %.2f, \"unit\": \"TFLOP/s\", \"ms_per_step\": %.3f, "
                    "\"steps\": %d, \"h2d_bytes_per_step\": %llu, \"d2h_bytes_per_step\": %llu}",
                    flops / (e2e_ms * 1e-3) / 1e12, e2e_ms, e2e_steps, static_cast<unsigned long long>(h2d),
                    static_cast<unsigned long long>(d2h));
    std::printf(", \"gpu_launches\": %d, \"input_generation_s\": %.2f}\n", launches, gen_s);
    return 0;
}
