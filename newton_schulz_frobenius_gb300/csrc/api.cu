// Host runtime of the Muon update library: argument validation, per-device
// state, workspace, shape bucketing, the Newton-Schulz orchestration (plain and Gram
// with segment restarts), the measured-cost autotune with its persistent cache,
// and the C ABI declared in include/muon.h.
//
// Shape-adaptive execution follows the "DMuon" pages: matrices are grouped by
// shape (news page, section 3; summary, section 2.2 "batching"), each distinct
// shape is timed once per candidate scheme and the fastest is cached and reused
// (summary, sections 2.3-2.4).  Gram NS with restarts is the "MuonX" page,
// section 3.2.
#include "muon_internal.cuh"

#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <fstream>
#include <functional>
#include <map>
#include <memory>
#include <new>
#include <stdexcept>
#include <mutex>
#include <queue>
#include <sstream>
#include <string>
#include <tuple>
#include <vector>

namespace muon {

// NVTX ranges around the host steps (a step, a bucket, its prologue and NS
// run, the fused small-matrix launches): free when no tool is attached.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Device allocations of the library's own storage (workspaces, counters,
// groups) go through here.  MUON_FAIL_ALLOC=1 makes every one of them fail, so
// that the allocation-failure paths can be exercised without exhausting a GPU.
static cudaError_t dev_alloc(void** p, size_t bytes) {
    const char* f = std::getenv("MUON_FAIL_ALLOC");
    if (f && f[0] == '1') {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}


// ---------------------------------------------------------------------------
// logging and errors
// ---------------------------------------------------------------------------

static int log_level() {
    static int lvl = [] {
        const char* e = std::getenv("MUON_LOG");
        return e ? std::atoi(e) : 0;
    }();
    return lvl;
}

static thread_local std::string t_last_error;

bool pdl_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("MUON_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

static void logf(int lvl, const char* fmt, ...) {
    if (log_level() < lvl) return;
    va_list ap;
    va_start(ap, fmt);
    std::fprintf(stderr, "[muon] ");
    std::vfprintf(stderr, fmt, ap);
    std::fprintf(stderr, "\n");
    va_end(ap);
}

static int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    logf(1, "error %d: %s", status, buf);
    return status;
}

static int cuda_fail(cudaError_t e, const char* what) {
    return fail(MUON_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Host containers sized by the caller's arguments can fail to allocate; every
// entry point that builds them ends in these handlers, so that no C++
// exception crosses the C boundary.
#define MUON_CATCH_ALL                                                                        \
    catch (const std::bad_alloc&) { return fail(MUON_ENOMEM, "host allocation failed"); }      \
    catch (const std::length_error&) { return fail(MUON_ENOMEM, "host allocation too large"); } \
    catch (const std::exception& ex_) { return fail(MUON_EINVAL, "internal error: %s", ex_.what()); } \
    catch (...) { return fail(MUON_EINVAL, "internal error"); }

#define MUON_CUDA(call)                                   \
    do {                                                  \
        cudaError_t e_ = (call);                          \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

// ---------------------------------------------------------------------------
// per-device state
// ---------------------------------------------------------------------------

struct DevCtx {
    int device = -1;
    int sms = 0;
    int major = 0, minor = 0;
    std::string name;
    int* status = nullptr;     // device status word
};

static std::mutex g_mu;                 // guards every global below
static std::map<int, DevCtx> g_dev;

static int get_dev(DevCtx& out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(dev);
    if (it == g_dev.end()) {
        cudaDeviceProp p;
        e = cudaGetDeviceProperties(&p, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        DevCtx c;
        c.device = dev;
        c.sms = p.multiProcessorCount;
        c.major = p.major;
        c.minor = p.minor;
        c.name = p.name;
        if (!(c.major == 10 && c.minor == 3))
            return fail(MUON_ENOTSUP, "device %d (%s) is sm_%d%d; this library is built for sm_103a", dev,
                        p.name, c.major, c.minor);
        e = cudaMalloc(&c.status, 64);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(status)");
        e = cudaMemset(c.status, 0, 64);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
        it = g_dev.emplace(dev, c).first;
    }
    out = it->second;
    return MUON_OK;
}

// ---------------------------------------------------------------------------
// workspace: one grow-only device buffer and a pinned staging ring for the
// matrix tables, per (device, stream)
// ---------------------------------------------------------------------------

constexpr int STAGE_SLOTS = 4;

struct Workspace {
    char* base = nullptr;
    size_t bytes = 0;
    int* pcnt = nullptr;        // prep kernel's per-matrix arrival counters (zero between launches)
    int pcnt_cap = 0;
    MatEntry* h_stage[STAGE_SLOTS] = {nullptr, nullptr, nullptr, nullptr};
    cudaEvent_t ev[STAGE_SLOTS] = {nullptr, nullptr, nullptr, nullptr};
    size_t stage_cap = 0;   // entries per slot
    int slot = 0;
};

static std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static int ws_get(int dev, cudaStream_t s, size_t need, Workspace** out) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace& w = g_ws[{dev, s}];
    if (w.bytes < need) {
        if (w.base) {
            cudaError_t e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize(workspace grow)");
            cudaFree(w.base);
            w.base = nullptr;
            w.bytes = 0;
        }
        size_t want = align_up(need + need / 4, 1 << 20);
        cudaError_t e = dev_alloc(reinterpret_cast<void**>(&w.base), want);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(MUON_ENOMEM, "workspace allocation of %zu bytes failed: %s", want, cudaGetErrorString(e));
        }
        w.bytes = want;
        logf(2, "workspace grown to %zu bytes on device %d", want, dev);
    }
    *out = &w;
    return MUON_OK;
}

// At least B prep counters for stream s on device dev, zero (grown, never
// shrunk; each launch leaves them at zero again).
static int prep_counters(int dev, cudaStream_t s, int B, int** out) {
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace& w = g_ws[{dev, s}];
    if (w.pcnt_cap < B) {
        if (w.pcnt) {
            cudaError_t e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize(counters grow)");
            cudaFree(w.pcnt);
            w.pcnt = nullptr;
            w.pcnt_cap = 0;
        }
        const int cap = std::max(B, 4096);
        cudaError_t e = dev_alloc(reinterpret_cast<void**>(&w.pcnt), (size_t)cap * sizeof(int));
        if (e != cudaSuccess) {
            cudaGetLastError();
            w.pcnt = nullptr;
            return fail(MUON_ENOMEM, "prep counters: %s", cudaGetErrorString(e));
        }
        e = cudaMemsetAsync(w.pcnt, 0, (size_t)cap * sizeof(int), s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(prep counters)");
        w.pcnt_cap = cap;
    }
    *out = w.pcnt;
    return MUON_OK;
}

// Copies `n` table entries to `d_dst` on stream `s` through the pinned ring.
static int upload_table(Workspace& w, const std::vector<MatEntry>& h, MatEntry* d_dst, cudaStream_t s) {
    if (h.empty()) return MUON_OK;
    std::lock_guard<std::mutex> lk(g_mu);
    if (w.stage_cap < h.size()) {
        for (int i = 0; i < STAGE_SLOTS; ++i) {
            if (w.ev[i]) cudaEventSynchronize(w.ev[i]);
            if (w.h_stage[i]) cudaFreeHost(w.h_stage[i]);
            w.h_stage[i] = nullptr;
        }
        size_t cap = std::max<size_t>(h.size(), 256);
        for (int i = 0; i < STAGE_SLOTS; ++i) {
            cudaError_t e = cudaMallocHost(reinterpret_cast<void**>(&w.h_stage[i]), cap * sizeof(MatEntry));
            if (e != cudaSuccess) return fail(MUON_ENOMEM, "pinned staging allocation failed");
            if (!w.ev[i]) {
                e = cudaEventCreateWithFlags(&w.ev[i], cudaEventDisableTiming);
                if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
            }
        }
        w.stage_cap = cap;
    }
    const int slot = w.slot;
    w.slot = (w.slot + 1) % STAGE_SLOTS;
    cudaError_t e = cudaEventSynchronize(w.ev[slot]);   // the copy made from this slot before has run
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize(stage)");
    std::memcpy(w.h_stage[slot], h.data(), h.size() * sizeof(MatEntry));
    e = cudaMemcpyAsync(d_dst, w.h_stage[slot], h.size() * sizeof(MatEntry), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(table)");
    e = cudaEventRecord(w.ev[slot], s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(stage)");
    return MUON_OK;
}

// ---------------------------------------------------------------------------
// launch accounting and optional per-launch event timing
// ---------------------------------------------------------------------------

static std::atomic<int64_t> g_launches{0};
static std::atomic<int> g_timing{0};

struct TimedLaunch {
    int kclass;
    cudaEvent_t a, b;
    double work;
};
static std::vector<TimedLaunch> g_timed;
static std::vector<cudaEvent_t> g_event_pool;
static thread_local int t_open = -1;   // index of the launch being recorded

static const char* kclass_name(int k) {
    static const char* names[KC_COUNT] = {"prep_momentum_norm", "norm_finalize", "gemm_tc_syrk",
                                          "gemm_tc_square", "gemm_tc_apply", "gemm_tc_apply_update",
                                          "gemm_fp32", "other", "small_ns_fused", "adamw", "pack"};
    return (k >= 0 && k < KC_COUNT) ? names[k] : "other";
}

static cudaEvent_t pool_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

void note_launch_begin(int kclass, cudaStream_t s) {
    g_launches.fetch_add(1);
    if (!g_timing.load()) return;
    std::lock_guard<std::mutex> lk(g_mu);
    TimedLaunch t{kclass, pool_event(), pool_event(), 0.0};
    cudaEventRecord(t.a, s);
    g_timed.push_back(t);
    t_open = (int)g_timed.size() - 1;
}

void note_launch_end(int kclass, double work, cudaStream_t s) {
    (void)kclass;
    if (!g_timing.load() || t_open < 0) return;
    std::lock_guard<std::mutex> lk(g_mu);
    if (t_open < (int)g_timed.size()) {
        cudaEventRecord(g_timed[t_open].b, s);
        g_timed[t_open].work = work;
    }
    t_open = -1;
}

// One-shot stall of the bounded-wait test hook: kind and stage + 1 packed in
// one word so that arming and taking are single atomic operations.
static std::atomic<int> g_stall{0};

int take_stall(int kind) {
    int v = g_stall.load();
    while (v != 0 && (v & 0xFF) == kind) {
        if (g_stall.compare_exchange_weak(v, 0)) return v >> 8;
    }
    return 0;
}

}  // namespace muon

namespace muon {

// ---------------------------------------------------------------------------
// NS configuration
// ---------------------------------------------------------------------------

struct NsConfig {
    float coeffs[3] = {3.4445f, -4.7750f, 2.0315f};
    int steps = 5;
    std::vector<int> segments{2, 2, 1};
    int path = MUON_PATH_AUTO;
    int ns_precision = -1;      // 16-bit parameters: -1 follow them, or MUON_BF16 / MUON_F16
};
static NsConfig g_cfg;
static std::atomic<uint64_t> g_cfg_version{1};   // bumped when plans may change (config, tune cache)

static int validate_segments(int steps, const int* segs, int nseg) {
    if (steps < 1 || steps > 64) return fail(MUON_EINVAL, "steps must be in [1, 64], got %d", steps);
    if (nseg < 0 || (nseg > 0 && !segs)) return fail(MUON_EINVAL, "bad segment list");
    if (nseg == 0) return MUON_OK;
    int sum = 0;
    for (int i = 0; i < nseg; ++i) {
        if (segs[i] < 1) return fail(MUON_EINVAL, "segment %d has length %d < 1", i, segs[i]);
        if (segs[i] > steps) return fail(MUON_EINVAL, "segment %d longer than steps (%d)", i, steps);
        sum += segs[i];
        if (sum > steps) break;                   // reported below; keeps the sum in range
    }
    if (sum != steps) return fail(MUON_EINVAL, "segments sum to %d, steps is %d", sum, steps);
    return MUON_OK;
}

// A resolved NS plan: the segment lengths actually run.  The plain path is
// the Gram orchestration with unit segments (per step: XX^T, P = aI + bA + cA^2,
// X <- P X), which performs the plain algorithm's products one for one.
struct NsPlan {
    float a, b, c;
    std::vector<int> segs;
    int path;       // MUON_PATH_PLAIN or MUON_PATH_GRAM
    int tile_n;     // tensor-core N extent of the long products
    int sym_tile_n; // tensor-core N extent of the symmetric products (128 or 256)
    int sym_dense;  // compute all tiles of the symmetric products (no mirroring)
    int gram_tf32;  // bf16 path: Gram-space matrices kept in TF32 (else bf16)
    int fused;      // run the whole update of each matrix in one CTA (small_ns.cu)
};

// Precision of the bf16 path's m x m Gram-space matrices (G, P, PG, Q).
// A bit-faithful CPU simulation of the iteration against the exact one gives,
// for the Gram path with bf16 Gram space, 0.8-1.2% relative error on every
// shape with m >= 128 and n >= 2m, but 1.5-4% on square and near-square shapes
// and 2.3% for m = 37; with TF32 Gram space all of them stay at or below 1.5%.
// The plain path's error is set by the bf16 X (0.8-1.9% either way), so it
// keeps bf16.  TF32 costs twice the operand bytes and half the tensor rate on
// the m^3 products, so it is used only where bf16 is not accurate enough.
static int gram_space_tf32(int path, int m, int n) {
    return (path == MUON_PATH_GRAM && (m < 128 || n < 2 * m)) ? 1 : 0;
}

static NsPlan make_plan(const float coeffs[3], int steps, const std::vector<int>& gram_segs, int path, int tile_n,
                        int m, int n, int sym_tile_n = 128, int sym_dense = 0) {
    NsPlan p;
    p.sym_tile_n = sym_tile_n;
    p.sym_dense = sym_dense;
    p.gram_tf32 = gram_space_tf32(path, m, n);
    p.fused = 0;
    p.a = coeffs[0];
    p.b = coeffs[1];
    p.c = coeffs[2];
    p.path = path;
    p.tile_n = tile_n;
    if (path == MUON_PATH_GRAM && !gram_segs.empty()) p.segs = gram_segs;
    else p.segs.assign(steps, 1);
    return p;
}

// ---------------------------------------------------------------------------
// products
// ---------------------------------------------------------------------------

static bool env_flag(const char* name, bool dflt);

static GemmArgs gemm_base(int dtype, int* status) {
    GemmArgs a;
    std::memset(&a, 0, sizeof a);
    a.dtype = dtype;
    a.c_dtype = is_half(dtype) ? dtype : MUON_F32;
    a.alpha = 1.0f;
    a.tile_n = 256;
    // 2-SM products for 128 x 256 tiles: measured 3-11% faster than single-SM
    // tiles on every product of the 2560x9728 and 4096x14336 paths (never
    // slower); MUON_PAIR=0 turns them off
    if (const char* f = std::getenv("MUON_PAIR")) a.pair = (f[0] == '1') ? 1 : 0;
    else a.pair = -1;
    a.status = status;
    a.b_kmajor = 1;
    return a;
}

static int run_gemm(const DevCtx& dc, cudaStream_t s, const GemmArgs& a, int kclass) {
    const double mnk = (double)a.M * a.N * a.K * a.batch;
    const double work = a.symmetric ? mnk : 2.0 * mnk;
    const bool tc = (is_half(a.dtype) || a.dtype == DT_TF32);
    const int kc = tc ? kclass : KC_SIMT;
    GemmArgs ga = a;
    if (tc) ga.stall = take_stall(STALL_PRODUCT);
    note_launch_begin(kc, s);
    cudaError_t e = tc ? launch_gemm_tc(ga, dc.sms, s) : launch_gemm_simt(a, s);
    note_launch_end(kc, work, s);
    if (e != cudaSuccess) return cuda_fail(e, "product launch");
    return MUON_OK;
}

static size_t esize(int dtype) { return is_half(dtype) ? 2 : 4; }

// Working precision of NS for parameters of this storage type: fp32 stays
// fp32; 16-bit parameters use the configured 16-bit type, by default their own.
static int ns_dtype(int param_dtype, const NsConfig& cfg) {
    if (!is_half(param_dtype)) return MUON_F32;
    return cfg.ns_precision < 0 ? param_dtype : cfg.ns_precision;
}

// Whether X holds the unscaled U (the 1 / ||U|| scale folded into the first
// products) or U already divided by its norm (the fp16 path).
static bool x_holds_u(int x_dtype) { return x_dtype != MUON_F16; }
static int64_t pad8(int64_t x) { return (x + 7) / 8 * 8; }

// Workspace of one chunk of B matrices of oriented shape m x n.
struct ChunkLayout {
    int64_t ldx, ldm;
    size_t x_bytes, m_bytes;            // one matrix
    size_t off_X, off_X2, off_G, off_S[3], off_inv, off_part, total;
    int nparts;
};

// X is stored in the path's dtype; the m x m Gram-space matrices are fp32 on
// both paths (TF32-rounded on the bf16 path).
static ChunkLayout chunk_layout(int m, int n, int B, int dtype) {
    ChunkLayout L;
    const size_t es = esize(dtype);
    L.ldx = pad8(n);
    L.ldm = pad8(m);
    L.x_bytes = (size_t)m * L.ldx * es;
    L.m_bytes = (size_t)m * L.ldm * 4;
    L.nparts = prep_num_parts(m, n);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.off_X = take(L.x_bytes * B);
    L.off_X2 = take(L.x_bytes * B);
    L.off_G = take(L.m_bytes * B);
    for (int i = 0; i < 3; ++i) L.off_S[i] = take(L.m_bytes * B);
    L.off_inv = take(sizeof(float) * B);
    L.off_part = take(sizeof(float) * (size_t)L.nparts * B);
    L.total = o;
    return L;
}

// Final epilogue of an NS run.
struct FinalEpi {
    int kind;               // EPI_UPDATE, EPI_OUT or EPI_STORE (autotune: into the workspace)
    const MatEntry* mats;   // device table (UPDATE / OUT)
    int out_dtype;
    float lr, wd, scale;
    const float* hyper = nullptr;   // device {lr, beta, wd, nesterov} read at run time, if set
};

// Runs NS on B oriented m x n matrices held (unnormalised when use_inv) in
// the chunk's X buffer, ending in `fin`.
//
// Precision of the bf16 path: X and the long products XX^T, QX are bf16 with
// fp32 accumulation; the m x m Gram-space matrices G, P, PG, Q are bf16, or,
// where gram_space_tf32() asks for it, TF32-rounded fp32 multiplied on the
// TF32 tensor path, with the transform applied to X rounded to bf16.
static int run_ns(const DevCtx& dc, cudaStream_t s, char* base, const ChunkLayout& L, int m, int n, int B,
                  int dtype, const NsPlan& plan, bool use_inv, const FinalEpi& fin) {
    char nvname[64];
    std::snprintf(nvname, sizeof nvname, "ns %dx%d x%d", m, n, B);
    NvtxRange nvr(nvname);
    char* X = base + L.off_X;
    char* Xn = base + L.off_X2;
    char* G = base + L.off_G;
    char* S[3] = {base + L.off_S[0], base + L.off_S[1], base + L.off_S[2]};
    const float* inv = reinterpret_cast<const float*>(base + L.off_inv);
    const int64_t strideX = (int64_t)m * L.ldx;
    const int64_t strideM = (int64_t)m * L.ldm;

    const bool tf = (dtype == MUON_BF16) && plan.gram_tf32;
    // Gram-space operands: fp16 on the fp16 path (ten mantissa bits, like
    // TF32), bf16 or TF32 on the bf16 path, fp32 on the FFMA path
    const int sq_dtype = is_half(dtype) ? (tf ? DT_TF32 : dtype) : MUON_F32;
    auto gram_out = [&](GemmArgs& g, bool feeds_apply) {
        // TF32 Gram space: TF32-rounded fp32, or bf16 when it is the
        // transform the long apply consumes; otherwise the path's own dtype
        if (!tf) return;
        if (feeds_apply) { g.c_dtype = MUON_BF16; g.round_tf32 = 0; }
        else { g.c_dtype = MUON_F32; g.round_tf32 = 1; }
    };
    auto sym = [&](const void* A, const void* Bm, void* C, bool feeds_apply) {
        GemmArgs g = gemm_base(sq_dtype, dc.status);
        g.A = A; g.lda = L.ldm; g.strideA = strideM;
        g.B = Bm; g.ldb = L.ldm; g.strideB = strideM;
        g.M = m; g.N = m; g.K = m; g.batch = B;
        g.symmetric = plan.sym_dense ? 0 : 1;
        g.epi = EPI_STORE;
        g.C = C; g.ldc = L.ldm; g.strideC = strideM;
        g.tile_n = plan.sym_tile_n;
        gram_out(g, feeds_apply);
        return g;
    };

    const int nseg = (int)plan.segs.size();
    for (int si = 0; si < nseg; ++si) {
        const int Lseg = plan.segs[si];
        const bool first = (si == 0);
        const bool last = (si == nseg - 1);

        // G = X X^T  (lower triangle, mirrored); first segment folds 1/||U||^2
        {
            GemmArgs g = gemm_base(dtype, dc.status);
            g.A = X; g.lda = L.ldx; g.strideA = strideX;
            g.B = X; g.ldb = L.ldx; g.strideB = strideX;
            g.M = m; g.N = m; g.K = n; g.batch = B;
            g.symmetric = plan.sym_dense ? 0 : 1;
            g.epi = EPI_STORE;
            g.C = G; g.ldc = L.ldm; g.strideC = strideM;
            g.tile_n = plan.sym_tile_n;
            gram_out(g, false);
            if (first && use_inv) { g.alpha_vec = inv; g.alpha_sq = 1; }
            int r = run_gemm(dc, s, g, KC_SYRK);
            if (r) return r;
        }

        bool used[3] = {false, false, false};
        auto grab = [&]() {
            for (int i = 0; i < 3; ++i)
                if (!used[i]) { used[i] = true; return i; }
            return -1;
        };
        int q = -1;
        for (int j = 1; j <= Lseg; ++j) {
            // P = aI + bG + cG^2, fused into the G^2 product
            const int p = grab();
            {
                GemmArgs g = sym(G, G, S[p], Lseg == 1);
                g.epi = EPI_POLY;
                g.Gin = G; g.ldg = L.ldm; g.strideG = strideM;
                g.pa = plan.a; g.pb = plan.b; g.pc = plan.c;
                int r = run_gemm(dc, s, g, KC_SQUARE);
                if (r) return r;
            }
            if (j == 1) {
                q = p;
            } else {
                const int qn = grab();     // Q <- P Q
                int r = run_gemm(dc, s, sym(S[p], S[q], S[qn], j == Lseg), KC_SQUARE);
                if (r) return r;
                used[q] = false;
                q = qn;
            }
            if (j < Lseg) {
                const int t = grab();      // G <- (P G) P
                int r = run_gemm(dc, s, sym(S[p], G, S[t], false), KC_SQUARE);
                if (r) return r;
                r = run_gemm(dc, s, sym(S[t], S[p], G, false), KC_SQUARE);
                if (r) return r;
                used[t] = false;
            }
            if (p != q) used[p] = false;
        }

        // X <- Q X: B operand is X itself, read MN-major
        GemmArgs g = gemm_base(dtype, dc.status);
        g.A = S[q]; g.lda = L.ldm; g.strideA = strideM;
        g.B = X; g.ldb = L.ldx; g.strideB = strideX; g.b_kmajor = 0;
        g.M = m; g.N = n; g.K = m; g.batch = B;
        g.tile_n = plan.tile_n;
        if (first && use_inv) { g.alpha_vec = inv; g.alpha_sq = 0; }
        int kc = KC_APPLY;
        if (!last || fin.kind == EPI_STORE) {
            g.epi = EPI_STORE;
            g.C = Xn; g.ldc = L.ldx; g.strideC = strideX;
        } else {
            g.epi = fin.kind;
            g.mats = fin.mats;
            g.out_dtype = fin.out_dtype;
            g.lr = fin.lr; g.wd = fin.wd; g.scale = fin.scale;
            g.hyper = fin.hyper;
            if (fin.kind == EPI_UPDATE) kc = KC_APPLY_UPDATE;
        }
        int r = run_gemm(dc, s, g, kc);
        if (r) return r;
        std::swap(X, Xn);
    }
    return MUON_OK;
}

static int run_prep(const DevCtx& dc, cudaStream_t s, char* base, const ChunkLayout& L, int m, int n, int B,
                    const MatEntry* d_mats, int in_dtype, int mom_dtype, int x_dtype, bool with_mom, int nesterov,
                    float beta, bool vec_ok, int* cnt, const float* hyper = nullptr) {
    char nvname[64];
    std::snprintf(nvname, sizeof nvname, "prep %dx%d x%d", m, n, B);
    NvtxRange nvr(nvname);
    PrepArgs p;
    std::memset(&p, 0, sizeof p);
    p.mats = d_mats;
    p.m = m; p.n = n; p.batch = B;
    p.in_dtype = in_dtype; p.mom_dtype = mom_dtype; p.x_dtype = x_dtype;
    p.with_momentum = with_mom ? 1 : 0;
    p.nesterov = nesterov;
    p.beta = beta;
    p.X = base + L.off_X; p.ldx = L.ldx; p.strideX = (int64_t)m * L.ldx;
    p.partials = reinterpret_cast<float*>(base + L.off_part);
    p.nparts = prep_grid_parts(m, n, B);       // CTAs per matrix, one partial each (<= L.nparts)
    p.vec_ok = vec_ok ? 1 : 0;
    p.hyper = hyper;
    p.write_x = 1;
    p.write_mom = 1;
    const double elems = (double)m * n * B;
    const double in_bytes = elems * (esize(in_dtype) + (with_mom ? esize(mom_dtype) : 0.0));
    const double bytes = in_bytes + elems * ((with_mom ? esize(mom_dtype) : 0.0) + esize(x_dtype));
    float* inv = reinterpret_cast<float*>(base + L.off_inv);
    const bool two_pass = !x_holds_u(x_dtype);
    // the (first) prep launch finalises the norm itself: its last CTA per
    // matrix writes inv (cnt: zero per-matrix counters, left at zero)
    PrepArgs pf = p;
    pf.counter = cnt;
    pf.inv = inv;
    pf.eps = 1e-7f;
    pf.status = dc.status;
    if (two_pass) {
        // fp16 X: sums of U^2 first (nothing written), then momentum and U / ||U||
        PrepArgs p1 = pf;
        p1.write_x = 0;
        p1.write_mom = 0;
        note_launch_begin(KC_PREP, s);
        cudaError_t e = launch_prep(p1, s);
        note_launch_end(KC_PREP, in_bytes, s);
        if (e != cudaSuccess) return cuda_fail(e, "prep launch");
        p.x_scale = inv;
    }
    note_launch_begin(KC_PREP, s);
    cudaError_t e = launch_prep(two_pass ? p : pf, s);
    note_launch_end(KC_PREP, bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "prep launch");
    return MUON_OK;
}

}  // namespace muon

namespace muon {

// ---------------------------------------------------------------------------
// measured-cost autotune and its cache
// ---------------------------------------------------------------------------

struct TuneEntry {
    int path;
    int tile_n;
    double ms_per_matrix;
    int fused;
    int sym_tile_n;
    int sym_dense;
};
using TuneKey = std::tuple<std::string, int, int, int64_t, int64_t, int>;   // device, sms, cudart, m, n, dtype
static std::map<TuneKey, TuneEntry> g_tune;
static std::map<std::tuple<int64_t, int64_t, int>, int> g_last_path;     // oriented m, n, dtype -> path

static int cudart_version() {
    int v = 0;
    cudaRuntimeGetVersion(&v);
    return v;
}

static TuneKey tune_key(const DevCtx& dc, int64_t m, int64_t n, int dtype) {
    return TuneKey{dc.name, dc.sms, cudart_version(), m, n, dtype};
}

static bool env_flag(const char* name, bool dflt) {
    const char* e = std::getenv(name);
    if (!e || !*e) return dflt;
    return !(e[0] == '0' || e[0] == 'n' || e[0] == 'N' || e[0] == 'f' || e[0] == 'F');
}

static int save_tune_file(const char* path);

// Whether the one-CTA-per-matrix kernel can run this plan (bf16, m <= 128,
// n <= 512, segments of length <= 2, bf16 Gram space).  MUON_SMALL=0 turns it off.
static bool small_eligible(const NsPlan& p, int m, int n, int dtype) {
    if (dtype != MUON_BF16 || p.gram_tf32 || !env_flag("MUON_SMALL", true)) return false;   // bf16 NS only
    return small_ns_fits(m, n, (int)p.segs.size(), p.segs.data());
}

__global__ void table_fill_kernel(MatEntry* t, char* base, int64_t stride_bytes, int trans, int batch) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < batch) {
        char* p = base + (int64_t)b * stride_bytes;
        t[b] = MatEntry{p, nullptr, p, trans, 0};
    }
}

static SmallBucket small_bucket(const NsPlan& p, const MatEntry* mats, int B, int m, int n, bool vec_ok) {
    SmallBucket bk;
    std::memset(&bk, 0, sizeof bk);
    bk.mats = mats;
    bk.batch = B; bk.m = m; bk.n = n;
    bk.nseg = std::min((int)p.segs.size(), 8);
    for (int i = 0; i < bk.nseg; ++i) bk.segs[i] = p.segs[i];
    bk.vec_ok = vec_ok ? 1 : 0;
    bk.scale = 0.2f * std::sqrt((float)n);
    return bk;
}

// Arguments of a fused launch over one bucket, CTA c taking matrices c, c + grid, ...
static SmallArgs small_args(const NsPlan& p, const MatEntry* mats, int B, int m, int n, int mode, int param_dtype,
                            int mom_dtype, int nesterov, float beta, float lr, float wd, bool vec_ok, int* status) {
    SmallArgs a;
    std::memset(&a, 0, sizeof a);
    a.nb = 1;
    a.bk[0] = small_bucket(p, mats, B, m, n, vec_ok);
    a.mode = mode;
    a.param_dtype = param_dtype; a.mom_dtype = mom_dtype;
    a.nesterov = nesterov;
    a.beta = beta; a.lr = lr; a.wd = wd;
    a.a = p.a; a.b = p.b; a.c = p.c;
    a.status = status;
    return a;
}

// Work lists of one fused launch over several buckets: every matrix is an
// item of its bucket's cost; items go, most expensive first, to the CTA with
// the least work so far (longest processing time first), which balances
// buckets whose matrix counts are not multiples of the SM count.  Output:
// grid, per-CTA offsets ptr[grid + 1] and items (bucket << 24 | index).
struct SmallWork {
    int grid = 0;
    std::vector<int> ptr, items;
};
static SmallWork small_work(const std::vector<int>& counts, const std::vector<double>& costs, int sms) {
    SmallWork w;
    std::vector<std::pair<double, int>> order;          // (cost, item)
    for (size_t bi = 0; bi < counts.size(); ++bi)
        for (int i = 0; i < counts[bi]; ++i) order.push_back({costs[bi], (int)(bi << 24) | i});
    std::stable_sort(order.begin(), order.end(), [](const auto& x, const auto& y) { return x.first > y.first; });
    const int total = (int)order.size();
    w.grid = std::max(1, std::min(total, sms));
    std::vector<std::vector<int>> lists((size_t)w.grid);
    std::priority_queue<std::pair<double, int>, std::vector<std::pair<double, int>>, std::greater<>> heap;
    for (int c = 0; c < w.grid; ++c) heap.push({0.0, c});
    std::vector<double> load((size_t)w.grid, 0.0);
    std::vector<std::vector<double>> lcost((size_t)w.grid);
    for (const auto& it : order) {
        auto top = heap.top();
        heap.pop();
        lists[(size_t)top.second].push_back(it.second);
        lcost[(size_t)top.second].push_back(it.first);
        load[(size_t)top.second] = top.first + it.first;
        heap.push({top.first + it.first, top.second});
    }
    // Improve the makespan: move one item out of the most loaded CTA, or swap
    // it for a cheaper one of another CTA, while that lowers the maximum of
    // the two loads below the current makespan (a few sweeps; LPT leaves the
    // last CTAs one item over when the items are few and coarse).
    const int sweeps = total <= 8 * w.grid ? 4 * w.grid : 0;   // fine-grained lists are near the bound already
    for (int sweep = 0; sweep < sweeps; ++sweep) {
        const size_t cm = (size_t)(std::max_element(load.begin(), load.end()) - load.begin());
        const double top = load[cm];
        double best = top;
        size_t bi = 0, bc = 0, bj = 0;
        bool bswap = false;
        for (size_t i = 0; i < lists[cm].size(); ++i) {
            const double ci = lcost[cm][i];
            for (size_t c = 0; c < (size_t)w.grid; ++c) {
                if (c == cm) continue;
                const double mv = std::max(top - ci, load[c] + ci);
                if (mv < best - 1e-12) { best = mv; bi = i; bc = c; bswap = false; }
                for (size_t j = 0; j < lists[c].size(); ++j) {
                    const double cj = lcost[c][j];
                    if (cj >= ci) continue;
                    const double sw = std::max(top - ci + cj, load[c] - cj + ci);
                    if (sw < best - 1e-12) { best = sw; bi = i; bc = c; bj = j; bswap = true; }
                }
            }
        }
        if (best >= top - 1e-12) break;
        const int item = lists[cm][bi];
        const double ci = lcost[cm][bi];
        lists[cm].erase(lists[cm].begin() + (long)bi);
        lcost[cm].erase(lcost[cm].begin() + (long)bi);
        load[cm] -= ci;
        if (bswap) {
            const int other = lists[bc][bj];
            const double cj = lcost[bc][bj];
            lists[bc][bj] = item;
            lcost[bc][bj] = ci;
            load[bc] += ci - cj;
            lists[cm].push_back(other);
            lcost[cm].push_back(cj);
            load[cm] += cj;
        } else {
            lists[bc].push_back(item);
            lcost[bc].push_back(ci);
            load[bc] += ci;
        }
    }
    // within a CTA, the costliest items first (the next one's inputs are
    // prefetched while the current one runs)
    for (int c = 0; c < w.grid; ++c) {
        std::vector<size_t> idx(lists[(size_t)c].size());
        for (size_t i = 0; i < idx.size(); ++i) idx[i] = i;
        std::stable_sort(idx.begin(), idx.end(),
                         [&](size_t x, size_t y) { return lcost[(size_t)c][x] > lcost[(size_t)c][y]; });
        std::vector<int> l2;
        for (size_t i : idx) l2.push_back(lists[(size_t)c][i]);
        lists[(size_t)c] = l2;
    }
    w.ptr.assign((size_t)w.grid + 1, 0);
    for (int c = 0; c < w.grid; ++c) {
        w.ptr[(size_t)c + 1] = w.ptr[(size_t)c] + (int)lists[(size_t)c].size();
        w.items.insert(w.items.end(), lists[(size_t)c].begin(), lists[(size_t)c].end());
    }
    return w;
}

// Algorithmic FLOPs of one NS update under this plan (symmetric results half).
static double plan_alg_flops(const NsPlan& p, int m, int n) {
    const double M = m, N = n;
    double f = 0.0;
    for (int L : p.segs) {
        f += M * M * N;                 // X X^T
        f += L * M * M * M;             // one G^2 per iteration
        f += (L - 1) * 3.0 * M * M * M; // P Q, P G and (P G) P for every further iteration
        f += 2.0 * M * M * N;           // Q X
    }
    return f;
}

static int run_small(const DevCtx& dc, cudaStream_t s, const SmallArgs& a, double alg_flops) {
    NvtxRange nvr("fused small-matrix launch");
    SmallArgs sa = a;
    sa.stall = take_stall(STALL_SMALL);
    note_launch_begin(KC_SMALL, s);
    cudaError_t e = launch_small_ns(sa, dc.sms, s);
    note_launch_end(KC_SMALL, alg_flops, s);
    if (e != cudaSuccess) return cuda_fail(e, "fused small-matrix launch");
    return MUON_OK;
}

// Fused launches of one step: the fused buckets in groups of at most
// SMALL_MAX_BUCKETS, each group one launch with LPT work lists.  Costs per
// matrix: the autotune's measured time of the fused kernel when every bucket
// of the group has one, else a model (FLOPs at 12 TFLOP/s and 10 bytes per
// element at 40 GB/s per SM; only the ratios matter).
struct FusedLaunch {
    std::vector<int> bks;       // bucket indices (into the caller's key order)
    SmallWork work;
    size_t off = 0;             // byte offset of ptr, items in the work block
    size_t bytes = 0;
};
static std::vector<FusedLaunch> plan_fused(const DevCtx& dc, const std::vector<NsPlan>& plans,
                                           const std::vector<std::pair<int, int>>& keys,
                                           const std::vector<int64_t>& counts, int nsd, size_t* total_bytes) {
    std::vector<FusedLaunch> out;
    FusedLaunch cur;
    for (size_t k = 0; k < keys.size(); ++k) {
        if (!plans[k].fused) continue;
        cur.bks.push_back((int)k);
        if ((int)cur.bks.size() == SMALL_MAX_BUCKETS) {
            out.push_back(cur);
            cur = FusedLaunch{};
        }
    }
    if (!cur.bks.empty()) out.push_back(cur);
    size_t off = 0;
    for (auto& fl : out) {
        std::vector<int> cnt;
        std::vector<double> measured, model;
        bool all_measured = true;
        for (int k : fl.bks) {
            const int m = keys[(size_t)k].first, n = keys[(size_t)k].second;
            cnt.push_back((int)counts[(size_t)k]);
            model.push_back(plan_alg_flops(plans[(size_t)k], m, n) / 12e12 + (double)m * n * 10.0 / 40e9);
            double ms = -1.0;
            {
                std::lock_guard<std::mutex> lk(g_mu);
                auto it = g_tune.find(tune_key(dc, m, n, nsd));
                if (it != g_tune.end() && it->second.fused) ms = it->second.ms_per_matrix;
            }
            measured.push_back(ms);
            all_measured = all_measured && ms > 0.0;
        }
        fl.work = small_work(cnt, all_measured ? measured : model, dc.sms);
        fl.off = off;
        fl.bytes = align_up(sizeof(int) * (fl.work.ptr.size() + fl.work.items.size()), 256);
        off += fl.bytes;
    }
    *total_bytes = off;
    return out;
}

// Copies the work lists of `fl` into a host byte block at fl.off.
static void pack_fused(const std::vector<FusedLaunch>& fl, char* block) {
    for (const auto& f : fl) {
        int* p = reinterpret_cast<int*>(block + f.off);
        std::memcpy(p, f.work.ptr.data(), sizeof(int) * f.work.ptr.size());
        std::memcpy(p + f.work.ptr.size(), f.work.items.data(), sizeof(int) * f.work.items.size());
    }
}

// Arguments of fused launch `f`; mats_of(k) gives bucket k's device table.
template <typename MatsOf>
static SmallArgs fused_args(const FusedLaunch& f, const char* d_block, const std::vector<NsPlan>& plans,
                            const std::vector<std::pair<int, int>>& keys, const std::vector<int64_t>& counts,
                            const std::vector<char>& vec_ok, MatsOf mats_of, int mode, int param_dtype,
                            int mom_dtype, int nesterov, float beta, float lr, float wd, int* status,
                            const float* hyper) {
    SmallArgs a;
    std::memset(&a, 0, sizeof a);
    a.nb = (int)f.bks.size();
    for (int j = 0; j < a.nb; ++j) {
        const int k = f.bks[(size_t)j];
        a.bk[j] = small_bucket(plans[(size_t)k], mats_of(k), (int)counts[(size_t)k], keys[(size_t)k].first,
                               keys[(size_t)k].second, vec_ok[(size_t)k] != 0);
    }
    const int* p = reinterpret_cast<const int*>(d_block + f.off);
    a.cta_ptr = p;
    a.items = p + f.work.ptr.size();
    a.grid = f.work.grid;
    a.mode = mode;
    a.param_dtype = param_dtype; a.mom_dtype = mom_dtype;
    a.nesterov = nesterov;
    a.beta = beta; a.lr = lr; a.wd = wd;
    const NsPlan& p0 = plans[(size_t)f.bks[0]];
    a.a = p0.a; a.b = p0.b; a.c = p0.c;
    a.status = status;
    a.hyper = hyper;
    return a;
}

static double fused_flops(const FusedLaunch& f, const std::vector<NsPlan>& plans,
                          const std::vector<std::pair<int, int>>& keys, const std::vector<int64_t>& counts) {
    double t = 0.0;
    for (int k : f.bks)
        t += plan_alg_flops(plans[(size_t)k], keys[(size_t)k].first, keys[(size_t)k].second) * (double)counts[(size_t)k];
    return t;
}

static int autotune_shape(const DevCtx& dc, cudaStream_t s, int m, int n, int dtype, int B, const NsConfig& cfg,
                          TuneEntry* out) {
    const ChunkLayout L = chunk_layout(m, n, B, dtype);
    const size_t table_off = align_up(L.total, 256);
    Workspace* w = nullptr;
    int r = ws_get(dc.device, s, table_off + align_up(sizeof(MatEntry) * (size_t)B, 256), &w);
    if (r) return r;
    char* base = w->base;

    cudaEvent_t e0, e1;
    MUON_CUDA(cudaEventCreate(&e0));
    MUON_CUDA(cudaEventCreate(&e1));
    FinalEpi fin{EPI_STORE, nullptr, dtype, 0.f, 0.f, 0.f};
    const float scale = std::sqrt(3.0f / ((float)m * (float)n));
    struct Cand { int path, tile_n, sym_tile_n, sym_dense; };
    const bool bf = is_half(dtype);
    TuneEntry best{MUON_PATH_PLAIN, 256, 1e300, 0, 128, 0};
    const int reps = 3;
    auto measure = [&](const Cand& c, double* out_ms) -> int {
        NsPlan plan = make_plan(cfg.coeffs, cfg.steps, cfg.segments, c.path, c.tile_n, m, n, c.sym_tile_n,
                                c.sym_dense);
        std::vector<float> times;
        for (int rep = 0; rep <= reps; ++rep) {
            cudaError_t e = launch_fill_synthetic(base + L.off_X, (int64_t)B * m * L.ldx, dtype, scale,
                                                  0x5eed0000u + (uint32_t)rep, s);
            if (e != cudaSuccess) return cuda_fail(e, "fill launch");
            MUON_CUDA(cudaEventRecord(e0, s));
            int rr = run_ns(dc, s, base, L, m, n, B, dtype, plan, false, fin);
            if (rr) return rr;
            MUON_CUDA(cudaEventRecord(e1, s));
            MUON_CUDA(cudaEventSynchronize(e1));
            float ms = 0.f;
            MUON_CUDA(cudaEventElapsedTime(&ms, e0, e1));
            if (rep > 0) times.push_back(ms);   // rep 0 is the warm-up
        }
        std::sort(times.begin(), times.end());
        *out_ms = times[times.size() / 2] / B;
        logf(2, "autotune %dx%d dtype %d path %d tile %d sym %d%s: %.4f ms/matrix", m, n, dtype, c.path, c.tile_n,
             c.sym_tile_n, c.sym_dense ? " dense" : "", *out_ms);
        if (*out_ms < best.ms_per_matrix) best = TuneEntry{c.path, c.tile_n, *out_ms, 0, c.sym_tile_n, c.sym_dense};
        return MUON_OK;
    };
    // stage 1: path x long-product tile, symmetric products as 128-wide lower-triangle tiles
    for (int tile : {256, 128}) {
        if (!bf && tile == 128) continue;
        for (int path : {MUON_PATH_PLAIN, MUON_PATH_GRAM}) {
            if (path == MUON_PATH_GRAM && cfg.segments.empty()) continue;
            double ms;
            if ((r = measure(Cand{path, tile, 128, 0}, &ms))) return r;
        }
    }
    // stage 2: the symmetric products' tile and form for the winning path and tile
    const int bp = best.path, bt = best.tile_n;
    for (const Cand& c : {Cand{bp, bt, 256, 0}, Cand{bp, bt, 128, 1}, Cand{bp, bt, 256, 1}}) {
        if (!bf && c.sym_tile_n == 256) continue;
        double ms;
        if ((r = measure(c, &ms))) return r;
    }
    // the one-CTA-per-matrix kernel, on B synthetic matrices stored contiguously
    for (int path : {MUON_PATH_PLAIN, MUON_PATH_GRAM}) {
        if (path == MUON_PATH_GRAM && cfg.segments.empty()) continue;
        NsPlan plan = make_plan(cfg.coeffs, cfg.steps, cfg.segments, path, 256, m, n);
        if (!small_eligible(plan, m, n, dtype)) continue;
        MatEntry* table = reinterpret_cast<MatEntry*>(base + table_off);
        char* mats = base + L.off_X2;
        table_fill_kernel<<<(B + 127) / 128, 128, 0, s>>>(table, mats, (int64_t)m * n * 2, 0, B);
        MUON_CUDA(cudaGetLastError());
        const SmallArgs sa = small_args(plan, table, B, m, n, 1, MUON_BF16, MUON_BF16, 0, 0.f, 0.f, 0.f,
                                        (m % 8 == 0) && (n % 8 == 0), dc.status);
        std::vector<float> times;
        for (int rep = 0; rep <= reps; ++rep) {
            cudaError_t e = launch_fill_synthetic(mats, (int64_t)B * m * n, dtype, scale, 0x5eed0000u + (uint32_t)rep, s);
            if (e != cudaSuccess) return cuda_fail(e, "fill launch");
            MUON_CUDA(cudaEventRecord(e0, s));
            if ((r = run_small(dc, s, sa, 0.0))) return r;
            MUON_CUDA(cudaEventRecord(e1, s));
            MUON_CUDA(cudaEventSynchronize(e1));
            float ms = 0.f;
            MUON_CUDA(cudaEventElapsedTime(&ms, e0, e1));
            if (rep > 0) times.push_back(ms);
        }
        std::sort(times.begin(), times.end());
        const double med = times[times.size() / 2] / B;
        logf(2, "autotune %dx%d fused path %d: %.4f ms/matrix", m, n, path, med);
        if (med < best.ms_per_matrix) best = TuneEntry{path, 256, med, 1, 128, 0};
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    *out = best;
    return MUON_OK;
}

// Chooses path and tile for one oriented shape.
static int choose_plan(const DevCtx& dc, cudaStream_t s, int m, int n, int dtype, int bucket_count,
                       const NsConfig& cfg, NsPlan* plan) {
    static std::once_flag load_once;      // MUON_TUNE_CACHE: measurements of an earlier process
    std::call_once(load_once, [] {
        if (const char* p = std::getenv("MUON_TUNE_CACHE")) muon_tune_load(p);
    });
    int path = cfg.path;
    if (const char* f = std::getenv("MUON_FORCE_PATH")) {
        if (!std::strcmp(f, "plain")) path = MUON_PATH_PLAIN;
        else if (!std::strcmp(f, "gram")) path = MUON_PATH_GRAM;
    }
    if (path == MUON_PATH_GRAM && cfg.segments.empty()) path = MUON_PATH_PLAIN;
    const TuneKey key = tune_key(dc, m, n, dtype);
    TuneEntry ent{-1, 256, 0.0, 0, 128, 0};
    bool have = false;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_tune.find(key);
        if (it != g_tune.end()) { ent = it->second; have = true; }
    }
    if (path == MUON_PATH_AUTO) {
        if (!have && env_flag("MUON_AUTOTUNE", true)) {
            const int B = std::max(1, std::min(bucket_count, 16));
            int r = autotune_shape(dc, s, m, n, dtype, B, cfg, &ent);
            if (r) return r;
            have = true;
            {
                std::lock_guard<std::mutex> lk(g_mu);
                g_tune[key] = ent;
            }
            if (const char* p = std::getenv("MUON_TUNE_CACHE")) save_tune_file(p);
        }
        if (have) {
            path = ent.path;
        } else {
            // without measurements: Gram needs 9m^2n + 11m^3 products, plain 15m^2n + 5m^3
            path = (n > m && !cfg.segments.empty()) ? MUON_PATH_GRAM : MUON_PATH_PLAIN;
        }
    }
    const int tile_n = (have && ent.path == path) ? ent.tile_n : 256;
    const int sym_tile_n = (have && ent.path == path) ? ent.sym_tile_n : 128;
    const int sym_dense = (have && ent.path == path) ? ent.sym_dense : 0;
    *plan = make_plan(cfg.coeffs, cfg.steps, cfg.segments, path, tile_n, m, n, sym_tile_n, sym_dense);
    if (const char* f = std::getenv("MUON_SYM_DENSE")) {    // override for tests: 0 triangle, 1 all tiles
        if (f[0] == '0' || f[0] == '1') plan->sym_dense = f[0] - '0';
    }
    // the fused small-matrix kernel: as measured, else whenever it applies
    const bool measured = have && ent.path == path;
    plan->fused = small_eligible(*plan, m, n, dtype) && (measured ? ent.fused != 0 : true);
    return MUON_OK;
}

static int save_tune_file(const char* path) {
    std::lock_guard<std::mutex> lk(g_mu);
    std::ofstream f(path);
    if (!f) return fail(MUON_EINVAL, "cannot write tune cache %s", path);
    f << "muon-tune v4\n";
    int nwritten = 0;
    for (auto& kv : g_tune) {
        std::string dev = std::get<0>(kv.first);
        std::replace(dev.begin(), dev.end(), '\t', ' ');
        f << dev << '\t' << std::get<1>(kv.first) << '\t' << std::get<2>(kv.first) << '\t' << std::get<3>(kv.first)
          << '\t' << std::get<4>(kv.first) << '\t' << std::get<5>(kv.first) << '\t' << kv.second.path << '\t'
          << kv.second.tile_n << '\t' << kv.second.ms_per_matrix << '\t' << kv.second.fused << '\t'
          << kv.second.sym_tile_n << '\t' << kv.second.sym_dense << '\n';
        ++nwritten;
    }
    return nwritten;
}

static int budget_bytes_chunk(size_t per_matrix, int count) {
    size_t budget = (size_t)8192 << 20;
    if (const char* e = std::getenv("MUON_WORKSPACE_MB")) {
        long v = std::atol(e);
        if (v > 0) budget = (size_t)v << 20;
    }
    size_t c = per_matrix ? budget / per_matrix : (size_t)count;
    if (c < 1) c = 1;
    if (c > (size_t)count) c = count;
    if (c > 65535) c = 65535;
    return (int)c;
}

static bool valid_dtype(int d) { return d == MUON_F32 || d == MUON_BF16 || d == MUON_F16; }

}  // namespace muon

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

using namespace muon;

extern "C" {

const char* muon_status_str(int status) {
    switch (status) {
        case MUON_OK: return "MUON_OK";
        case MUON_EINVAL: return "MUON_EINVAL: invalid argument";
        case MUON_EDTYPE: return "MUON_EDTYPE: unsupported dtype";
        case MUON_ENOMEM: return "MUON_ENOMEM: workspace allocation failed";
        case MUON_ECUDA: return "MUON_ECUDA: CUDA call failed";
        case MUON_ENONFINITE: return "MUON_ENONFINITE: non-finite Frobenius norm";
        case MUON_ETIMEOUT: return "MUON_ETIMEOUT: a bounded device wait gave up";
        case MUON_ENOTSUP: return "MUON_ENOTSUP: no sm_103a device";
        default: return "unknown muon status";
    }
}

const char* muon_last_error_message(void) { return t_last_error.c_str(); }

int muon_set_ns_config(const float coeffs[3], int steps, const int* segments, int num_segments, int path) try {
    int r = validate_segments(steps, segments, num_segments);
    if (r) return r;
    if (path != MUON_PATH_AUTO && path != MUON_PATH_PLAIN && path != MUON_PATH_GRAM)
        return fail(MUON_EINVAL, "bad path %d", path);
    if (coeffs && !(std::isfinite(coeffs[0]) && std::isfinite(coeffs[1]) && std::isfinite(coeffs[2])))
        return fail(MUON_EINVAL, "non-finite coefficients");
    std::lock_guard<std::mutex> lk(g_mu);
    if (coeffs) std::memcpy(g_cfg.coeffs, coeffs, sizeof g_cfg.coeffs);
    g_cfg.steps = steps;
    g_cfg.segments.assign(segments, segments + num_segments);
    g_cfg.path = path;
    g_cfg_version.fetch_add(1);
    return MUON_OK;
} MUON_CATCH_ALL

int muon_set_ns_precision(int dtype) {
    if (dtype != -1 && dtype != MUON_BF16 && dtype != MUON_F16)
        return fail(MUON_EDTYPE, "NS precision must be -1, MUON_BF16 or MUON_F16, got %d", dtype);
    std::lock_guard<std::mutex> lk(g_mu);
    g_cfg.ns_precision = dtype;
    g_cfg_version.fetch_add(1);
    return MUON_OK;
}

int muon_ns_orthogonalize(void* ptr, int64_t m, int64_t n, int64_t batch, int dtype, const float coeffs[3],
                          int steps, const int* segments, int num_segments, void* stream) try {
    muon::NvtxRange nvr("muon_ns_orthogonalize");
    if (!ptr) return fail(MUON_EINVAL, "ptr is NULL");
    if (m < 1 || n < 1 || batch < 1) return fail(MUON_EINVAL, "m, n, batch must be >= 1");
    if (m > (1 << 20) || n > (1 << 20)) return fail(MUON_EINVAL, "matrix side above 2^20");
    if (batch > INT32_MAX || batch > (INT64_MAX / 8) / (m * n))
        return fail(MUON_EINVAL, "batch x m x n overflows the byte range");
    if (!valid_dtype(dtype)) return fail(MUON_EDTYPE, "dtype %d", dtype);
    if (!coeffs || !(std::isfinite(coeffs[0]) && std::isfinite(coeffs[1]) && std::isfinite(coeffs[2])))
        return fail(MUON_EINVAL, "coeffs missing or non-finite");
    int r = validate_segments(steps, segments, num_segments);
    if (r) return r;
    DevCtx dc;
    if ((r = get_dev(dc))) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    const int trans = m > n;
    const int om = (int)std::min(m, n), on = (int)std::max(m, n);
    const int path = num_segments > 0 ? MUON_PATH_GRAM : MUON_PATH_PLAIN;
    std::vector<int> segs(segments, segments + num_segments);
    int tile_n = 256;
    int nsd;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        nsd = ns_dtype(dtype, g_cfg);
        auto it = g_tune.find(tune_key(dc, om, on, nsd));
        if (it != g_tune.end() && it->second.path == path) tile_n = it->second.tile_n;
    }
    NsPlan plan = make_plan(coeffs, steps, segs, path, tile_n, om, on);

    const size_t es = esize(dtype);
    if (dtype == MUON_BF16 && small_eligible(plan, om, on, nsd) && batch <= (1 << 20)) {
        const size_t tb = align_up(sizeof(MatEntry) * (size_t)batch, 256);
        Workspace* w = nullptr;
        if ((r = ws_get(dc.device, s, tb, &w))) return r;
        std::vector<MatEntry> h((size_t)batch);
        for (int64_t b = 0; b < batch; ++b) {
            char* p = static_cast<char*>(ptr) + (size_t)b * m * n * es;
            h[b] = MatEntry{p, nullptr, p, trans, 0};
        }
        MatEntry* d_table = reinterpret_cast<MatEntry*>(w->base);
        if ((r = upload_table(*w, h, d_table, s))) return r;
        const bool vec_ok = (reinterpret_cast<uintptr_t>(ptr) % 16 == 0) && (m % 8 == 0) && (n % 8 == 0);
        const SmallArgs sa = small_args(plan, d_table, (int)batch, om, on, 1, dtype, dtype, 0, 0.f, 0.f, 0.f, vec_ok,
                                        dc.status);
        if ((r = run_small(dc, s, sa, plan_alg_flops(plan, om, on) * (double)batch))) return r;
        std::lock_guard<std::mutex> lk(g_mu);
        g_last_path[{om, on, dtype}] = path;
        return MUON_OK;
    }
    const size_t per = chunk_layout(om, on, 1, nsd).total;
    const int chunk = budget_bytes_chunk(per, (int)std::min<int64_t>(batch, 65535));
    const size_t table_bytes = align_up(sizeof(MatEntry) * (size_t)batch, 256);
    const ChunkLayout L = chunk_layout(om, on, chunk, nsd);
    Workspace* w = nullptr;
    if ((r = ws_get(dc.device, s, table_bytes + L.total, &w))) return r;

    std::vector<MatEntry> h((size_t)batch);
    for (int64_t b = 0; b < batch; ++b) {
        char* p = static_cast<char*>(ptr) + (size_t)b * m * n * es;
        h[b] = MatEntry{p, nullptr, p, trans, 0};
    }
    MatEntry* d_table = reinterpret_cast<MatEntry*>(w->base);
    if ((r = upload_table(*w, h, d_table, s))) return r;
    char* cbase = w->base + table_bytes;
    const bool vec_ok = (reinterpret_cast<uintptr_t>(ptr) % 16 == 0) && (m % 8 == 0) && (n % 8 == 0);
    for (int64_t b0 = 0; b0 < batch; b0 += chunk) {
        const int B = (int)std::min<int64_t>(chunk, batch - b0);
        const ChunkLayout LB = chunk_layout(om, on, B, nsd);
        int* pc = nullptr;
        if ((r = prep_counters(dc.device, s, B, &pc))) return r;
        if ((r = run_prep(dc, s, cbase, LB, om, on, B, d_table + b0, dtype, dtype, nsd, false, 0, 0.f, vec_ok, pc)))
            return r;
        FinalEpi fin{EPI_OUT, d_table + b0, dtype, 0.f, 0.f, 0.f};
        if ((r = run_ns(dc, s, cbase, LB, om, on, B, nsd, plan, x_holds_u(nsd), fin))) return r;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_last_path[{om, on, dtype}] = path;
    }
    return MUON_OK;
} MUON_CATCH_ALL

int muon_step(void* const* params, const void* const* grads, void* const* moms, const int64_t* ms,
              const int64_t* ns, int64_t count, int param_dtype, int mom_dtype, float lr, float beta, float wd,
              int nesterov, void* stream) try {
    muon::NvtxRange nvr("muon_step");
    if (count < 0) return fail(MUON_EINVAL, "count < 0");
    if (count == 0) return MUON_OK;
    if (!params || !grads || !moms || !ms || !ns) return fail(MUON_EINVAL, "NULL array argument");
    if (!valid_dtype(param_dtype) || !valid_dtype(mom_dtype))
        return fail(MUON_EDTYPE, "dtypes %d / %d", param_dtype, mom_dtype);
    if (!std::isfinite(lr) || !std::isfinite(beta) || !std::isfinite(wd))
        return fail(MUON_EINVAL, "non-finite hyper-parameter");
    for (int64_t i = 0; i < count; ++i) {
        if (!params[i] || !grads[i] || !moms[i]) return fail(MUON_EINVAL, "NULL matrix pointer at %lld", (long long)i);
        if (ms[i] < 1 || ns[i] < 1) return fail(MUON_EINVAL, "matrix %lld has shape %lld x %lld", (long long)i,
                                                (long long)ms[i], (long long)ns[i]);
        if (ms[i] > (1 << 20) || ns[i] > (1 << 20)) return fail(MUON_EINVAL, "matrix side above 2^20");
    }
    int r;
    DevCtx dc;
    if ((r = get_dev(dc))) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    NsConfig cfg;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        cfg = g_cfg;
    }

    // shape buckets in order of first appearance
    std::vector<std::pair<int, int>> keys;
    std::map<std::pair<int, int>, std::vector<int64_t>> buckets;
    for (int64_t i = 0; i < count; ++i) {
        std::pair<int, int> k{(int)std::min(ms[i], ns[i]), (int)std::max(ms[i], ns[i])};
        auto it = buckets.find(k);
        if (it == buckets.end()) {
            keys.push_back(k);
            buckets[k] = {i};
        } else {
            it->second.push_back(i);
        }
    }
    const int nsd = ns_dtype(param_dtype, cfg);
    std::vector<NsPlan> plans(keys.size());
    std::vector<int> chunks(keys.size());
    size_t chunk_need = 0;
    for (size_t k = 0; k < keys.size(); ++k) {
        const int m = keys[k].first, n = keys[k].second;
        const int cnt = (int)buckets[keys[k]].size();
        if ((r = choose_plan(dc, s, m, n, nsd, cnt, cfg, &plans[k]))) return r;
        // the fused kernel reads bf16 parameters and bf16 or fp32 momentum
        if (param_dtype != MUON_BF16 || mom_dtype == MUON_F16) plans[k].fused = 0;
        if (plans[k].fused) {
            chunks[k] = cnt;            // one launch, no workspace beyond the table
            continue;
        }
        chunks[k] = budget_bytes_chunk(chunk_layout(m, n, 1, nsd).total, cnt);
        chunk_need = std::max(chunk_need, chunk_layout(m, n, chunks[k], nsd).total);
    }
    // per bucket: matrix count, first table row, 16-byte access
    std::vector<int64_t> counts(keys.size()), firsts(keys.size());
    std::vector<char> vecs(keys.size());
    {
        int64_t f = 0;
        for (size_t k = 0; k < keys.size(); ++k) {
            const auto& idx = buckets[keys[k]];
            counts[k] = (int64_t)idx.size();
            firsts[k] = f;
            f += counts[k];
            bool v = (keys[k].first % 8 == 0) && (keys[k].second % 8 == 0);
            for (int64_t i : idx)
                v = v && (reinterpret_cast<uintptr_t>(grads[i]) % 16 == 0) &&
                    (reinterpret_cast<uintptr_t>(moms[i]) % 16 == 0);
            vecs[k] = v ? 1 : 0;
        }
    }
    size_t work_bytes = 0;
    const std::vector<FusedLaunch> fused = plan_fused(dc, plans, keys, counts, nsd, &work_bytes);
    const size_t table_bytes = align_up(sizeof(MatEntry) * (size_t)count, 256);
    Workspace* w = nullptr;
    if ((r = ws_get(dc.device, s, table_bytes + work_bytes + chunk_need, &w))) return r;

    // the matrix table and the fused launches' work lists, as one byte block
    static_assert(256 % sizeof(MatEntry) == 0, "ring rows tile 256 bytes");
    std::vector<MatEntry> h((table_bytes + work_bytes) / sizeof(MatEntry));
    {
        size_t row = 0;
        for (auto& k : keys)
            for (int64_t i : buckets[k])
                h[row++] = MatEntry{grads[i], moms[i], params[i], ms[i] > ns[i] ? 1 : 0, 0};
        pack_fused(fused, reinterpret_cast<char*>(h.data()) + table_bytes);
    }
    MatEntry* d_table = reinterpret_cast<MatEntry*>(w->base);
    if ((r = upload_table(*w, h, d_table, s))) return r;
    char* cbase = w->base + table_bytes + work_bytes;

    // every fused bucket in one launch per group of buckets
    for (const auto& f : fused) {
        const SmallArgs sa = fused_args(f, w->base + table_bytes, plans, keys, counts, vecs,
                                        [&](int k) { return d_table + firsts[(size_t)k]; }, 0, param_dtype, mom_dtype,
                                        nesterov, beta, lr, wd, dc.status, nullptr);
        if ((r = run_small(dc, s, sa, fused_flops(f, plans, keys, counts)))) return r;
        std::lock_guard<std::mutex> lk(g_mu);
        for (int k : f.bks) g_last_path[{keys[(size_t)k].first, keys[(size_t)k].second, param_dtype}] = plans[(size_t)k].path;
    }

    size_t first = 0;
    for (size_t k = 0; k < keys.size(); ++k) {
        const int m = keys[k].first, n = keys[k].second;
        const auto& idx = buckets[keys[k]];
        const bool vec_ok = vecs[k] != 0;
        const float scale = 0.2f * std::sqrt((float)n);
        if (plans[k].fused) {
            first += idx.size();
            continue;
        }
        for (size_t c0 = 0; c0 < idx.size(); c0 += chunks[k]) {
            const int B = (int)std::min<size_t>(chunks[k], idx.size() - c0);
            const ChunkLayout L = chunk_layout(m, n, B, nsd);
            const MatEntry* dm = d_table + first + c0;
            int* pc = nullptr;
            if ((r = prep_counters(dc.device, s, B, &pc))) return r;
            if ((r = run_prep(dc, s, cbase, L, m, n, B, dm, param_dtype, mom_dtype, nsd, true, nesterov, beta,
                              vec_ok, pc)))
                return r;
            FinalEpi fin{EPI_UPDATE, dm, param_dtype, lr, wd, scale};
            if ((r = run_ns(dc, s, cbase, L, m, n, B, nsd, plans[k], x_holds_u(nsd), fin))) return r;
        }
        first += idx.size();
        std::lock_guard<std::mutex> lk(g_mu);
        g_last_path[{m, n, param_dtype}] = plans[k].path;
    }
    return MUON_OK;
} MUON_CATCH_ALL

int muon_autotune(const int64_t* ms, const int64_t* ns, int64_t count, int dtype, void* stream) try {
    if (count < 0 || (count > 0 && (!ms || !ns))) return fail(MUON_EINVAL, "bad shape arrays");
    if (!valid_dtype(dtype)) return fail(MUON_EDTYPE, "dtype %d", dtype);
    for (int64_t i = 0; i < count; ++i)
        if (ms[i] < 1 || ns[i] < 1 || ms[i] > (1 << 20) || ns[i] > (1 << 20))
            return fail(MUON_EINVAL, "shape %lld: sides must lie in [1, 2^20]", (long long)i);
    int r;
    DevCtx dc;
    if ((r = get_dev(dc))) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    NsConfig cfg;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        cfg = g_cfg;
    }
    std::map<std::pair<int, int>, int> shapes;
    for (int64_t i = 0; i < count; ++i) {
        shapes[{(int)std::min(ms[i], ns[i]), (int)std::max(ms[i], ns[i])}] += 1;
    }
    const int nsd = ns_dtype(dtype, cfg);
    for (auto& kv : shapes) {
        TuneEntry ent;
        const int B = std::max(1, std::min(kv.second, 16));
        if ((r = autotune_shape(dc, s, kv.first.first, kv.first.second, nsd, B, cfg, &ent))) return r;
        std::lock_guard<std::mutex> lk(g_mu);
        g_tune[tune_key(dc, kv.first.first, kv.first.second, nsd)] = ent;
    }
    if (const char* p = std::getenv("MUON_TUNE_CACHE")) save_tune_file(p);
    g_cfg_version.fetch_add(1);
    return MUON_OK;
} MUON_CATCH_ALL

int muon_tune_save(const char* path) try {
    if (!path) return fail(MUON_EINVAL, "path is NULL");
    int r = save_tune_file(path);
    return r < 0 ? r : MUON_OK;
} MUON_CATCH_ALL

int muon_tune_load(const char* path) try {
    if (!path) return fail(MUON_EINVAL, "path is NULL");
    std::ifstream f(path);
    if (!f) return 0;
    std::string line;
    if (!std::getline(f, line) || line != "muon-tune v4") return 0;
    DevCtx dc;
    int r = get_dev(dc);
    if (r) return r;
    const int cv = cudart_version();
    int loaded = 0;
    while (std::getline(f, line)) {
        std::istringstream ss(line);
        std::string dev, tok;
        std::vector<std::string> cols;
        while (std::getline(ss, tok, '\t')) cols.push_back(tok);
        if (cols.size() != 12) continue;
        try {
            const int sms = std::stoi(cols[1]), cuv = std::stoi(cols[2]);
            const int64_t m = std::stoll(cols[3]), n = std::stoll(cols[4]);
            const int dt = std::stoi(cols[5]), path = std::stoi(cols[6]), tile = std::stoi(cols[7]);
            const double ms = std::stod(cols[8]);
            const int fused = std::stoi(cols[9]);
            const int sym_tile = std::stoi(cols[10]);
            const int sym_dense = std::stoi(cols[11]);
            if (sym_dense != 0 && sym_dense != 1) continue;
            if (fused != 0 && fused != 1) continue;
            if (sym_tile != 128 && sym_tile != 256) continue;
            if (!std::isfinite(ms) || ms < 0.0) continue;     // costs feed the owner planner's sort
            if (cols[0] != dc.name || sms != dc.sms || cuv != cv) continue;          // stale: other device/runtime
            if (m < 1 || n < m || !valid_dtype(dt)) continue;
            if (path != MUON_PATH_PLAIN && path != MUON_PATH_GRAM) continue;
            if (tile != 128 && tile != 256) continue;
            std::lock_guard<std::mutex> lk(g_mu);
            g_tune[TuneKey{dc.name, sms, cuv, m, n, dt}] = TuneEntry{path, tile, ms, fused, sym_tile, sym_dense};
            ++loaded;
            g_cfg_version.fetch_add(1);
        } catch (...) {
            continue;   // corrupt line
        }
    }
    return loaded;
} MUON_CATCH_ALL

int muon_last_path(int64_t m, int64_t n, int dtype, int* path_out) {
    if (!path_out) return fail(MUON_EINVAL, "path_out is NULL");
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_last_path.find({std::min(m, n), std::max(m, n), dtype});
    if (it == g_last_path.end()) return MUON_EINVAL;
    *path_out = it->second;
    return MUON_OK;
}

int muon_sync_status(void* stream) {
    DevCtx dc;
    int r = get_dev(dc);
    if (r) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MUON_CUDA(cudaStreamSynchronize(s));
    int v = 0;
    MUON_CUDA(cudaMemcpy(&v, dc.status, sizeof v, cudaMemcpyDeviceToHost));
    if (v) MUON_CUDA(cudaMemset(dc.status, 0, sizeof v));
    if (v & STATUS_TIMEOUT) return MUON_ETIMEOUT;
    if (v & STATUS_NONFINITE) return MUON_ENONFINITE;
    return MUON_OK;
}

int muon_ns_flops(int64_t m, int64_t n, int path, const int* segments, int num_segments, double* nominal,
                  double* algorithmic) {
    if (m < 1 || n < 1 || !nominal || !algorithmic) return fail(MUON_EINVAL, "bad arguments");
    const double M = (double)std::min(m, n), N = (double)std::max(m, n);
    double nom = 0, alg = 0;
    auto prod = [&](double a, double b, double k, bool sym) {
        nom += 2 * a * b * k;
        alg += sym ? a * b * k : 2 * a * b * k;
    };
    if (path == MUON_PATH_PLAIN) {
        int steps = 0;
        if (num_segments > 0) {
            if (!segments || num_segments > 64) return fail(MUON_EINVAL, "segments NULL or more than 64");
            for (int i = 0; i < num_segments; ++i) {
                if (segments[i] < 1 || segments[i] > 64) return fail(MUON_EINVAL, "segment length outside [1, 64]");
                steps += segments[i];
            }
        } else {
            steps = 5;
        }
        for (int k = 0; k < steps; ++k) {
            prod(M, M, N, true);    // A = X X^T
            prod(M, M, M, true);    // A^2
            prod(M, N, M, false);   // B X
        }
    } else if (path == MUON_PATH_GRAM) {
        if (num_segments < 1 || !segments) return fail(MUON_EINVAL, "Gram path needs segments");
        if (num_segments > 64) return fail(MUON_EINVAL, "more than 64 segments");
        for (int si = 0; si < num_segments; ++si) {
            const int L = segments[si];
            if (L < 1 || L > 64) return fail(MUON_EINVAL, "segment length outside [1, 64]");
            prod(M, M, N, true);    // G = X X^T
            for (int j = 1; j <= L; ++j) {
                prod(M, M, M, true);                 // G^2
                if (j > 1) prod(M, M, M, true);      // P Q
                if (j < L) {
                    prod(M, M, M, true);             // P G
                    prod(M, M, M, true);             // (P G) P
                }
            }
            prod(M, N, M, false);   // Q X
        }
    } else {
        return fail(MUON_EINVAL, "path must be plain or gram");
    }
    *nominal = nom;
    *algorithmic = alg;
    return MUON_OK;
}

int64_t muon_launch_count(void) { return g_launches.load(); }

int muon_debug_arm_stall(int kernel, int stage) {
    if (kernel == STALL_NONE) {
        g_stall.store(0);
        return MUON_OK;
    }
    if ((kernel != STALL_PRODUCT && kernel != STALL_SMALL) || stage < 0 || stage > (1 << 20))
        return fail(MUON_EINVAL, "kernel must be 0, 1 or 2 and stage in [0, 2^20]");
    g_stall.store(((stage + 1) << 8) | kernel);
    return MUON_OK;
}

int muon_set_kernel_timing(int enable) {
    g_timing.store(enable ? 1 : 0);
    return MUON_OK;
}

int muon_kernel_timing_read(char* names, int64_t* launches, double* total_ms, double* work, int max_classes) try {
    if (max_classes < 0) return fail(MUON_EINVAL, "max_classes < 0");
    std::vector<TimedLaunch> recs;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        recs.swap(g_timed);
    }
    double ms_acc[KC_COUNT] = {0};
    double work_acc[KC_COUNT] = {0};
    int64_t cnt[KC_COUNT] = {0};
    for (auto& t : recs) {
        float ms = 0.f;
        if (cudaEventSynchronize(t.b) == cudaSuccess && cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess) {
            ms_acc[t.kclass] += ms;
            work_acc[t.kclass] += t.work;
            cnt[t.kclass] += 1;
        }
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (auto& t : recs) {
            g_event_pool.push_back(t.a);
            g_event_pool.push_back(t.b);
        }
    }
    const int n = std::min<int>(max_classes, KC_COUNT);
    for (int k = 0; k < n; ++k) {
        if (names) {
            std::strncpy(names + 32 * k, kclass_name(k), 31);
            names[32 * k + 31] = 0;
        }
        if (launches) launches[k] = cnt[k];
        if (total_ms) total_ms[k] = ms_acc[k];
        if (work) work[k] = work_acc[k];
    }
    return n;
} MUON_CATCH_ALL

int muon_debug_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t batch,
                    int dtype, int b_kmajor, int symmetric, int poly, float alpha, float pa, float pb, float pc,
                    int tile_n, void* stream) try {
    if (!A || !B || !C) return fail(MUON_EINVAL, "NULL operand");
    if (M < 1 || N < 1 || K < 1 || batch < 1) return fail(MUON_EINVAL, "bad sizes");
    if (M > (1 << 20) || N > (1 << 20) || K > (1 << 20)) return fail(MUON_EINVAL, "size above 2^20");
    if (!valid_dtype(dtype) && dtype != DT_TF32) return fail(MUON_EDTYPE, "dtype %d", dtype);
    if (dtype == DT_TF32 && !b_kmajor) return fail(MUON_EINVAL, "TF32 products need a K-major B");
    if ((symmetric || poly) && M != N) return fail(MUON_EINVAL, "symmetric product needs M == N");
    if (poly && (!symmetric || K != M)) return fail(MUON_EINVAL, "poly needs a symmetric square product");
    if (tile_n != 0 && tile_n != 128 && tile_n != 256) return fail(MUON_EINVAL, "tile_n must be 0, 128 or 256");
    if (is_half(dtype) || dtype == DT_TF32) {
        const int64_t ldb = b_kmajor ? K : N;
        const int64_t epr = dtype == DT_TF32 ? 4 : 8;
        if ((K % epr) || (ldb % epr) || (reinterpret_cast<uintptr_t>(A) % 16) || (reinterpret_cast<uintptr_t>(B) % 16))
            return fail(MUON_EINVAL, "tensor-core operands need 16-byte aligned rows");
    }
    int r;
    DevCtx dc;
    if ((r = get_dev(dc))) return r;
    GemmArgs g = gemm_base(dtype, dc.status);
    g.A = A; g.lda = K; g.strideA = M * K;
    g.B = B; g.b_kmajor = b_kmajor ? 1 : 0;
    g.ldb = b_kmajor ? K : N; g.strideB = N * K;
    g.M = (int)M; g.N = (int)N; g.K = (int)K; g.batch = (int)batch;
    g.symmetric = symmetric ? 1 : 0;
    g.alpha = alpha;
    g.C = C; g.ldc = N; g.strideC = M * N;
    g.tile_n = tile_n;   // 0: the launcher's default for the product kind
    if (poly) {
        g.epi = EPI_POLY;
        g.Gin = A; g.ldg = K; g.strideG = M * K;
        g.pa = pa; g.pb = pb; g.pc = pc;
    }
    return run_gemm(dc, reinterpret_cast<cudaStream_t>(stream), g, KC_OTHER);
} MUON_CATCH_ALL

}  // extern "C"

// ---------------------------------------------------------------------------
// Orthogonalisation without any allocation.
//
// Some callers may not allocate device memory at all: code running where the
// process's memory is owned by someone else's allocator (a framework's caching
// pool, a fixed per-job budget), or a real-time loop that forbids allocation
// after start-up.  muon_ns_orthogonalize grows a library workspace with
// cudaMalloc; this variant instead works inside one fixed array compiled into
// the library, so it calls no cudaMalloc, cudaFree, cudaMallocHost or other
// allocating routine.
//
// The array is NOALLOC_SCRATCH_BYTES long and every GPU that loads the library
// holds it until the process exits.  It holds, in order, a status word, the
// matrix table, and the NS buffers of the whole batch (no chunking), so a call
// whose batch does not fit is rejected with MUON_EINVAL.  All calls share the
// array and it keeps the last call's contents: the prep kernel's arrival
// counters are cleared on the caller's stream at the start of every call, and
// every other byte a call reads, except the status word, is written by that
// call first.
// Two calls that overlap on the GPU (different streams, or different host
// threads) race on the array; the next call after such a race starts clean.
// Device-detected errors of these calls (a bounded wait that gave up, a
// non-finite norm) accumulate in the array's status word (zero at load),
// which muon_noalloc_sync_status reads and clears without allocating.
// ---------------------------------------------------------------------------

namespace muon {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];
// the prep kernel's per-matrix arrival counters (cleared by every call)
constexpr int NOALLOC_MAX_BATCH = 65535;
static __device__ int g_noalloc_prep_cnt[NOALLOC_MAX_BATCH + 1];

struct NoallocDev {
    char* base = nullptr;   // device address of g_noalloc_scratch on this device
    int* pcnt = nullptr;    // device address of g_noalloc_prep_cnt
    int sms = 0;
};
static std::map<int, NoallocDev> g_noalloc_dev;

// Once per device, with that device current: the device address of the array
// (host code only sees a stand-in symbol) and the SM count.
static int noalloc_setup(NoallocDev& out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_noalloc_dev.find(dev);
    if (it == g_noalloc_dev.end()) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (!(major == 10 && minor == 3))
            return fail(MUON_ENOTSUP, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
        NoallocDev d;
        d.base = static_cast<char*>(p);
        e = cudaGetSymbolAddress(&p, g_noalloc_prep_cnt);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(counters)");
        d.pcnt = static_cast<int*>(p);
        d.sms = sms;
        it = g_noalloc_dev.emplace(dev, d).first;
    }
    out = it->second;
    return MUON_OK;
}

__global__ void noalloc_table_kernel(MatEntry* t, char* base, int64_t stride_bytes, int trans, int batch) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < batch) {
        char* p = base + (int64_t)b * stride_bytes;
        t[b] = MatEntry{p, nullptr, p, trans, 0};
    }
}

}  // namespace muon

extern "C" int muon_ns_orthogonalize_noalloc(void* ptr, int64_t m, int64_t n, int64_t batch, int dtype,
                                             const float coeffs[3], int steps, const int* segments,
                                             int num_segments, void* stream) try {
    if (!ptr) return fail(MUON_EINVAL, "ptr is NULL");
    if (m < 1 || n < 1 || batch < 1) return fail(MUON_EINVAL, "m, n, batch must be >= 1");
    if (m > (1 << 20) || n > (1 << 20) || batch > NOALLOC_MAX_BATCH) return fail(MUON_EINVAL, "size out of range");
    if (!valid_dtype(dtype)) return fail(MUON_EDTYPE, "dtype %d", dtype);
    if (!coeffs || !(std::isfinite(coeffs[0]) && std::isfinite(coeffs[1]) && std::isfinite(coeffs[2])))
        return fail(MUON_EINVAL, "coeffs missing or non-finite");
    int r = validate_segments(steps, segments, num_segments);
    if (r) return r;

    const int om = (int)std::min(m, n), on = (int)std::max(m, n);
    int nsd;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        nsd = ns_dtype(dtype, g_cfg);
    }
    const ChunkLayout L = chunk_layout(om, on, (int)batch, nsd);
    const size_t status_bytes = 256;
    const size_t table_bytes = align_up(sizeof(MatEntry) * (size_t)batch, 256);
    const size_t need = status_bytes + table_bytes + L.total;
    if (need > NOALLOC_SCRATCH_BYTES)
        return fail(MUON_EINVAL, "%lld matrices of %lld x %lld need %zu bytes of scratch; the fixed scratch holds %zu",
                    (long long)batch, (long long)m, (long long)n, need, NOALLOC_SCRATCH_BYTES);

    NoallocDev nd;
    if ((r = noalloc_setup(nd))) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DevCtx dc;
    dc.sms = nd.sms;
    dc.status = reinterpret_cast<int*>(nd.base);
    // the arrival counters start at zero: a call that raced with another one
    // (or was cut short) may have left them non-zero.  The status word is not
    // cleared here: it keeps every call's errors until it is read.
    MUON_CUDA(cudaMemsetAsync(nd.pcnt, 0, sizeof(int) * (size_t)batch, s));

    MatEntry* d_table = reinterpret_cast<MatEntry*>(nd.base + status_bytes);
    char* cbase = nd.base + status_bytes + table_bytes;
    const int64_t stride_bytes = m * n * (int64_t)esize(dtype);
    note_launch_begin(KC_OTHER, s);
    noalloc_table_kernel<<<(int)((batch + 127) / 128), 128, 0, s>>>(d_table, static_cast<char*>(ptr), stride_bytes,
                                                                     m > n ? 1 : 0, (int)batch);
    note_launch_end(KC_OTHER, 0.0, s);
    MUON_CUDA(cudaGetLastError());

    const int path = num_segments > 0 ? MUON_PATH_GRAM : MUON_PATH_PLAIN;
    std::vector<int> segs(segments, segments + num_segments);
    NsPlan plan = make_plan(coeffs, steps, segs, path, 256, om, on);
    const bool vec_ok = (reinterpret_cast<uintptr_t>(ptr) % 16 == 0) && (m % 8 == 0) && (n % 8 == 0);
    if ((r = run_prep(dc, s, cbase, L, om, on, (int)batch, d_table, dtype, dtype, nsd, false, 0, 0.f, vec_ok,
                      nd.pcnt)))
        return r;
    FinalEpi fin{EPI_OUT, d_table, dtype, 0.f, 0.f, 0.f};
    return run_ns(dc, s, cbase, L, om, on, (int)batch, nsd, plan, x_holds_u(nsd), fin);
} MUON_CATCH_ALL

extern "C" int muon_noalloc_sync_status(void* stream) try {
    NoallocDev nd;
    int r = noalloc_setup(nd);
    if (r) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MUON_CUDA(cudaStreamSynchronize(s));
    int v = 0;
    MUON_CUDA(cudaMemcpy(&v, nd.base, sizeof v, cudaMemcpyDeviceToHost));
    if (v) MUON_CUDA(cudaMemset(nd.base, 0, sizeof v));
    if (v & STATUS_TIMEOUT) return MUON_ETIMEOUT;
    if (v & STATUS_NONFINITE) return MUON_ENONFINITE;
    return MUON_OK;
} MUON_CATCH_ALL

// ---------------------------------------------------------------------------
// Persistent groups: a fixed set of matrices stepped many times (the optimizer
// object of a training loop).  Bucketing, plans, the pointer table and the
// workspace are built once; every step is then one replay of a CUDA graph
// captured on the group's own stream, preceded by a 16-byte copy of the
// step's hyper-parameters into a device block the kernels read.
// ---------------------------------------------------------------------------

struct muon_group {
    int device = -1;
    DevCtx dc;
    int64_t count = 0;
    int param_dtype = 0, mom_dtype = 0;
    int ns_dtype = 0;                               // NS working precision of the current plans
    std::vector<MatEntry> entries;                  // bucket order
    std::vector<std::pair<int, int>> keys;          // oriented shape per bucket
    std::vector<int64_t> bucket_first, bucket_size;
    std::vector<char> vec_ok;
    std::vector<FusedLaunch> fused;                 // fused launches and their work lists
    char* d_work = nullptr;                         // work lists on the device
    std::vector<NsPlan> plans;
    std::vector<int> chunks;
    char* ws = nullptr;
    size_t ws_bytes = 0;
    int* pcnt = nullptr;                            // prep counters at the end of ws (zero between launches)
    MatEntry* d_table = nullptr;
    float* d_hyper = nullptr;
    char* cbase = nullptr;
    float* h_hyper[4] = {nullptr, nullptr, nullptr, nullptr};
    cudaEvent_t hev[4] = {nullptr, nullptr, nullptr, nullptr};
    int hslot = 0;
    cudaStream_t cap = nullptr;                     // private capture stream
    cudaGraphExec_t exec = nullptr;
    int64_t graph_launches = 0;                     // kernels in the captured graph
    bool graph_failed = false;
    bool direct_done = false;                       // a direct step ran since the last (re)plan
    uint64_t version = 0;                           // g_cfg_version the plans were made for
};

namespace muon {

static int group_enqueue(muon_group* g, cudaStream_t s) {
    NvtxRange nvr("muon_group_step");
    int r;
    for (const auto& f : g->fused) {
        const SmallArgs sa = fused_args(f, g->d_work, g->plans, g->keys, g->bucket_size, g->vec_ok,
                                        [&](int k) { return g->d_table + g->bucket_first[(size_t)k]; }, 0,
                                        g->param_dtype, g->mom_dtype, 0, 0.f, 0.f, 0.f, g->dc.status, g->d_hyper);
        if ((r = run_small(g->dc, s, sa, fused_flops(f, g->plans, g->keys, g->bucket_size)))) return r;
    }
    for (size_t k = 0; k < g->keys.size(); ++k) {
        const int m = g->keys[k].first, n = g->keys[k].second;
        const int64_t first = g->bucket_first[k], cnt = g->bucket_size[k];
        const NsPlan& plan = g->plans[k];
        if (plan.fused) continue;
        const float scale = 0.2f * std::sqrt((float)n);
        for (int64_t c0 = 0; c0 < cnt; c0 += g->chunks[k]) {
            const int B = (int)std::min<int64_t>(g->chunks[k], cnt - c0);
            const ChunkLayout L = chunk_layout(m, n, B, g->ns_dtype);
            const MatEntry* dm = g->d_table + first + c0;
            if ((r = run_prep(g->dc, s, g->cbase, L, m, n, B, dm, g->param_dtype, g->mom_dtype, g->ns_dtype, true,
                              0, 0.f, g->vec_ok[k] != 0, g->pcnt, g->d_hyper)))
                return r;
            FinalEpi fin{EPI_UPDATE, dm, g->param_dtype, 0.f, 0.f, scale, g->d_hyper};
            if ((r = run_ns(g->dc, s, g->cbase, L, m, n, B, g->ns_dtype, plan, x_holds_u(g->ns_dtype), fin))) return r;
        }
    }
    return MUON_OK;
}

static void group_drop_graph(muon_group* g) {
    if (g->exec) cudaGraphExecDestroy(g->exec);
    g->exec = nullptr;
    g->graph_launches = 0;
}

// (Re)plans the group: paths and tiles per bucket (autotuning shapes not in the
// cache), workspace and pointer table.  Synchronises the stream when it grows.
static int group_plan(muon_group* g, cudaStream_t s) {
    NsConfig cfg;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        cfg = g_cfg;
    }
    const uint64_t version = g_cfg_version.load();
    int r;
    size_t chunk_need = 0;
    g->plans.assign(g->keys.size(), NsPlan{});
    g->chunks.assign(g->keys.size(), 1);
    g->ns_dtype = ns_dtype(g->param_dtype, cfg);
    for (size_t k = 0; k < g->keys.size(); ++k) {
        const int m = g->keys[k].first, n = g->keys[k].second;
        const int cnt = (int)g->bucket_size[k];
        if ((r = choose_plan(g->dc, s, m, n, g->ns_dtype, cnt, cfg, &g->plans[k]))) return r;
        // the fused kernel reads bf16 parameters and bf16 or fp32 momentum
        if (g->param_dtype != MUON_BF16 || g->mom_dtype == MUON_F16) g->plans[k].fused = 0;
        if (g->plans[k].fused) {
            g->chunks[k] = cnt;
            continue;
        }
        g->chunks[k] = budget_bytes_chunk(chunk_layout(m, n, 1, g->ns_dtype).total, cnt);
        chunk_need = std::max(chunk_need, chunk_layout(m, n, g->chunks[k], g->ns_dtype).total);
    }
    size_t work_bytes = 0;
    g->fused = plan_fused(g->dc, g->plans, g->keys, g->bucket_size, g->ns_dtype, &work_bytes);
    const size_t table_bytes = align_up(sizeof(MatEntry) * (size_t)g->count, 256);
    const size_t cnt_off = align_up(table_bytes + 256 + work_bytes + chunk_need, 256);
    const size_t need = cnt_off + sizeof(int) * (size_t)g->count;
    if (g->ws_bytes < need) {
        MUON_CUDA(cudaStreamSynchronize(s));
        group_drop_graph(g);
        if (g->ws) cudaFree(g->ws);
        g->ws = nullptr;
        g->ws_bytes = 0;
        cudaError_t e = dev_alloc(reinterpret_cast<void**>(&g->ws), need);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(MUON_ENOMEM, "group workspace of %zu bytes: %s", need, cudaGetErrorString(e));
        }
        g->ws_bytes = need;
        g->d_table = reinterpret_cast<MatEntry*>(g->ws);
        g->d_hyper = reinterpret_cast<float*>(g->ws + table_bytes);
        MUON_CUDA(cudaMemcpy(g->d_table, g->entries.data(), sizeof(MatEntry) * g->entries.size(),
                             cudaMemcpyHostToDevice));
    }
    // the fused launches' work lists after the hyper-parameter block, then the chunks
    g->d_work = g->ws + table_bytes + 256;
    g->cbase = g->d_work + work_bytes;
    if (work_bytes) {
        std::vector<char> blk(work_bytes);
        pack_fused(g->fused, blk.data());
        MUON_CUDA(cudaStreamSynchronize(s));
        MUON_CUDA(cudaMemcpy(g->d_work, blk.data(), work_bytes, cudaMemcpyHostToDevice));
    }
    // the prep counters after the chunks (they move with them): zeroed
    g->pcnt = reinterpret_cast<int*>(g->ws + cnt_off);
    MUON_CUDA(cudaMemsetAsync(g->pcnt, 0, sizeof(int) * (size_t)g->count, s));
    group_drop_graph(g);
    g->direct_done = false;
    g->version = version;
    return MUON_OK;
}

}  // namespace muon

extern "C" {

int muon_group_create(void* const* params, const void* const* grads, void* const* moms, const int64_t* ms,
                      const int64_t* ns, int64_t count, int param_dtype, int mom_dtype, muon_group** out) try {
    if (!out) return fail(MUON_EINVAL, "out is NULL");
    *out = nullptr;
    if (count < 1) return fail(MUON_EINVAL, "a group needs at least one matrix");
    if (!params || !grads || !moms || !ms || !ns) return fail(MUON_EINVAL, "NULL array argument");
    if (!valid_dtype(param_dtype) || !valid_dtype(mom_dtype))
        return fail(MUON_EDTYPE, "dtypes %d / %d", param_dtype, mom_dtype);
    for (int64_t i = 0; i < count; ++i) {
        if (!params[i] || !grads[i] || !moms[i]) return fail(MUON_EINVAL, "NULL matrix pointer at %lld", (long long)i);
        if (ms[i] < 1 || ns[i] < 1 || ms[i] > (1 << 20) || ns[i] > (1 << 20))
            return fail(MUON_EINVAL, "matrix %lld has shape %lld x %lld", (long long)i, (long long)ms[i],
                        (long long)ns[i]);
    }
    int r;
    DevCtx dc;
    if ((r = get_dev(dc))) return r;
    muon_group* g = new (std::nothrow) muon_group();
    if (!g) return fail(MUON_ENOMEM, "group allocation");
    // released to the caller on success; destroyed on every early return or throw
    std::unique_ptr<muon_group, int (*)(muon_group*)> holder(g, muon_group_destroy);
    g->device = dc.device;
    g->dc = dc;
    g->count = count;
    g->param_dtype = param_dtype;
    g->mom_dtype = mom_dtype;
    std::map<std::pair<int, int>, std::vector<int64_t>> buckets;
    for (int64_t i = 0; i < count; ++i) {
        std::pair<int, int> k{(int)std::min(ms[i], ns[i]), (int)std::max(ms[i], ns[i])};
        if (!buckets.count(k)) g->keys.push_back(k);
        buckets[k].push_back(i);
    }
    for (auto& k : g->keys) {
        const auto& idx = buckets[k];
        g->bucket_first.push_back((int64_t)g->entries.size());
        g->bucket_size.push_back((int64_t)idx.size());
        bool vec = (k.first % 8 == 0) && (k.second % 8 == 0);
        for (int64_t i : idx) {
            g->entries.push_back(MatEntry{grads[i], moms[i], params[i], ms[i] > ns[i] ? 1 : 0, 0});
            vec = vec && (reinterpret_cast<uintptr_t>(grads[i]) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(moms[i]) % 16 == 0);
        }
        g->vec_ok.push_back(vec ? 1 : 0);
    }
    cudaError_t e = cudaStreamCreateWithFlags(&g->cap, cudaStreamNonBlocking);
    for (int i = 0; i < 4 && e == cudaSuccess; ++i) {
        e = cudaMallocHost(reinterpret_cast<void**>(&g->h_hyper[i]), 4 * sizeof(float));
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&g->hev[i], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return cuda_fail(e, "group stream/event/pinned setup");
    *out = holder.release();
    return MUON_OK;
} MUON_CATCH_ALL

int muon_group_step(muon_group* g, float lr, float beta, float wd, int nesterov, void* stream) try {
    if (!g) return fail(MUON_EINVAL, "group is NULL");
    if (!std::isfinite(lr) || !std::isfinite(beta) || !std::isfinite(wd))
        return fail(MUON_EINVAL, "non-finite hyper-parameter");
    int dev = -1;
    MUON_CUDA(cudaGetDevice(&dev));
    if (dev != g->device) return fail(MUON_EINVAL, "group belongs to device %d, current device is %d", g->device, dev);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int r;
    if (g->version != g_cfg_version.load() || !g->ws)
        if ((r = group_plan(g, s))) return r;

    // this step's hyper-parameters -> device block (ordered before the step on s)
    const int slot = g->hslot;
    g->hslot = (g->hslot + 1) % 4;
    MUON_CUDA(cudaEventSynchronize(g->hev[slot]));
    float* h = g->h_hyper[slot];
    h[0] = lr; h[1] = beta; h[2] = wd; h[3] = nesterov ? 1.f : 0.f;
    MUON_CUDA(cudaMemcpyAsync(g->d_hyper, h, 4 * sizeof(float), cudaMemcpyHostToDevice, s));
    MUON_CUDA(cudaEventRecord(g->hev[slot], s));

    // the first step after (re)planning runs directly; later ones replay a graph
    const bool use_graph = g->direct_done && !g->graph_failed && !g_timing.load() && env_flag("MUON_GRAPH", true);
    if (!use_graph) {
        if ((r = group_enqueue(g, s))) return r;
        g->direct_done = true;
    } else {
        if (!g->exec) {
            // capture on the private stream, so the caller's stream may be the legacy one
            const int64_t l0 = g_launches.load();
            cudaGraph_t graph = nullptr;
            cudaError_t e = cudaStreamBeginCapture(g->cap, cudaStreamCaptureModeThreadLocal);
            if (e == cudaSuccess) {
                r = group_enqueue(g, g->cap);
                e = cudaStreamEndCapture(g->cap, &graph);
                if (r == MUON_OK && e == cudaSuccess) e = cudaGraphInstantiate(&g->exec, graph, 0);
                if (graph) cudaGraphDestroy(graph);
            }
            const int64_t captured = g_launches.load() - l0;
            g_launches.fetch_sub(captured);            // counted when replayed
            if (r != MUON_OK || e != cudaSuccess || !g->exec) {
                cudaGetLastError();
                group_drop_graph(g);
                g->graph_failed = true;
                logf(1, "group graph capture failed (%s); stepping with direct launches",
                     e != cudaSuccess ? cudaGetErrorString(e) : "launch error");
                if ((r = group_enqueue(g, s))) return r;
                goto done;
            }
            g->graph_launches = captured;
        }
        MUON_CUDA(cudaGraphLaunch(g->exec, s));
        g_launches.fetch_add(g->graph_launches);
    }
done:
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (size_t k = 0; k < g->keys.size(); ++k)
            g_last_path[{g->keys[k].first, g->keys[k].second, g->param_dtype}] = g->plans[k].path;
    }
    return MUON_OK;
} MUON_CATCH_ALL

int muon_group_destroy(muon_group* g) {
    if (!g) return MUON_OK;
    int dev = -1;
    cudaGetDevice(&dev);
    if (dev == g->device) {
        if (g->cap) cudaStreamSynchronize(g->cap);
        for (int i = 0; i < 4; ++i)
            if (g->hev[i]) cudaEventSynchronize(g->hev[i]);
    }
    group_drop_graph(g);
    if (g->ws) cudaFree(g->ws);
    for (int i = 0; i < 4; ++i) {
        if (g->h_hyper[i]) cudaFreeHost(g->h_hyper[i]);
        if (g->hev[i]) cudaEventDestroy(g->hev[i]);
    }
    if (g->cap) cudaStreamDestroy(g->cap);
    delete g;
    return MUON_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Owner placement for a multi-rank step: every matrix gets one owner rank
// that runs its update ("DMuon" news page, section 3; summary, section 2.3).
// The pages minimise the predicted makespan with an MILP over measured
// per-shape costs and fall back to a greedy heuristic when the search space
// is too large; this is that fallback, longest processing time first.
// ---------------------------------------------------------------------------

extern "C" int muon_owner_plan(const int64_t* ms, const int64_t* ns, int64_t count, int dtype, int ranks,
                               int* owner_out, double* load_out, double* makespan_out, int* measured_out) try {
    if (count < 0 || ranks < 1) return fail(MUON_EINVAL, "count < 0 or ranks < 1");
    if (count > 0 && (!ms || !ns || !owner_out)) return fail(MUON_EINVAL, "NULL array argument");
    if (!valid_dtype(dtype)) return fail(MUON_EDTYPE, "dtype %d", dtype);
    for (int64_t i = 0; i < count; ++i) {
        if (ms[i] < 1 || ns[i] < 1) return fail(MUON_EINVAL, "matrix %lld has a zero side", (long long)i);
        if (ms[i] > (1 << 20) || ns[i] > (1 << 20)) return fail(MUON_EINVAL, "matrix %lld: side above 2^20", (long long)i);
    }
    NsConfig cfg;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        cfg = g_cfg;
    }
    // cost per matrix: measured ms per matrix when every shape has a tune entry
    // (measured on this process's device), else algorithmic FLOPs of the path
    // the library picks without measurements
    std::vector<double> cost((size_t)count, 0.0);
    bool measured = count > 0;
    const int nsd = ns_dtype(dtype, cfg);       // tune entries are kept per NS precision
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int64_t i = 0; i < count && measured; ++i) {
            const int64_t m = std::min(ms[i], ns[i]), n = std::max(ms[i], ns[i]);
            bool found = false;
            for (auto& kv : g_tune) {
                if (std::get<3>(kv.first) == m && std::get<4>(kv.first) == n && std::get<5>(kv.first) == nsd) {
                    cost[(size_t)i] = kv.second.ms_per_matrix;
                    found = true;
                    break;
                }
            }
            measured = found;
        }
    }
    if (!measured) {
        for (int64_t i = 0; i < count; ++i) {
            const int m = (int)std::min(ms[i], ns[i]), n = (int)std::max(ms[i], ns[i]);
            const int path = (n > m && !cfg.segments.empty()) ? MUON_PATH_GRAM : MUON_PATH_PLAIN;
            cost[(size_t)i] = plan_alg_flops(make_plan(cfg.coeffs, cfg.steps, cfg.segments, path, 256, m, n), m, n);
        }
    }
    std::vector<int64_t> order((size_t)count);
    for (int64_t i = 0; i < count; ++i) order[(size_t)i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](int64_t x, int64_t y) { return cost[(size_t)x] > cost[(size_t)y]; });
    std::vector<double> load((size_t)ranks, 0.0);
    for (int64_t i : order) {
        int best = 0;
        for (int rk = 1; rk < ranks; ++rk)
            if (load[(size_t)rk] < load[(size_t)best]) best = rk;
        owner_out[i] = best;
        load[(size_t)best] += cost[(size_t)i];
    }
    double mk = 0.0;
    for (double l : load) mk = std::max(mk, l);
    if (load_out)
        for (int rk = 0; rk < ranks; ++rk) load_out[rk] = load[(size_t)rk];
    if (makespan_out) *makespan_out = mk;
    if (measured_out) *measured_out = measured ? 1 : 0;
    return MUON_OK;
} MUON_CATCH_ALL

// ---------------------------------------------------------------------------
// Packed exchange buffers ("DMuon" summary, sections 2.1 and 2.3): each rank's
// owned matrices contiguous in one segment, segments of equal length so that
// one reduce-scatter (gradients to their owners) or all-gather (updated
// parameters from their owners) moves the whole buffer.
// ---------------------------------------------------------------------------

extern "C" int muon_pack_plan(const int64_t* ms, const int64_t* ns, const int* owner, int64_t count, int ranks,
                              int64_t align_elems, int64_t* offset_out, int64_t* seg_elems_out) try {
    if (count < 0 || ranks < 1 || align_elems < 1) return fail(MUON_EINVAL, "count < 0, ranks < 1 or align < 1");
    if (!seg_elems_out || (count > 0 && (!ms || !ns || !owner || !offset_out)))
        return fail(MUON_EINVAL, "NULL array argument");
    for (int64_t i = 0; i < count; ++i) {
        if (ms[i] < 1 || ns[i] < 1) return fail(MUON_EINVAL, "matrix %lld has a zero side", (long long)i);
        if (owner[i] < 0 || owner[i] >= ranks) return fail(MUON_EINVAL, "owner of matrix %lld out of range", (long long)i);
        if (ms[i] > ((int64_t)1 << 31) / ns[i]) return fail(MUON_EINVAL, "matrix %lld above 2^31 elements", (long long)i);
    }
    auto up = [&](int64_t x) { return (x + align_elems - 1) / align_elems * align_elems; };
    std::vector<int64_t> cur((size_t)ranks, 0);
    for (int64_t i = 0; i < count; ++i) {       // ascending index within each rank
        int64_t& c = cur[(size_t)owner[i]];
        offset_out[i] = up(c);
        c = offset_out[i] + ms[i] * ns[i];
    }
    int64_t seg = 0;
    for (int64_t c : cur) seg = std::max(seg, up(c));
    for (int64_t i = 0; i < count; ++i) offset_out[i] += (int64_t)owner[i] * seg;
    *seg_elems_out = seg;
    return MUON_OK;
} MUON_CATCH_ALL

extern "C" int muon_pack(void* const* mats, const int64_t* ms, const int64_t* ns, const int64_t* offsets,
                         int64_t count, int dtype, void* packed, int to_packed, void* stream) try {
    if (count < 0) return fail(MUON_EINVAL, "count < 0");
    if (count == 0) return MUON_OK;
    if (!mats || !ms || !ns || !offsets || !packed) return fail(MUON_EINVAL, "NULL argument");
    if (!valid_dtype(dtype)) return fail(MUON_EDTYPE, "dtype %d", dtype);
    if (count > INT32_MAX) return fail(MUON_EINVAL, "more than 2^31 - 1 matrices");
    const int es = (int)esize(dtype);
    const bool pk16 = (reinterpret_cast<uintptr_t>(packed) & 15) == 0;
    int64_t nchunks = 0;                        // checked before any table is built
    for (int64_t i = 0; i < count; ++i) {
        if (!mats[i]) return fail(MUON_EINVAL, "NULL matrix pointer at %lld", (long long)i);
        if (ms[i] < 1 || ns[i] < 1 || offsets[i] < 0) return fail(MUON_EINVAL, "bad size or offset at %lld", (long long)i);
        if (ms[i] > (INT64_MAX / 16) / ns[i] || offsets[i] > INT64_MAX / 16 - ms[i] * ns[i])
            return fail(MUON_EINVAL, "matrix %lld: size or offset overflows the byte range", (long long)i);
        nchunks += (ms[i] * ns[i] + PACK_CHUNK_ELEMS - 1) / PACK_CHUNK_ELEMS;
        if (nchunks > INT32_MAX) return fail(MUON_EINVAL, "too many elements");
    }
    std::vector<PackMat> pm((size_t)count);
    std::vector<PackChunk> chunks;
    chunks.reserve((size_t)nchunks);
    for (int64_t i = 0; i < count; ++i) {
        const int64_t numel = ms[i] * ns[i];
        const bool v = pk16 && (reinterpret_cast<uintptr_t>(mats[i]) & 15) == 0 && (offsets[i] * es) % 16 == 0;
        pm[(size_t)i] = PackMat{mats[i], offsets[i], v ? 1 : 0, 0};
        for (int64_t s0 = 0; s0 < numel; s0 += PACK_CHUNK_ELEMS)
            chunks.push_back(PackChunk{s0, (int)i, (int)std::min<int64_t>(PACK_CHUNK_ELEMS, numel - s0)});
    }
    int r;
    DevCtx dc;
    if ((r = get_dev(dc))) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t tb = align_up(sizeof(PackMat) * pm.size(), 256);
    const size_t cb = align_up(sizeof(PackChunk) * chunks.size(), 256);
    Workspace* w = nullptr;
    if ((r = ws_get(dc.device, s, tb + cb, &w))) return r;
    static_assert(256 % sizeof(MatEntry) == 0, "ring rows tile 256 bytes");
    std::vector<MatEntry> rows((tb + cb) / sizeof(MatEntry));
    std::memcpy(rows.data(), pm.data(), sizeof(PackMat) * pm.size());
    std::memcpy(reinterpret_cast<char*>(rows.data()) + tb, chunks.data(), sizeof(PackChunk) * chunks.size());
    if ((r = upload_table(*w, rows, reinterpret_cast<MatEntry*>(w->base), s))) return r;
    PackArgs a;
    a.mats = reinterpret_cast<const PackMat*>(w->base);
    a.chunks = reinterpret_cast<const PackChunk*>(w->base + tb);
    a.packed = packed;
    a.esize = es;
    a.to_packed = to_packed ? 1 : 0;
    double bytes = 0;
    for (int64_t i = 0; i < count; ++i) bytes += 2.0 * (double)(ms[i] * ns[i]) * es;
    note_launch_begin(KC_PACK, s);
    cudaError_t e = launch_pack(a, (int)chunks.size(), s);
    note_launch_end(KC_PACK, bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    return MUON_OK;
} MUON_CATCH_ALL

// ---------------------------------------------------------------------------
// AdamW for the non-matrix parameters ("MuonX" page, section 2)
// ---------------------------------------------------------------------------

extern "C" int muon_adamw_step(void* const* params, const void* const* grads, void* const* exp_avg,
                               void* const* exp_avg_sq, const int64_t* numels, int64_t count, int param_dtype,
                               int state_dtype, float lr, float beta1, float beta2, float eps, float wd,
                               int64_t step, void* stream) try {
    if (count < 0) return fail(MUON_EINVAL, "count < 0");
    if (count == 0) return MUON_OK;
    if (!params || !grads || !exp_avg || !exp_avg_sq || !numels) return fail(MUON_EINVAL, "NULL array argument");
    if (!valid_dtype(param_dtype) || !(state_dtype == MUON_F32 || state_dtype == MUON_BF16))
        return fail(MUON_EDTYPE, "dtypes %d / %d (moments: fp32 or bf16)", param_dtype, state_dtype);
    if (step < 1) return fail(MUON_EINVAL, "step counts from 1");
    if (!std::isfinite(lr) || !std::isfinite(beta1) || !std::isfinite(beta2) || !std::isfinite(eps) ||
        !std::isfinite(wd) || beta1 < 0.f || beta1 >= 1.f || beta2 < 0.f || beta2 >= 1.f || eps < 0.f)
        return fail(MUON_EINVAL, "bad hyper-parameter");
    if (count > INT32_MAX) return fail(MUON_EINVAL, "more than 2^31 - 1 tensors");
    int64_t nchunks = 0;                        // checked before any table is built
    for (int64_t i = 0; i < count; ++i) {
        if (!params[i] || !grads[i] || !exp_avg[i] || !exp_avg_sq[i])
            return fail(MUON_EINVAL, "NULL tensor pointer at %lld", (long long)i);
        if (numels[i] < 0 || numels[i] > INT64_MAX / 16) return fail(MUON_EINVAL, "bad size at %lld", (long long)i);
        nchunks += (numels[i] + ADAM_CHUNK_ELEMS - 1) / ADAM_CHUNK_ELEMS;
        if (nchunks > INT32_MAX) return fail(MUON_EINVAL, "too many elements");
    }
    std::vector<AdamTensor> tens((size_t)count);
    std::vector<AdamChunk> chunks;
    chunks.reserve((size_t)nchunks);
    for (int64_t i = 0; i < count; ++i) {
        auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
        tens[(size_t)i] = AdamTensor{params[i], grads[i], exp_avg[i], exp_avg_sq[i],
                                     (a16(params[i]) && a16(grads[i]) && a16(exp_avg[i]) && a16(exp_avg_sq[i])) ? 1 : 0, 0};
        for (int64_t s0 = 0; s0 < numels[i]; s0 += ADAM_CHUNK_ELEMS)
            chunks.push_back(AdamChunk{s0, (int)i, (int)std::min<int64_t>(ADAM_CHUNK_ELEMS, numels[i] - s0)});
    }
    if (chunks.empty()) return MUON_OK;
    int r;
    DevCtx dc;
    if ((r = get_dev(dc))) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t tb = align_up(sizeof(AdamTensor) * tens.size(), 256);
    const size_t cb = align_up(sizeof(AdamChunk) * chunks.size(), 256);
    Workspace* w = nullptr;
    if ((r = ws_get(dc.device, s, tb + cb, &w))) return r;
    // both tables through the pinned staging ring, as one byte block (tb and cb
    // are multiples of 256, so the block is a whole number of ring rows)
    static_assert(256 % sizeof(MatEntry) == 0, "ring rows tile 256 bytes");
    std::vector<MatEntry> rows((tb + cb) / sizeof(MatEntry));
    std::memcpy(rows.data(), tens.data(), sizeof(AdamTensor) * tens.size());
    std::memcpy(reinterpret_cast<char*>(rows.data()) + tb, chunks.data(), sizeof(AdamChunk) * chunks.size());
    if ((r = upload_table(*w, rows, reinterpret_cast<MatEntry*>(w->base), s))) return r;
    AdamArgs a;
    a.tensors = reinterpret_cast<const AdamTensor*>(w->base);
    a.chunks = reinterpret_cast<const AdamChunk*>(w->base + tb);
    a.param_dtype = param_dtype;
    a.state_dtype = state_dtype;
    a.beta1 = beta1; a.beta2 = beta2; a.eps = eps;
    const double bc1 = 1.0 - std::pow((double)beta1, (double)step);
    const double bc2 = 1.0 - std::pow((double)beta2, (double)step);
    a.lr_wd = (float)((double)lr * (double)wd);
    a.step_size = (float)((double)lr / bc1);
    a.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
    double bytes = 0;
    for (int64_t i = 0; i < count; ++i) bytes += (double)numels[i] * (3.0 * esize(param_dtype) + 4.0 * esize(state_dtype));
    note_launch_begin(KC_ADAMW, s);
    cudaError_t e = launch_adamw(a, (int)chunks.size(), s);
    note_launch_end(KC_ADAMW, bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "adamw launch");
    return MUON_OK;
} MUON_CATCH_ALL
