// Runtime of the Muon update library: logging and the C boundary's error
// handling, per-device state and its status word, the grow-only workspace
// per (device, stream) with its pinned table ring, launch accounting with
// optional per-launch event timing, and the diagnostics entry points.
#include "host.h"

namespace muon {

// Device allocations of the library's own storage (workspaces, counters,
// groups) go through here.  MUON_FAIL_ALLOC=1 makes every one of them fail, so
// that the allocation-failure paths can be exercised without exhausting a GPU.
cudaError_t dev_alloc(void** p, size_t bytes) {
    const char* f = std::getenv("MUON_FAIL_ALLOC");
    if (f && f[0] == '1') {
        *p = nullptr;
        return cudaErrorMemoryAllocation;
    }
    return cudaMalloc(p, bytes);
}

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

void logf(int lvl, const char* fmt, ...) {
    if (log_level() < lvl) return;
    va_list ap;
    va_start(ap, fmt);
    std::fprintf(stderr, "[muon] ");
    std::vfprintf(stderr, fmt, ap);
    std::fprintf(stderr, "\n");
    va_end(ap);
}

int fail(int status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    logf(1, "error %d: %s", status, buf);
    return status;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(MUON_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::mutex g_mu;                 // guards every global below
std::map<int, DevCtx> g_dev;

int get_dev(DevCtx& out) {
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

std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

int ws_get(int dev, cudaStream_t s, size_t need, Workspace** out) {
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
int prep_counters(int dev, cudaStream_t s, int B, int** out) {
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
int upload_table(Workspace& w, const std::vector<MatEntry>& h, MatEntry* d_dst, cudaStream_t s) {
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

std::atomic<int64_t> g_launches{0};
std::atomic<int> g_timing{0};

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


bool env_flag(const char* name, bool dflt) {
    const char* e = std::getenv(name);
    if (!e || !*e) return dflt;
    return !(e[0] == '0' || e[0] == 'n' || e[0] == 'N' || e[0] == 'f' || e[0] == 'F');
}

}  // namespace muon

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

}  // extern "C"
