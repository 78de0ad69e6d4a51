// Persistent groups (muon_group_*): the optimizer object of a training loop.

#include "host.h"

using namespace muon;

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
    // host I/O (muon_group_set_host_io), per entry in bucket order
    std::vector<size_t> entry_bytes;                // parameter bytes of the entry
    std::vector<int64_t> caller_index;              // the entry's index in the caller's arrays
    std::vector<const void*> host_g;                // pinned host gradients (empty: no copy in)
    std::vector<void*> host_p;                      // pinned host parameters (empty: no copy out)
    cudaStream_t io_in = nullptr, io_out = nullptr; // copy streams
    std::vector<cudaEvent_t> io_ev;                 // fork, join and two per unit of work
};

namespace muon {

// The step's units of work in launch order: each fused small-matrix launch
// (all matrices of its buckets), then every chunk of every other bucket.
// A unit is a list of entry ranges [first, first + count).
struct GroupUnit {
    int fused = -1;                                 // index into g->fused, or -1: bucket k, chunk at c0
    size_t k = 0;
    int64_t c0 = 0;
    int B = 0;
    std::vector<std::pair<int64_t, int64_t>> ranges;
};

static std::vector<GroupUnit> group_units(const muon_group* g) {
    std::vector<GroupUnit> units;
    for (size_t f = 0; f < g->fused.size(); ++f) {
        GroupUnit u;
        u.fused = (int)f;
        for (int k : g->fused[f].bks) u.ranges.push_back({g->bucket_first[(size_t)k], g->bucket_size[(size_t)k]});
        units.push_back(u);
    }
    for (size_t k = 0; k < g->keys.size(); ++k) {
        if (g->plans[k].fused) continue;
        const int64_t cnt = g->bucket_size[k];
        for (int64_t c0 = 0; c0 < cnt; c0 += g->chunks[k]) {
            GroupUnit u;
            u.k = k;
            u.c0 = c0;
            u.B = (int)std::min<int64_t>(g->chunks[k], cnt - c0);
            u.ranges.push_back({g->bucket_first[k] + c0, u.B});
            units.push_back(u);
        }
    }
    return units;
}

static int group_run_unit(muon_group* g, const GroupUnit& u, cudaStream_t s) {
    int r;
    if (u.fused >= 0) {
        const FusedLaunch& f = g->fused[(size_t)u.fused];
        const SmallArgs sa = fused_args(f, g->d_work, g->plans, g->keys, g->bucket_size, g->vec_ok,
                                        [&](int k) { return g->d_table + g->bucket_first[(size_t)k]; }, 0,
                                        g->param_dtype, g->mom_dtype, 0, 0.f, 0.f, 0.f, g->dc.status, g->d_hyper);
        return run_small(g->dc, s, sa, fused_flops(f, g->plans, g->keys, g->bucket_size));
    }
    const int m = g->keys[u.k].first, n = g->keys[u.k].second;
    const NsPlan& plan = g->plans[u.k];
    const float scale = 0.2f * std::sqrt((float)n);
    const ChunkLayout L = chunk_layout(m, n, u.B, g->ns_dtype, plan.fp32_tc);
    const MatEntry* dm = g->d_table + g->bucket_first[u.k] + u.c0;
    if ((r = run_prep(g->dc, s, g->cbase, L, m, n, u.B, dm, g->param_dtype, g->mom_dtype, g->ns_dtype, true, 0, 0.f,
                      g->vec_ok[u.k] != 0, g->pcnt, g->d_hyper)))
        return r;
    FinalEpi fin{EPI_UPDATE, dm, g->param_dtype, 0.f, 0.f, scale, g->d_hyper};
    return run_ns(g->dc, s, g->cbase, L, m, n, u.B, g->ns_dtype, plan, x_holds_u(g->ns_dtype), fin);
}

// Events the host I/O of a step needs (fork, join, two per unit), created
// outside any capture.
static int group_io_events(muon_group* g) {
    if (g->host_g.empty() && g->host_p.empty()) return MUON_OK;
    const size_t need = 2 + 2 * group_units(g).size();
    while (g->io_ev.size() < need) {
        cudaEvent_t e = nullptr;
        MUON_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        g->io_ev.push_back(e);
    }
    return MUON_OK;
}

// With host I/O, only the first unit's gradients and the last unit's
// parameters cross NVLink-C2C while no unit computes: the smallest unit (in
// parameter bytes) goes first and the next smallest last, the rest keep
// their order.  Units are independent, so the results do not change.
static void order_for_io(const muon_group* g, std::vector<GroupUnit>& units) {
    if (units.size() < 3) return;
    std::vector<size_t> bytes(units.size(), 0);
    for (size_t i = 0; i < units.size(); ++i)
        for (const auto& rg : units[i].ranges)
            for (int64_t e = rg.first; e < rg.first + rg.second; ++e) bytes[i] += g->entry_bytes[(size_t)e];
    std::vector<size_t> idx(units.size());
    for (size_t i = 0; i < idx.size(); ++i) idx[i] = i;
    std::stable_sort(idx.begin(), idx.end(), [&](size_t x, size_t y) { return bytes[x] < bytes[y]; });
    const size_t first = idx[0], last = idx[1];
    std::vector<GroupUnit> out;
    out.reserve(units.size());
    out.push_back(units[first]);
    for (size_t i = 0; i < units.size(); ++i)
        if (i != first && i != last) out.push_back(units[i]);
    out.push_back(units[last]);
    units.swap(out);
}

static int group_enqueue(muon_group* g, cudaStream_t s) {
    NvtxRange nvr("muon_group_step");
    int r;
    std::vector<GroupUnit> units = group_units(g);
    const bool cin = !g->host_g.empty(), cout = !g->host_p.empty();
    if (cin || cout) order_for_io(g, units);
    if (!cin && !cout) {
        for (const GroupUnit& u : units)
            if ((r = group_run_unit(g, u, s))) return r;
        return MUON_OK;
    }
    // host I/O: fork both copy streams off s; every gradient copy in launch
    // order on io_in (one event per unit); each unit waits for its own
    // gradients, and its parameters leave on io_out once it is done; both
    // streams join s at the end
    if (g->io_ev.size() < 2 + 2 * units.size()) return fail(MUON_EINVAL, "host I/O events missing");
    cudaEvent_t fork = g->io_ev[0], join = g->io_ev[1];
    MUON_CUDA(cudaEventRecord(fork, s));
    MUON_CUDA(cudaStreamWaitEvent(g->io_in, fork, 0));
    MUON_CUDA(cudaStreamWaitEvent(g->io_out, fork, 0));
    if (cin) {
        for (size_t i = 0; i < units.size(); ++i) {
            for (const auto& rg : units[i].ranges)
                for (int64_t e = rg.first; e < rg.first + rg.second; ++e)
                    MUON_CUDA(cudaMemcpyAsync(const_cast<void*>(g->entries[(size_t)e].grad), g->host_g[(size_t)e],
                                              g->entry_bytes[(size_t)e], cudaMemcpyHostToDevice, g->io_in));
            MUON_CUDA(cudaEventRecord(g->io_ev[2 + 2 * i], g->io_in));
        }
    }
    for (size_t i = 0; i < units.size(); ++i) {
        if (cin) MUON_CUDA(cudaStreamWaitEvent(s, g->io_ev[2 + 2 * i], 0));
        if ((r = group_run_unit(g, units[i], s))) return r;
        if (cout) {
            MUON_CUDA(cudaEventRecord(g->io_ev[3 + 2 * i], s));
            MUON_CUDA(cudaStreamWaitEvent(g->io_out, g->io_ev[3 + 2 * i], 0));
            for (const auto& rg : units[i].ranges)
                for (int64_t e = rg.first; e < rg.first + rg.second; ++e)
                    MUON_CUDA(cudaMemcpyAsync(g->host_p[(size_t)e], g->entries[(size_t)e].w, g->entry_bytes[(size_t)e],
                                              cudaMemcpyDeviceToHost, g->io_out));
        }
    }
    // join: io_in ended with the last unit's gradients (waited on by s when
    // copying in); io_out ends with the last unit's parameters
    MUON_CUDA(cudaEventRecord(join, g->io_out));
    MUON_CUDA(cudaStreamWaitEvent(s, join, 0));
    if (!cin) {
        MUON_CUDA(cudaEventRecord(g->io_ev[2], g->io_in));
        MUON_CUDA(cudaStreamWaitEvent(s, g->io_ev[2], 0));
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
        g->chunks[k] = budget_bytes_chunk(chunk_layout(m, n, 1, g->ns_dtype, g->plans[k].fp32_tc).total, cnt);
        chunk_need = std::max(chunk_need, chunk_layout(m, n, g->chunks[k], g->ns_dtype, g->plans[k].fp32_tc).total);
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
            g->entry_bytes.push_back((size_t)ms[i] * (size_t)ns[i] * esize(param_dtype));
            g->caller_index.push_back(i);
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
    if ((r = group_io_events(g))) return r;

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
    for (cudaEvent_t e : g->io_ev) cudaEventDestroy(e);
    if (g->io_in) cudaStreamDestroy(g->io_in);
    if (g->io_out) cudaStreamDestroy(g->io_out);
    if (g->cap) cudaStreamDestroy(g->cap);
    delete g;
    return MUON_OK;
}

int muon_group_set_host_io(muon_group* g, const void* const* host_grads, void* const* host_params) try {
    if (!g) return fail(MUON_EINVAL, "group is NULL");
    int dev = -1;
    MUON_CUDA(cudaGetDevice(&dev));
    if (dev != g->device) return fail(MUON_EINVAL, "group belongs to device %d, current device is %d", g->device, dev);
    auto pinned = [](const void* p) {
        cudaPointerAttributes a;
        if (!p || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        return a.type == cudaMemoryTypeHost;
    };
    std::vector<const void*> hg;
    std::vector<void*> hp;
    for (size_t e = 0; e < g->entries.size(); ++e) {
        const int64_t i = g->caller_index[e];
        if (host_grads) {
            if (!pinned(host_grads[i]))
                return fail(MUON_EINVAL, "host_grads[%lld] is NULL or not pinned host memory", (long long)i);
            hg.push_back(host_grads[i]);
        }
        if (host_params) {
            if (!pinned(host_params[i]))
                return fail(MUON_EINVAL, "host_params[%lld] is NULL or not pinned host memory", (long long)i);
            hp.push_back(host_params[i]);
        }
    }
    if ((host_grads || host_params) && !g->io_in) {
        MUON_CUDA(cudaStreamCreateWithFlags(&g->io_in, cudaStreamNonBlocking));
        MUON_CUDA(cudaStreamCreateWithFlags(&g->io_out, cudaStreamNonBlocking));
    }
    // steps already enqueued with the old buffers (on whatever streams the
    // caller stepped on) finish first
    MUON_CUDA(cudaDeviceSynchronize());
    g->host_g.swap(hg);
    g->host_p.swap(hp);
    group_drop_graph(g);        // the step's structure changed: capture it again
    return MUON_OK;
} MUON_CATCH_ALL

}  // extern "C"
