// Per-shape plans: the measured-cost autotune ("DMuon" news page, section 3;
// summary, sections 2.3-2.4: each distinct shape is timed once per candidate
// scheme and the fastest is cached and reused), its persistent cache, and the
// work lists of the fused small-matrix launches (summary, section 2.2).
#include "host.h"

namespace muon {

std::map<TuneKey, TuneEntry> g_tune;
std::map<std::tuple<int64_t, int64_t, int>, int> g_last_path;     // oriented m, n, dtype -> path

static int cudart_version() {
    int v = 0;
    cudaRuntimeGetVersion(&v);
    return v;
}

TuneKey tune_key(const DevCtx& dc, int64_t m, int64_t n, int dtype) {
    return TuneKey{dc.name, dc.sms, cudart_version(), m, n, dtype};
}

// Whether the one-CTA-per-matrix kernel can run this plan (bf16, m <= 128,
// n <= 512, segments of length <= 2, bf16 Gram space).  MUON_SMALL=0 turns it off.
bool small_eligible(const NsPlan& p, int m, int n, int dtype) {
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

SmallBucket small_bucket(const NsPlan& p, const MatEntry* mats, int B, int m, int n, bool vec_ok) {
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
SmallArgs small_args(const NsPlan& p, const MatEntry* mats, int B, int m, int n, int mode, int param_dtype,
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

SmallWork small_work(const std::vector<int>& counts, const std::vector<double>& costs, int sms) {
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
double plan_alg_flops(const NsPlan& p, int m, int n) {
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

int run_small(const DevCtx& dc, cudaStream_t s, const SmallArgs& a, double alg_flops) {
    NvtxRange nvr("fused small-matrix launch");
    SmallArgs sa = a;
    sa.stall = take_stall(STALL_SMALL);
    note_launch_begin(KC_SMALL, s);
    cudaError_t e = launch_small_ns(sa, dc.sms, s);
    note_launch_end(KC_SMALL, alg_flops, s);
    if (e != cudaSuccess) return cuda_fail(e, "fused small-matrix launch");
    return MUON_OK;
}

std::vector<FusedLaunch> plan_fused(const DevCtx& dc, const std::vector<NsPlan>& plans,
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
void pack_fused(const std::vector<FusedLaunch>& fl, char* block) {
    for (const auto& f : fl) {
        int* p = reinterpret_cast<int*>(block + f.off);
        std::memcpy(p, f.work.ptr.data(), sizeof(int) * f.work.ptr.size());
        std::memcpy(p + f.work.ptr.size(), f.work.items.data(), sizeof(int) * f.work.items.size());
    }
}

double fused_flops(const FusedLaunch& f, const std::vector<NsPlan>& plans,
                          const std::vector<std::pair<int, int>>& keys, const std::vector<int64_t>& counts) {
    double t = 0.0;
    for (int k : f.bks)
        t += plan_alg_flops(plans[(size_t)k], keys[(size_t)k].first, keys[(size_t)k].second) * (double)counts[(size_t)k];
    return t;
}

int autotune_shape(const DevCtx& dc, cudaStream_t s, int m, int n, int dtype, int B, const NsConfig& cfg,
                          TuneEntry* out) {
    const int ftc = fp32_tc_choice(dtype, m, n, B);
    const ChunkLayout L = chunk_layout(m, n, B, dtype, ftc);
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
int choose_plan(const DevCtx& dc, cudaStream_t s, int m, int n, int dtype, int bucket_count,
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
        // accuracy before speed: with bf16 X and fewer than 64 rows the plain
        // iteration (five bf16 transforms of X) errs by up to 2-4 % against
        // the fp64 result (m = 3-5 and m = 32: a CPU simulation of the
        // kernels' roundings, and 3.8-4.1 % measured for 4 x 549 and
        // 4 x 168), the Gram path by at most 1.9 % over the same shapes; fp16
        // (ten mantissa bits) stays below 1 % either way
        if (dtype == MUON_BF16 && m < 64 && !cfg.segments.empty()) path = MUON_PATH_GRAM;
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
    plan->fp32_tc = fp32_tc_choice(dtype, m, n, bucket_count);
    return MUON_OK;
}

int save_tune_file(const char* path) {
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

}  // namespace muon

using namespace muon;

extern "C" {

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

}  // extern "C"
