// Host side of an owner-centric multi-rank step ("DMuon" summary, sections
// 2.1 and 2.3): owner placement, the packed exchange layout, and the
// one-launch pack/unpack entry point.

#include "host.h"

using namespace muon;

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
