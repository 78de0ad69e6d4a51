// Newton-Schulz orchestration of the Muon update: the NS configuration, the
// resolved plan of a shape, the product launches of plain and Gram NS with
// segment restarts ("MuonX" page, section 3.2), the momentum/norm prologue,
// and the entry points muon_ns_orthogonalize, muon_step, muon_ns_flops and
// muon_debug_gemm.  Matrices are bucketed by oriented shape ("DMuon" news
// page, section 3; summary, section 2.2 "batching").
#include "host.h"

namespace muon {

NsConfig g_cfg;
std::atomic<uint64_t> g_cfg_version{1};   // bumped when plans may change (config, tune cache)

int validate_segments(int steps, const int* segs, int nseg) {
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

// Precision of the bf16 path's m x m Gram-space matrices (G, P, PG, Q).
// A bit-faithful CPU simulation of the iteration against the exact one gives,
// for the Gram path with bf16 Gram space, 0.8-1.2% relative error on every
// shape with m >= 128 and n >= 2m, but 1.5-4% on square and near-square shapes
// and 2.3% for m = 37; with TF32 Gram space all of them stay at or below 1.5%.
// The plain path's error is set by the bf16 X (0.8-1.9% either way from 64
// rows up; below that up to 4%, so the automatic choice takes the Gram path
// there, see choose_plan), so it keeps bf16 Gram space.  TF32 costs twice the operand bytes and half the tensor rate on
// the m^3 products, so it is used only where bf16 is not accurate enough.
int gram_space_tf32(int path, int m, int n) {
    return (path == MUON_PATH_GRAM && (m < 128 || n < 2 * m)) ? 1 : 0;
}

NsPlan make_plan(const float coeffs[3], int steps, const std::vector<int>& gram_segs, int path, int tile_n,
                        int m, int n, int sym_tile_n, int sym_dense) {
    NsPlan p;
    p.sym_tile_n = sym_tile_n;
    p.sym_dense = sym_dense;
    p.gram_tf32 = gram_space_tf32(path, m, n);
    p.fused = 0;
    p.fp32_tc = 0;
    p.a = coeffs[0];
    p.b = coeffs[1];
    p.c = coeffs[2];
    p.path = path;
    p.tile_n = tile_n;
    if (path == MUON_PATH_GRAM && !gram_segs.empty()) p.segs = gram_segs;
    else p.segs.assign(steps, 1);
    return p;
}

GemmArgs gemm_base(int dtype, int* status) {
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
    // paired products as 4-CTA clusters sharing the A rows by multicast;
    // MUON_MC=0/1 overrides
    if (const char* f = std::getenv("MUON_MC")) a.mc = (f[0] == '1') ? 1 : 0;
    else a.mc = 0;
    a.status = status;
    a.b_kmajor = 1;
    return a;
}

// fp32 products on the TF32 tensor path as three passes (tf32x3.cu, the
// k-blocks accumulated in chunks added in round-to-nearest fp32) or on FFMA.
// MUON_FP32_TC=1 or 0 forces one; otherwise the tensor path takes buckets of
// at least 2^30 multiply-adds of X X^T (m^2 n per matrix, times the count).
// Measured (muon_ns_orthogonalize, best of plain and Gram, ms, FFMA against
// the tensor path): 640x2560 0.76 / 0.88, 512x2048 0.44 / 0.73, 256x1024 x 4
// 0.30 / 0.52 below the mark; 1024^2 0.95 / 0.85, 512^2 x 8 0.96 / 0.71,
// 256x1024 x 16 0.83 / 0.68, 768x3072 1.26 / 1.03, 2048x8192 12.9 / 3.3,
// 4096^2 29.5 / 9.8 at or above it.  With whole-K accumulation the tensor
// path missed the 1e-4 fp32 bar from about 768x3072 (its error grew with K);
// in chunks it holds at every size tested.
int fp32_tc_choice(int dtype, int m, int n, int64_t count) {
    if (dtype != MUON_F32) return 0;
    const char* f = std::getenv("MUON_FP32_TC");
    if (f && (f[0] == '0' || f[0] == '1')) return f[0] == '1' ? 1 : 0;
    return (double)m * m * (double)n * (double)count >= 1073741824.0 ? 1 : 0;
}

int run_gemm(const DevCtx& dc, cudaStream_t s, const GemmArgs& a, int kclass, int64_t work_k) {
    const double mnk = (double)a.M * a.N * (double)(work_k > 0 ? work_k : a.K) * a.batch;
    const double work = a.symmetric ? mnk : 2.0 * mnk;
    const bool tc = (is_half(a.dtype) || a.dtype == DT_TF32);
    const int kc = tc ? kclass : KC_SIMT;
    GemmArgs ga = a;
    if (tc) ga.stall = take_stall(STALL_PRODUCT);
    note_launch_begin(kc, s);
    cudaError_t e = tc ? launch_gemm_tc(ga, dc.sms, s) : launch_gemm_simt(a, dc.sms, s);
    note_launch_end(kc, work, s);
    if (e != cudaSuccess) return cuda_fail(e, "product launch");
    return MUON_OK;
}

// An fp32 product as one TF32 tensor-core product over K' = 3 Kp: A' = [hi |
// hi | lo] of A's rows, B' = [hi | lo | hi] of op(B)'s columns (tf32x3.cu),
// written to SA and SB; the epilogue is the fp32 product's own.
int run_gemm_tf32x3(const DevCtx& dc, cudaStream_t s, const GemmArgs& a, int kclass, float* SA, float* SB) {
    const int64_t Kp = pad4(a.K), K3 = 3 * Kp;
    SplitArgs sa;
    std::memset(&sa, 0, sizeof sa);
    sa.src = a.A; sa.ld_src = a.lda; sa.stride_src = a.strideA;
    sa.rows = a.M; sa.K = a.K; sa.Kp = Kp; sa.transposed = 0; sa.order = SPLIT_HHL;
    sa.dst = SA; sa.stride_dst = (int64_t)a.M * K3; sa.batch = a.batch;
    SplitArgs sb = sa;
    sb.src = a.B; sb.ld_src = a.ldb; sb.stride_src = a.strideB;
    sb.rows = a.N; sb.transposed = a.b_kmajor ? 0 : 1; sb.order = SPLIT_HLH;
    sb.dst = SB; sb.stride_dst = (int64_t)a.N * K3;
    for (const SplitArgs* sp : {&sa, &sb}) {
        note_launch_begin(KC_OTHER, s);
        cudaError_t e = launch_tf32_split(*sp, dc.sms, s);
        note_launch_end(KC_OTHER, 0.0, s);
        if (e != cudaSuccess) return cuda_fail(e, "operand split launch");
    }
    GemmArgs t = a;
    t.dtype = DT_TF32;
    t.A = SA; t.lda = K3; t.strideA = (int64_t)a.M * K3;
    t.B = SB; t.ldb = K3; t.strideB = (int64_t)a.N * K3; t.b_kmajor = 1;
    t.K = (int)K3;
    t.c_dtype = MUON_F32;
    t.round_tf32 = 0;
    // the tensor core's fp32 accumulation does not round to nearest: summed
    // over the whole tripled K its error grows with K (1.2e-4 relative for
    // K = 3 x 8192); chunk sums added in round-to-nearest fp32 bound it
    t.kchunk = TF32_KCHUNK;
    return run_gemm(dc, s, t, kclass, a.K);   // work counted on the fp32 product's K
}

// X is stored in the path's dtype; the m x m Gram-space matrices are fp32 on
// both paths (TF32-rounded on the bf16 path).
ChunkLayout chunk_layout(int m, int n, int B, int dtype, int fp32_tc) {
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
    L.tf32x3 = (dtype == MUON_F32 && fp32_tc) ? 1 : 0;
    L.off_SA = L.off_SB = 0;
    if (L.tf32x3) {
        // XX^T: m x 3 pad4(n) both; Gram-space products m x 3 pad4(m) both;
        // QX: A' m x 3 pad4(m), B' n x 3 pad4(m)
        const size_t pm = (size_t)pad4(m), pn = (size_t)pad4(n);
        const size_t sa = 3 * sizeof(float) * std::max((size_t)m * pn, (size_t)m * pm);
        const size_t sb = 3 * sizeof(float) * std::max({(size_t)m * pn, (size_t)m * pm, (size_t)n * pm});
        L.off_SA = take(sa * B);
        L.off_SB = take(sb * B);
    }
    L.total = o;
    return L;
}

// Runs NS on B oriented m x n matrices held (unnormalised when use_inv) in
// the chunk's X buffer, ending in `fin`.
//
// Precision of the bf16 path: X and the long products XX^T, QX are bf16 with
// fp32 accumulation; the m x m Gram-space matrices G, P, PG, Q are bf16, or,
// where gram_space_tf32() asks for it, TF32-rounded fp32 multiplied on the
// TF32 tensor path, with the transform applied to X rounded to bf16.
int run_ns(const DevCtx& dc, cudaStream_t s, char* base, const ChunkLayout& L, int m, int n, int B,
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

    // every product of the iteration; fp32 ones on the three-pass TF32 path
    // when the layout holds its split operands
    auto product = [&](const GemmArgs& g, int kclass) {
        if (L.tf32x3 && g.dtype == MUON_F32)
            return run_gemm_tf32x3(dc, s, g, kclass, reinterpret_cast<float*>(base + L.off_SA),
                                   reinterpret_cast<float*>(base + L.off_SB));
        return run_gemm(dc, s, g, kclass);
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
            int r = product(g, KC_SYRK);
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
                int r = product(g, KC_SQUARE);
                if (r) return r;
            }
            if (j == 1) {
                q = p;
            } else {
                const int qn = grab();     // Q <- P Q
                int r = product(sym(S[p], S[q], S[qn], j == Lseg), KC_SQUARE);
                if (r) return r;
                used[q] = false;
                q = qn;
            }
            if (j < Lseg) {
                const int t = grab();      // G <- (P G) P
                int r = product(sym(S[p], G, S[t], false), KC_SQUARE);
                if (r) return r;
                r = product(sym(S[t], S[p], G, false), KC_SQUARE);
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
        int r = product(g, kc);
        if (r) return r;
        std::swap(X, Xn);
    }
    return MUON_OK;
}

int run_prep(const DevCtx& dc, cudaStream_t s, char* base, const ChunkLayout& L, int m, int n, int B,
                    const MatEntry* d_mats, int in_dtype, int mom_dtype, int x_dtype, bool with_mom, int nesterov,
                    float beta, bool vec_ok, int* cnt, const float* hyper) {
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

int budget_bytes_chunk(size_t per_matrix, int count) {
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

}  // namespace muon

using namespace muon;

extern "C" {

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
    plan.fp32_tc = fp32_tc_choice(nsd, om, on, batch);
    const size_t per = chunk_layout(om, on, 1, nsd, plan.fp32_tc).total;
    const int chunk = budget_bytes_chunk(per, (int)std::min<int64_t>(batch, 65535));
    const size_t table_bytes = align_up(sizeof(MatEntry) * (size_t)batch, 256);
    const ChunkLayout L = chunk_layout(om, on, chunk, nsd, plan.fp32_tc);
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
        const ChunkLayout LB = chunk_layout(om, on, B, nsd, plan.fp32_tc);
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
        chunks[k] = budget_bytes_chunk(chunk_layout(m, n, 1, nsd, plans[k].fp32_tc).total, cnt);
        chunk_need = std::max(chunk_need, chunk_layout(m, n, chunks[k], nsd, plans[k].fp32_tc).total);
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
            const ChunkLayout L = chunk_layout(m, n, B, nsd, plans[k].fp32_tc);
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

int muon_debug_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K, int64_t batch,
                    int dtype, int b_kmajor, int symmetric, int poly, float alpha, float pa, float pb, float pc,
                    int tile_n, void* stream) try {
    if (!A || !B || !C) return fail(MUON_EINVAL, "NULL operand");
    if (M < 1 || N < 1 || K < 1 || batch < 1) return fail(MUON_EINVAL, "bad sizes");
    if (M > (1 << 20) || N > (1 << 20) || K > (1 << 20)) return fail(MUON_EINVAL, "size above 2^20");
    if (!valid_dtype(dtype) && dtype != DT_TF32 && dtype != DT_TF32_CHUNKED) return fail(MUON_EDTYPE, "dtype %d", dtype);
    const bool chunked = (dtype == DT_TF32_CHUNKED);
    if (chunked) dtype = DT_TF32;
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
    if (chunked) g.kchunk = TF32_KCHUNK;
    if (poly) {
        g.epi = EPI_POLY;
        g.Gin = A; g.ldg = K; g.strideG = M * K;
        g.pa = pa; g.pb = pb; g.pc = pc;
    }
    return run_gemm(dc, reinterpret_cast<cudaStream_t>(stream), g, KC_OTHER);
} MUON_CATCH_ALL

}  // extern "C"
