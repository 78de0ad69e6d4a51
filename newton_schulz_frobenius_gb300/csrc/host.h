// Host-side declarations shared by the library's host translation units
// (runtime.cu, ns.cu, plan.cu, group.cu, noalloc.cu, owner.cu, adamw.cu):
// logging and status helpers, per-device state, the workspace, the NS plan
// and its orchestration, and the tuned per-shape plans.
#pragma once

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
#include <mutex>
#include <new>
#include <queue>
#include <sstream>
#include <stdexcept>
#include <string>
#include <tuple>
#include <vector>

namespace muon {

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

// NVTX ranges around the host steps (a step, a bucket, its prologue and NS
// run, the fused small-matrix launches): free when no tool is attached.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

struct DevCtx {
    int device = -1;
    int sms = 0;
    int major = 0, minor = 0;
    std::string name;
    int* status = nullptr;     // device status word
};

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

struct NsConfig {
    float coeffs[3] = {3.4445f, -4.7750f, 2.0315f};
    int steps = 5;
    std::vector<int> segments{2, 2, 1};
    int path = MUON_PATH_AUTO;
    int ns_precision = -1;      // 16-bit parameters: -1 follow them, or MUON_BF16 / MUON_F16
};

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
    int fp32_tc;    // fp32 path: products as three TF32 tensor-core passes (else FFMA)
};

// Workspace of one chunk of B matrices of oriented shape m x n.
struct ChunkLayout {
    int64_t ldx, ldm;
    size_t x_bytes, m_bytes;            // one matrix
    size_t off_X, off_X2, off_G, off_S[3], off_inv, off_part, total;
    size_t off_SA, off_SB;              // fp32 on the TF32 tensor path: split operands
    int tf32x3;                         // fp32 products as three TF32 passes (else FFMA)
    int nparts;
};

// Final epilogue of an NS run.
struct FinalEpi {
    int kind;               // EPI_UPDATE, EPI_OUT or EPI_STORE (autotune: into the workspace)
    const MatEntry* mats;   // device table (UPDATE / OUT)
    int out_dtype;
    float lr, wd, scale;
    const float* hyper = nullptr;   // device {lr, beta, wd, nesterov} read at run time, if set
};

struct TuneEntry {
    int path;
    int tile_n;
    double ms_per_matrix;
    int fused;
    int sym_tile_n;
    int sym_dense;
};

using TuneKey = std::tuple<std::string, int, int, int64_t, int64_t, int>;   // device, sms, cudart, m, n, dtype

// Work lists of one fused launch over several buckets: every matrix is an
// item of its bucket's cost; items go, most expensive first, to the CTA with
// the least work so far (longest processing time first), which balances
// buckets whose matrix counts are not multiples of the SM count.  Output:
// grid, per-CTA offsets ptr[grid + 1] and items (bucket << 24 | index).
struct SmallWork {
    int grid = 0;
    std::vector<int> ptr, items;
};

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

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline size_t esize(int dtype) { return is_half(dtype) ? 2 : 4; }
// Whether X holds the unscaled U (the 1 / ||U|| scale folded into the first
// products) or U already divided by its norm (the fp16 path).
inline bool x_holds_u(int x_dtype) { return x_dtype != MUON_F16; }
inline int64_t pad8(int64_t x) { return (x + 7) / 8 * 8; }
inline int64_t pad4(int64_t x) { return (x + 3) / 4 * 4; }
inline bool valid_dtype(int d) { return d == MUON_F32 || d == MUON_BF16 || d == MUON_F16; }
// Working precision of NS for parameters of this storage type: fp32 stays
// fp32; 16-bit parameters use the configured 16-bit type, by default their own.
inline int ns_dtype(int param_dtype, const NsConfig& cfg) {
    if (!is_half(param_dtype)) return MUON_F32;
    return cfg.ns_precision < 0 ? param_dtype : cfg.ns_precision;
}

// launch accounting: kernels launched, per-launch event timing on or off
extern std::atomic<int64_t> g_launches;
extern std::atomic<int> g_timing;

// state shared between the translation units, guarded by g_mu
extern std::mutex g_mu;
extern NsConfig g_cfg;
extern std::atomic<uint64_t> g_cfg_version;   // bumped when plans may change (config, tune cache)
extern std::map<TuneKey, TuneEntry> g_tune;
extern std::map<std::tuple<int64_t, int64_t, int>, int> g_last_path;     // oriented m, n, dtype -> path

cudaError_t dev_alloc(void** p, size_t bytes);
void logf(int lvl, const char* fmt, ...);
int fail(int status, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);
int get_dev(DevCtx& out);
int ws_get(int dev, cudaStream_t s, size_t need, Workspace** out);
int prep_counters(int dev, cudaStream_t s, int B, int** out);
int upload_table(Workspace& w, const std::vector<MatEntry>& h, MatEntry* d_dst, cudaStream_t s);
bool env_flag(const char* name, bool dflt);
int validate_segments(int steps, const int* segs, int nseg);
int gram_space_tf32(int path, int m, int n);
NsPlan make_plan(const float coeffs[3], int steps, const std::vector<int>& gram_segs, int path, int tile_n,
                 int m, int n, int sym_tile_n = 128, int sym_dense = 0);
GemmArgs gemm_base(int dtype, int* status);
// work_k: the contraction length the recorded work counts (0: a.K)
int run_gemm(const DevCtx& dc, cudaStream_t s, const GemmArgs& a, int kclass, int64_t work_k = 0);
// fp32_tc: the fp32 path's products as three TF32 passes (the layout then
// holds their split operands); ignored for 16-bit dtypes
ChunkLayout chunk_layout(int m, int n, int B, int dtype, int fp32_tc = 0);
// Whether fp32 products of `count` oriented m x n matrices run as three TF32
// passes (MUON_FP32_TC=1; else FFMA).
int fp32_tc_choice(int dtype, int m, int n, int64_t count);
int run_ns(const DevCtx& dc, cudaStream_t s, char* base, const ChunkLayout& L, int m, int n, int B,
           int dtype, const NsPlan& plan, bool use_inv, const FinalEpi& fin);
int run_prep(const DevCtx& dc, cudaStream_t s, char* base, const ChunkLayout& L, int m, int n, int B,
             const MatEntry* d_mats, int in_dtype, int mom_dtype, int x_dtype, bool with_mom, int nesterov,
             float beta, bool vec_ok, int* cnt, const float* hyper = nullptr);
int budget_bytes_chunk(size_t per_matrix, int count);
TuneKey tune_key(const DevCtx& dc, int64_t m, int64_t n, int dtype);
bool small_eligible(const NsPlan& p, int m, int n, int dtype);
SmallBucket small_bucket(const NsPlan& p, const MatEntry* mats, int B, int m, int n, bool vec_ok);
SmallArgs small_args(const NsPlan& p, const MatEntry* mats, int B, int m, int n, int mode, int param_dtype,
                     int mom_dtype, int nesterov, float beta, float lr, float wd, bool vec_ok, int* status);
SmallWork small_work(const std::vector<int>& counts, const std::vector<double>& costs, int sms);
double plan_alg_flops(const NsPlan& p, int m, int n);
int run_small(const DevCtx& dc, cudaStream_t s, const SmallArgs& a, double alg_flops);
std::vector<FusedLaunch> plan_fused(const DevCtx& dc, const std::vector<NsPlan>& plans,
                                    const std::vector<std::pair<int, int>>& keys,
                                    const std::vector<int64_t>& counts, int nsd, size_t* total_bytes);
void pack_fused(const std::vector<FusedLaunch>& fl, char* block);
double fused_flops(const FusedLaunch& f, const std::vector<NsPlan>& plans,
                   const std::vector<std::pair<int, int>>& keys, const std::vector<int64_t>& counts);
int autotune_shape(const DevCtx& dc, cudaStream_t s, int m, int n, int dtype, int B, const NsConfig& cfg,
                   TuneEntry* out);
int choose_plan(const DevCtx& dc, cudaStream_t s, int m, int n, int dtype, int bucket_count,
                const NsConfig& cfg, NsPlan* plan);
int save_tune_file(const char* path);

// Arguments of fused launch `f`; mats_of(k) gives bucket k's device table.
template <typename MatsOf>
SmallArgs fused_args(const FusedLaunch& f, const char* d_block, const std::vector<NsPlan>& plans,
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

}  // namespace muon
