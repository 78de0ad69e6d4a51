// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/muon.h"

namespace muon {

// Internal storage/arithmetic code next to MUON_F32, MUON_BF16 and MUON_F16:
// fp32 storage whose values are consumed by the tensor cores as TF32 (10-bit
// mantissa).  The bf16 path keeps some m x m Gram-space matrices in this form.
constexpr int DT_TF32 = 3;
// debug product code: TF32 with chunked accumulation (TF32_KCHUNK k-blocks of
// 32 elements per chunk, chunk sums added in round-to-nearest fp32)
constexpr int DT_TF32_CHUNKED = 4;
constexpr int TF32_KCHUNK = 32;

// 16-bit storage that the kind::f16 tensor-core products take (bf16 or fp16).
__host__ __device__ constexpr bool is_half(int dtype) { return dtype == MUON_BF16 || dtype == MUON_F16; }

// Bits of the per-device status word (read by muon_sync_status).
enum : int { STATUS_NONFINITE = 1, STATUS_TIMEOUT = 2 };

// A bounded wait gives up after this long (nanoseconds of %globaltimer); no
// legitimate wait inside one of the library's kernels comes near it.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;

// One matrix of a pointer-table launch (momentum kernel, fused update, output).
// Oriented shape is m x n (m <= n); trans = 1 means the caller's matrix is
// n x m and the oriented matrix is its transpose.
struct MatEntry {
    const void* grad;   // caller gradient (param dtype) or NS input
    void* mom;          // caller momentum (mom dtype), may be null
    void* w;            // caller weights (update) or NS output
    int trans;
    int pad;
};

enum EpiKind : int {
    EPI_STORE = 0,   // C = alpha * acc
    EPI_POLY = 1,    // C = pa*I + pb*Gin + pc*alpha*acc   (symmetric only)
    EPI_UPDATE = 2,  // W = W (1 - lr wd) - lr * scale * alpha * acc   (via mats)
    EPI_OUT = 3      // O = alpha * acc written to the caller's buffer (via mats)
};

// One (batched) product C[b] = epilogue(A[b] * op(B[b])).
// A is M x K row-major (K contiguous).  b_kmajor: B stored N x K (op = ^T);
// otherwise B stored K x N (op = identity).  dtype is the operand type of A, B
// and Gin (MUON_BF16, MUON_F32 on the FFMA path, or DT_TF32); c_dtype is the
// storage type of C (MUON_BF16 or MUON_F32); round_tf32 rounds fp32 results to
// the nearest TF32 value (ties to even) before they are stored.
struct GemmArgs {
    const void* A; int64_t lda; int64_t strideA;
    const void* B; int64_t ldb; int64_t strideB;
    int b_kmajor;
    int M, N, K, batch;
    int symmetric;          // M == N, lower-triangle tiles only, mirrored store
    int dtype;
    int c_dtype;
    int round_tf32;
    int epi;
    float alpha;            // scalar factor
    const float* alpha_vec; // optional per-batch factor (device), may be null
    int alpha_sq;           // use alpha_vec[b]^2
    void* C; int64_t ldc; int64_t strideC;
    const void* Gin; int64_t ldg; int64_t strideG;
    float pa, pb, pc;
    const MatEntry* mats;   // device table indexed by b (EPI_UPDATE / EPI_OUT)
    int out_dtype;          // storage type of the caller's W / O
    float lr, wd, scale;
    int tile_n;             // tensor-core tile N extent (128 or 256)
    int pair;               // tile_n 256 as 2-SM products on 2-CTA clusters: 0 off, otherwise on
    int mc;                 // paired launches as 4-CTA clusters of two pairs sharing A by TMA multicast
    int tma_c;              // set by the launcher: 16-bit workspace output written by tile stores
    int* status;            // device status word
    const float* hyper;     // optional device block {lr, beta, wd, nesterov}: overrides lr, wd
    int stall;              // test hook: k + 1 = CTA 0 leaves k-block k of its first tile unfilled; 0 = off
    int kchunk;             // TF32: k-blocks per accumulation chunk (sums added in round-to-nearest fp32); 0 = whole K
};

// Launchers (return the CUDA error of the launch).
cudaError_t launch_gemm_tc(const GemmArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_gemm_simt(const GemmArgs& a, int num_sms, cudaStream_t s);
int simt_split(int64_t tiles, int K, int num_sms);

// fp32 operand split for three-pass TF32 products (tf32x3.cu): per batch
// index, dst row r = [hi | hi | lo] (SPLIT_HHL) or [hi | lo | hi] (SPLIT_HLH)
// of source row r, each third Kp >= K wide (Kp % 4 == 0, zero beyond K).
// transposed: the source is K x rows with rows contiguous (leading dim ld_src).
enum SplitOrder : int { SPLIT_HHL = 0, SPLIT_HLH = 1 };
struct SplitArgs {
    const void* src; int64_t ld_src; int64_t stride_src;
    int rows, K;
    int64_t Kp;
    int transposed;
    int order;
    float* dst; int64_t stride_dst;   // rows x 3 Kp per batch index
    int batch;
};
cudaError_t launch_tf32_split(const SplitArgs& p, int num_sms, cudaStream_t s);

// Momentum (+Nesterov) or plain copy, orientation and Frobenius partial sums.
struct PrepArgs {
    const MatEntry* mats;   // device table, one entry per batch index
    int m, n, batch;        // oriented shape
    int in_dtype;           // dtype of grad (or NS input)
    int mom_dtype;
    int x_dtype;            // workspace X dtype
    int with_momentum;      // 0: U = input (NS only)
    int nesterov;
    float beta;
    void* X; int64_t ldx; int64_t strideX;
    float* partials;        // [batch][nparts]
    int nparts;             // CTAs per matrix (the grid's x), each writing one partial
    int vec_ok;             // caller rows are 16-byte aligned for vector access
    const float* hyper;     // optional device block {lr, beta, wd, nesterov}: overrides beta, nesterov
    int write_x;            // store U (times x_scale) into X
    int write_mom;          // store M' (0: a first pass that only sums U^2)
    const float* x_scale;   // optional per-matrix factor applied to U before it is stored
    // Optional in-kernel finalisation: per-matrix arrival counters (zero
    // before the launch, zero again after it); the last CTA of matrix b
    // writes inv[b] = 1/(||U||_F + eps) and flags a non-finite sum in status.
    int* counter;
    float* inv;
    float eps;
    int* status;
};
int prep_num_parts(int m, int n);              // 64 x 64 tiles of one matrix (partials capacity)
int prep_grid_parts(int m, int n, int batch);   // CTAs (partials) per matrix of one launch
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);

// Whole update of small matrices, one CTA per matrix (see small_ns.cu): the
// oriented shapes of up to SMALL_MAX_BUCKETS buckets in one launch, each
// bucket m <= 128 with n <= 512 (segments of length 1 or 2), or plain NS with
// 128 < m <= n <= 256; bf16 parameters.
constexpr int SMALL_MAX_BUCKETS = 8;
struct SmallBucket {
    const MatEntry* mats;   // device table, one entry per matrix of the bucket
    int batch, m, n;        // oriented shape
    int nseg;
    int segs[8];
    int vec_ok;             // caller rows 16-byte aligned, 8-element multiples
    float scale;            // shape scale of the update, 0.2 sqrt(n)
};
struct SmallArgs {
    int nb;
    SmallBucket bk[SMALL_MAX_BUCKETS];
    // Work order: null: one bucket, CTA c takes matrices c, c + grid, ...;
    // else CTA c takes items[cta_ptr[c] .. cta_ptr[c+1]), item = bucket << 24 | index
    const int* cta_ptr;
    const int* items;
    int grid;               // CTAs of the launch (with a work list: its CTA count)
    int mode;               // 0: Muon step (momentum + fused update), 1: write O
    int param_dtype;        // MUON_BF16
    int mom_dtype;
    int nesterov;
    float beta, lr, wd;
    float a, b, c;
    int* status;
    const float* hyper;     // optional device block {lr, beta, wd, nesterov}
    int stall;              // test hook: k + 1 = CTA 0 issues no copy for its prologue piece k; 0 = off
};
bool small_ns_fits(int m, int n, int nseg, const int* segs);
cudaError_t launch_small_ns(const SmallArgs& a, int num_sms, cudaStream_t s);

// AdamW over many tensors in one launch (adamw.cu).
constexpr int ADAM_CHUNK_ELEMS = 8192;
struct AdamTensor {
    void* p;
    const void* g;
    void* m;
    void* v;
    int vec_ok;             // all four pointers 16-byte aligned
    int pad;
};
struct AdamChunk {
    int64_t start;          // first element of the chunk within its tensor
    int tensor;
    int len;
};
struct AdamArgs {
    const AdamTensor* tensors;
    const AdamChunk* chunks;
    int param_dtype, state_dtype;
    float beta1, beta2, eps;
    float lr_wd;            // lr * wd
    float step_size;        // lr / (1 - beta1^t)
    float inv_sqrt_bc2;     // 1 / sqrt(1 - beta2^t)
};
cudaError_t launch_adamw(const AdamArgs& a, int nchunks, cudaStream_t s);

// Packed exchange buffers (see pack.cu): chunk k moves elements
// [start, start + len) of matrix `mat` between the caller's storage and the
// packed buffer at element offset mats[mat].off + start.
constexpr int PACK_CHUNK_ELEMS = 32768;
struct PackMat {
    void* p;                // caller storage, row-major
    int64_t off;            // element offset in the packed buffer
    int vec_ok;             // both sides 16-byte aligned at every chunk start
    int pad;
};
struct PackChunk {
    int64_t start;
    int mat;
    int len;
};
struct PackArgs {
    const PackMat* mats;
    const PackChunk* chunks;
    void* packed;
    int esize;              // bytes per element
    int to_packed;          // 1: matrices -> packed buffer, 0: packed buffer -> matrices
};
cudaError_t launch_pack(const PackArgs& a, int nchunks, cudaStream_t s);

// Fills `count` elements of a workspace buffer with bounded pseudo-random values
// (autotune input only; never touches caller data).
cudaError_t launch_fill_synthetic(void* X, int64_t count, int dtype, float scale,
                                  uint32_t seed, cudaStream_t s);

// Programmatic dependent launch: a kernel launched this way may start (and run
// its set-up: barrier init, TMEM allocation, tensor-map prefetch) while the
// previous kernel on the stream finishes.  Every library kernel executes
// pdl_wait() before it reads anything another kernel produced and
// pdl_trigger() only after that, so a dependent grid launches only once all
// CTAs of its predecessor are resident or done.  MUON_PDL=0 turns it off.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Kernel-class bookkeeping for launch counting and optional event timing.
enum KernelClass : int {
    KC_PREP = 0, KC_NORM = 1 /* no longer launched: prep finalises */, KC_SYRK = 2, KC_SQUARE = 3, KC_APPLY = 4,
    KC_APPLY_UPDATE = 5, KC_SIMT = 6, KC_OTHER = 7, KC_SMALL = 8, KC_ADAMW = 9, KC_PACK = 10, KC_COUNT = 11
};
void note_launch_begin(int kclass, cudaStream_t s);
void note_launch_end(int kclass, double work, cudaStream_t s);

// Test hook of the bounded waits (muon_debug_arm_stall): the stage to leave
// unfilled (+1) in the next launch of the given kernel kind, consumed by that
// launch; 0 when nothing is armed.
enum StallKind : int { STALL_NONE = 0, STALL_PRODUCT = 1, STALL_SMALL = 2 };
int take_stall(int kind);

}  // namespace muon
