/*
 * muon.h -- C ABI of the GB300 (sm_103a) Muon update library.
 *
 * One Muon update of a 2-D weight matrix W with gradient G and momentum M is
 *
 *   M' = beta M + G;   U = G + beta M' (Nesterov) or U = M'
 *   X0 = U / (||U||_F + 1e-7)                       (oriented so rows <= cols)
 *   O  = NS(X0)                                     (plain or Gram Newton-Schulz)
 *   W' = W (1 - lr wd) - lr * 0.2 * sqrt(max(rows, cols)) * O
 *
 * Sources (page title, section):
 *   "MuonX: DMuon 调整多卡分工, Gram NS 降低计算量" (CSDN), section 2: momentum
 *     smooths the gradient, Newton-Schulz orthogonalises it; section 3.2
 *     "Gram NS": iterate on the Gram matrix XX^T, accumulate the transform,
 *     apply it to the long matrix only at segment boundaries, 2+2+1 segments.
 *   "DMuon: Efficient Distributed Muon Training with Near-Adam Overhead"
 *     (gist.science summary), section 2.2: Gram recursion for m < n, SYRK-style
 *     symmetric products, batching of same-shape matrices; section 2.3-2.4:
 *     per-shape measured cost, cached tuned kernel choice.
 * The pages give neither the momentum rule, the NS polynomial, eps nor the
 * update; the plain readings above are used (quintic coefficients
 * (3.4445, -4.7750, 2.0315), 5 steps, sum-form Nesterov, decoupled decay).
 *
 * Conventions for every entry point
 *   - Matrices are caller-owned DEVICE memory, row-major and contiguous.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     All GPU work is enqueued on it; calls return once it is enqueued.
 *   - Host-detectable errors return a negative muon_status and enqueue nothing.
 *     Device-detected errors (non-finite norm, a bounded wait that gave up) are
 *     recorded in a per-device status word read by muon_sync_status().
 *   - No C++ exception crosses the ABI; no call aborts the process.  A failed
 *     host allocation (tables sized by the arguments) returns MUON_ENOMEM.
 *   - The library keeps a workspace per (device, stream) that only grows; the
 *     first call of a new shape set may allocate and therefore must not be made
 *     while the stream is being captured into a CUDA graph.
 *   - Host threads may call the library concurrently on different streams.
 *     Calls on one stream from several host threads must be serialised by the
 *     caller (a growing workspace is freed once the stream drains, while
 *     another thread's call on that stream may still be using it).
 *   - There is no CPU fallback: every step runs in the library's CUDA kernels.
 */
#ifndef MUON_GB300_H
#define MUON_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MUON_OK = 0,
    MUON_EINVAL = -1,      /* bad pointer, size, segment list or hyper-parameter */
    MUON_EDTYPE = -2,      /* dtype not in muon_dtype or not supported for this call */
    MUON_ENOMEM = -3,      /* workspace allocation failed */
    MUON_ECUDA = -4,       /* a CUDA runtime/driver call failed (no device, launch error) */
    MUON_ENONFINITE = -5,  /* device saw a non-finite Frobenius norm */
    MUON_ETIMEOUT = -6,    /* a kernel's bounded wait gave up */
    MUON_ENOTSUP = -7      /* no sm_103a device / feature unavailable */
} muon_status;

/* Storage types.  MUON_F16 (IEEE binary16) is the working type of the
 * open-source Gram NS the "MuonX" page (section 3.2) mentions, which splits the
 * five steps into segments of 2 and 3; MuonX itself keeps bf16 with 2+2+1.
 * Both are reachable: the segment list through muon_set_ns_config, the
 * working type through the storage type or muon_set_ns_precision. */
typedef enum { MUON_F32 = 0, MUON_BF16 = 1, MUON_F16 = 2 } muon_dtype;

typedef enum { MUON_PATH_AUTO = 0, MUON_PATH_PLAIN = 1, MUON_PATH_GRAM = 2 } muon_path;

/*
 * Newton-Schulz orthogonalisation in place ("MuonX" page, section 3.2; "DMuon"
 * summary, section 2.2).
 *   ptr        device pointer to `batch` matrices of m x n, stride m*n elements.
 *              Read as the NS input U, overwritten with O = NS(U/(||U||_F+eps)).
 *              Each matrix is normalised on its own.  A matrix with m > n is
 *              processed as its transpose; the result is written back untransposed.
 *   dtype      storage type of the matrices: MUON_F32 (fp32 path: fp32 FFMA
 *              products, or, from 2^30 multiply-adds of X X^T per call (m^2 n
 *              times batch), three TF32 tensor-core passes per product with K
 *              accumulated in chunks added in round-to-nearest fp32; the
 *              environment's MUON_FP32_TC=1 or 0 forces one),
 *              MUON_BF16 or MUON_F16 (16-bit tensor-core products,
 *              fp32 accumulation, 16-bit intermediates of the NS precision:
 *              the storage type unless muon_set_ns_precision chose the other).
 *   coeffs     (a, b, c) of one NS step X <- aX + (bA + cA^2)X, A = XX^T.
 *   steps      number of NS steps (>= 1).
 *   segments   NULL or num_segments == 0: plain NS.  Otherwise Gram NS with
 *              these segment lengths (each >= 1, sum == steps): per segment
 *              G = XX^T, then P = aI + bG + cG^2, Q <- P (first) or PQ,
 *              G <- PGP (not after the last), then X <- QX.
 * Returns MUON_EINVAL for NULL ptr, m/n/batch < 1, a side above 2^20, a batch
 * above 2^31 - 1 or whose byte range overflows, steps < 1 or bad segments.
 */
int muon_ns_orthogonalize(void* ptr, int64_t m, int64_t n, int64_t batch, int dtype,
                          const float coeffs[3], int steps, const int* segments,
                          int num_segments, void* stream);

/*
 * muon_ns_orthogonalize for callers that must not allocate device memory.
 * The pages have no counterpart: this entry point exists for code that runs
 * where device memory belongs to someone else's allocator (a framework's
 * caching pool, a fixed per-job memory budget) or where allocation after
 * start-up is forbidden (a real-time training loop).  It computes the same
 * result with the same arguments and conventions as muon_ns_orthogonalize,
 * but inside one fixed 64 MiB array compiled into the library (every GPU that
 * loads the library holds it until the process exits) and it calls no
 * cudaMalloc, cudaFree, cudaMallocHost or other allocating routine.
 *   - The status word, the matrix table and the NS buffers of the whole batch
 *     must fit in the 64 MiB: one 1024 x 4096 bf16 matrix, 31 of 256 x 1024
 *     bf16, 127 of 128 x 512 bf16 (2048 x 2048 does not fit); batch at most
 *     65535.  A call that does not fit returns
 *     MUON_EINVAL (see muon_last_error_message) and enqueues nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call reuses the same array, which keeps the last call's contents;
 *     calls that overlap on the GPU (two streams, or two host threads) race.
 *     Each call first clears, on `stream`, the counters it relies on, so a
 *     call that follows a race starts clean.
 *   - Device-detected errors (a non-finite norm, a bounded wait that gave
 *     up) accumulate in a status word inside the array, not in the one
 *     muon_sync_status reads: read and clear them with
 *     muon_noalloc_sync_status.  A non-finite input gives a non-finite output.
 *   - With muon_set_kernel_timing(1) the timing records create CUDA events.
 */
int muon_ns_orthogonalize_noalloc(void* ptr, int64_t m, int64_t n, int64_t batch, int dtype,
                                  const float coeffs[3], int steps, const int* segments,
                                  int num_segments, void* stream);

/* Companion of muon_ns_orthogonalize_noalloc, equally free of allocation:
 * synchronise `stream`, then read and clear the status word inside the fixed
 * array on the current device: MUON_OK, MUON_ENONFINITE or MUON_ETIMEOUT for
 * the no-alloc calls since the last read (MUON_ECUDA if the sync failed).
 * The first call on a device looks up the array's address, like the first
 * muon_ns_orthogonalize_noalloc. */
int muon_noalloc_sync_status(void* stream);

/*
 * One Muon step over `count` matrices (the optimizer call the pages' drop-in
 * API names the participating matrices for: "DMuon" news page, section 3;
 * "MuonX" page, section 3.3).
 *   params[i]  device pointer, ms[i] x ns[i] weights, updated in place (param_dtype).
 *   grads[i]   device pointer, same shape, read only (param_dtype).
 *   moms[i]    device pointer, same shape, momentum updated in place (mom_dtype).
 *   lr, beta, wd, nesterov   hyper-parameters of the update above.
 * Matrices are bucketed by oriented shape; each bucket runs the NS path chosen
 * by muon_set_ns_config (auto: measured-cost autotune per shape, cached).
 * param_dtype MUON_F32 selects the fp32 path, MUON_BF16 or MUON_F16 the
 * tensor-core path (NS in the precision muon_set_ns_precision selects, by
 * default the parameters' own); mom_dtype may be any of the three.  Arrays are
 * host arrays of length `count`.
 */
int muon_step(void* const* params, const void* const* grads, void* const* moms,
              const int64_t* ms, const int64_t* ns, int64_t count,
              int param_dtype, int mom_dtype, float lr, float beta, float wd,
              int nesterov, void* stream);

/*
 * Persistent groups: the optimizer object of a training loop.  The caller
 * registers a fixed set of matrices once (same arguments as muon_step); the
 * group buckets them, chooses the paths (autotuning shapes not yet measured),
 * and owns its workspace and device pointer table.  muon_group_step then runs
 * one Muon step over the whole set: the first step after creation (or after a
 * configuration or tune-cache change) launches its kernels directly and the
 * following steps replay a CUDA graph captured on the group's own stream,
 * preceded on `stream` by a 16-byte copy of the step's hyper-parameters into a
 * device block the kernels read, so learning-rate schedules need no recapture.
 * MUON_GRAPH=0 disables the replay.  The pointers must stay valid for the
 * group's lifetime; a group belongs to the device that was current at
 * creation and is used by one host thread at a time.  The group's workspace is
 * allocated at its first step, so make that step before any stream capture of
 * your own.  muon_group_destroy synchronises the group's work and frees it.
 */
typedef struct muon_group muon_group;
int muon_group_create(void* const* params, const void* const* grads, void* const* moms,
                      const int64_t* ms, const int64_t* ns, int64_t count,
                      int param_dtype, int mom_dtype, muon_group** out);
int muon_group_step(muon_group* group, float lr, float beta, float wd, int nesterov, void* stream);
int muon_group_destroy(muon_group* group);

/*
 * Host-resident gradients and parameters for a group (a training loop that
 * keeps them in host memory, e.g. an offloaded optimizer, or that reads the
 * updated parameters back every step).  After this call every
 * muon_group_step also copies each gradient in from host_grads[i] and each
 * updated parameter out to host_params[i], on two copy streams of the group:
 * all gradient copies are issued at the start of the step in the order the
 * step processes its chunks of same-shape matrices, each chunk's update waits
 * only for its own gradients, and each chunk's parameters leave as soon as it
 * is updated, so the transfers overlap the tensor-core work of the other
 * chunks.  The whole step, copies included, is ordered on `stream` as before.
 *   host_grads   NULL, or `count` pointers (the group's matrix order) to
 *                pinned host memory (cudaMallocHost, cudaHostAlloc or
 *                cudaHostRegister) holding ms[i] x ns[i] elements of
 *                param_dtype; read every step into grads[i]
 *   host_params  NULL, or `count` pointers to pinned host memory that receive
 *                params[i] after its update every step
 * NULL for both turns the copies off again.  MUON_EINVAL for a NULL entry or
 * memory that is not pinned host memory; the previous setting is kept then.
 * The call synchronises the device (steps already enqueued with the previous
 * buffers finish first); the buffers must stay valid while the group steps
 * with them.
 */
int muon_group_set_host_io(muon_group* group, const void* const* host_grads, void* const* host_params);

/*
 * NS configuration used by muon_step (process-wide, mutex-guarded).
 * coeffs/steps as above; segments/num_segments give the Gram segmentation
 * (default 2+2+1: "MuonX" page, section 3.2); path is a muon_path.
 * NULL coeffs keeps the current coefficients.  The default is the quintic
 * coefficients, 5 steps, 2+2+1, MUON_PATH_AUTO.
 */
int muon_set_ns_config(const float coeffs[3], int steps, const int* segments,
                       int num_segments, int path);

/*
 * Working precision of NS for 16-bit parameters (process-wide, like the
 * configuration above): -1 (default) uses the parameters' own type, MUON_BF16
 * or MUON_F16 forces that type for X and the m x m iteration matrices.  fp16
 * keeps three more mantissa bits than bf16 at the cost of range, so its path
 * stores X already divided by ||U||_F (the momentum kernel runs twice: first
 * the sum of squares, then momentum and the scaled U).  fp32 parameters always
 * take the fp32 path.  Returns MUON_EDTYPE for any other value.
 */
int muon_set_ns_precision(int dtype);

/*
 * Measured-cost autotune ("DMuon" news page, section 3; "DMuon" summary,
 * sections 2.3-2.4): for each distinct oriented shape in (ms[i], ns[i]) times
 * the plain and the Gram path (and the tile choices of the long products) on
 * synthetic data in the workspace with CUDA events (median of several runs)
 * and caches the fastest.  Synchronises `stream`.  Never touches caller data.
 * Sides must lie in [1, 2^20], else MUON_EINVAL before any device work.
 */
int muon_autotune(const int64_t* ms, const int64_t* ns, int64_t count, int dtype, void* stream);

/* Persist / reload the tune cache (text file, keyed by device name, SM count,
 * CUDA runtime version, shape and dtype).  A missing file or a stale or
 * corrupt entry is ignored; returns the number of entries loaded (>= 0) or a
 * negative status. */
int muon_tune_save(const char* path);
int muon_tune_load(const char* path);

/* Which NS path (MUON_PATH_PLAIN / MUON_PATH_GRAM) muon_step last ran for this
 * oriented-or-not shape and dtype.  MUON_EINVAL if the shape has not run. */
int muon_last_path(int64_t m, int64_t n, int dtype, int* path_out);

/* Synchronise `stream`, then read and clear the current device's status word:
 * MUON_OK, MUON_ENONFINITE or MUON_ETIMEOUT (or MUON_ECUDA if the sync failed). */
int muon_sync_status(void* stream);

/* Human-readable name of a muon_status value (static string). */
const char* muon_status_str(int status);

/* Message of the last host-detected error on the calling thread ("" if none);
 * valid until the thread's next failing call. */
const char* muon_last_error_message(void);

/*
 * Product count of one NS update of an m x n matrix (oriented internally):
 * nominal = sum of 2*M*N*K over the products ("MuonX" page, section 3.2 counts
 * 1.443 -> 1.134 TFLOPs for 2560 x 9728); algorithmic counts products with a
 * symmetric result (XX^T and products of polynomials in the same Gram matrix)
 * as half.  path is MUON_PATH_PLAIN or MUON_PATH_GRAM (segments required).
 * At most 64 segments, each of length 1..64 (for the plain path they only
 * give the step count); MUON_EINVAL otherwise.
 */
int muon_ns_flops(int64_t m, int64_t n, int path, const int* segments, int num_segments,
                  double* nominal, double* algorithmic);

/*
 * AdamW step for the parameters that stay off Muon ("MuonX" page, section 2:
 * hidden 2-D weight matrices use Muon while embeddings and biases stay on
 * AdamW), all tensors in one launch.  The pages do not print AdamW; this is
 * the standard decoupled-decay form with 1-based step t:
 *   m' = b1 m + (1 - b1) g,  v' = b2 v + (1 - b2) g^2,
 *   p' = p (1 - lr wd) - lr m'/(1 - b1^t) / (sqrt(v'/(1 - b2^t)) + eps).
 *   params[i], grads[i]      device pointers, numels[i] elements (param_dtype:
 *                            MUON_F32, MUON_BF16 or MUON_F16)
 *   exp_avg[i], exp_avg_sq[i] device pointers, moments (state_dtype: MUON_F32 or
 *                            MUON_BF16; fp16 lacks the range of v), in place
 * Tensors may have any shape (flattened) and alignment; 16-byte aligned ones
 * take the vector path.  The pointer tables travel through the library's
 * workspace, so the first call may allocate.
 */
int muon_adamw_step(void* const* params, const void* const* grads, void* const* exp_avg,
                    void* const* exp_avg_sq, const int64_t* numels, int64_t count,
                    int param_dtype, int state_dtype, float lr, float beta1, float beta2,
                    float eps, float wd, int64_t step, void* stream);

/*
 * Owner placement for a multi-rank optimizer step ("DMuon" news page, section 3;
 * "DMuon" summary, section 2.3): each of `count` matrices (shapes ms[i] x ns[i])
 * gets one owner rank in [0, ranks) that runs its update, so that the
 * predicted per-rank time is balanced.  Costs: the tune cache's measured
 * milliseconds per matrix when every oriented shape has an entry for `dtype`
 * (*measured_out = 1), otherwise the algorithmic FLOPs of the path the library
 * picks without measurements (*measured_out = 0).  Greedy longest-processing-
 * time first, the pages' fallback to their MILP: matrices in decreasing cost
 * (stable in index), each to the least-loaded rank (ties to the lower rank).
 * Host-only and deterministic, so every rank computes the same plan.  Sides
 * must lie in [1, 2^20] (the limit of muon_step), else MUON_EINVAL.
 *   owner_out     count entries (required when count > 0)
 *   load_out      ranks entries or NULL: predicted cost per rank
 *   makespan_out  NULL or the largest per-rank cost
 *   measured_out  NULL or 1 / 0 as above
 */
int muon_owner_plan(const int64_t* ms, const int64_t* ns, int64_t count, int dtype, int ranks,
                    int* owner_out, double* load_out, double* makespan_out, int* measured_out);

/*
 * Packed exchange layout ("DMuon" summary, section 2.1: gradients are reduced
 * into owner-contiguous buffers before the orthogonalisation and the updated
 * parameters are published from them afterwards).  One buffer of
 * ranks x seg elements: rank r's segment [r seg, (r+1) seg) holds the matrices
 * it owns (owner[i], e.g. from muon_owner_plan) in ascending index, each
 * starting on a multiple of align_elems within the segment (pass 8 for
 * 16-byte starts of 16-bit elements); every segment is padded to the longest,
 * so that one reduce-scatter of the buffer hands each owner its summed
 * gradients and one all-gather hands every rank the owners' updated
 * parameters.  Host-only and deterministic (every rank computes the same
 * layout); each matrix at most 2^31 elements.
 *   offset_out    count entries: element offset of matrix i in the buffer
 *   seg_elems_out the segment length in elements
 */
int muon_pack_plan(const int64_t* ms, const int64_t* ns, const int* owner, int64_t count, int ranks,
                   int64_t align_elems, int64_t* offset_out, int64_t* seg_elems_out);

/*
 * Moves `count` row-major device matrices (mats[i], ms[i] x ns[i] elements of
 * dtype) to (to_packed != 0) or from (to_packed == 0) a packed device buffer,
 * matrix i at element offset offsets[i] (from muon_pack_plan), in one launch
 * on `stream`.  Elements between the matrices are neither read nor written.
 * The caller owns every buffer; regions must not overlap.  16-byte vector
 * copies where a matrix pointer, the buffer and offsets[i] * element size are
 * all 16-byte aligned, element copies otherwise.
 */
int muon_pack(void* const* mats, const int64_t* ms, const int64_t* ns, const int64_t* offsets,
              int64_t count, int dtype, void* packed, int to_packed, void* stream);

/* ---- diagnostics (not part of the method) ---------------------------------- */

/* Total kernels this library has launched in this process. */
int64_t muon_launch_count(void);

/*
 * Test hook of the kernels' bounded waits (not part of the method).  Arms a
 * one-shot stall that the next launch of one kernel takes: its CTA 0 issues
 * no copy for one pipeline stage, so the consumer's bounded wait for that
 * stage runs out (after about two seconds); the kernel then raises
 * MUON_ETIMEOUT in the status word, waits (bounded) for what it has in
 * flight, frees its tensor memory and returns, leaving the device usable.
 *   kernel 1  the tensor-core product kernel, unpaired launches (128-column
 *             tiles or pairing off): k-block `stage` of CTA 0's first tile
 *   kernel 2  the fused small-matrix kernel: prologue piece `stage` of CTA 0
 *             (16-byte aligned matrices)
 *   kernel 0  disarm.
 * MUON_EINVAL for another kernel or a stage outside [0, 2^20].
 */
int muon_debug_arm_stall(int kernel, int stage);

/* Enable (1) or disable (0) per-launch CUDA-event timing of the library's
 * kernels, recorded on the launching stream.  Reading resets the record. */
int muon_set_kernel_timing(int enable);

/*
 * Read the per-class timing record: for class k (0 <= k < max_classes)
 * writes its name into names (max_classes x 32 chars), its launches, total
 * milliseconds, and its algorithmic work per class (flops for products,
 * bytes for elementwise kernels).  Synchronises the recorded events.
 * Returns the number of classes written.
 */
int muon_kernel_timing_read(char* names, int64_t* launches, double* total_ms,
                            double* work, int max_classes);

/*
 * Single product launch for kernel-level tests (bf16 or fp32 path):
 *   C[b] = alpha * A[b] * op(B[b])  for b < batch, row-major, device pointers.
 *   A is M x K.  b_kmajor != 0: B is stored N x K and op(B) = B^T;
 *   b_kmajor == 0: B is stored K x N and op(B) = B.
 *   symmetric != 0 requires M == N and writes only the lower triangle's
 *   values, mirrored (C[j][i] = C[i][j]); valid when the exact product is
 *   symmetric.  poly != 0 (symmetric only, A == B == G) writes
 *   pa*I + pb*G + pc*(G G) instead of the product.
 *   C is M x N.  dtype is the storage type of A, B and C: MUON_BF16 or MUON_F16
 *   (16-bit tensor cores), MUON_F32 (fp32 FFMA), or 3 = fp32 storage
 *   multiplied on the TF32 tensor path (the kind the bf16 NS path uses for
 *   some Gram-space products; B must be K-major), or 4 = as 3 with the
 *   K-blocks accumulated in chunks of 32 (1024 elements), each chunk from zero,
 *   the chunk sums added in round-to-nearest fp32 (the fp32 path's three-pass
 *   products; 128 x 128 tiles, or 2-SM pairs when tile_n is 256).  tile_n selects the N extent of the
 *   tensor-core tile (0 = default, 128 or 256).
 */
int muon_debug_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                    int64_t batch, int dtype, int b_kmajor, int symmetric, int poly,
                    float alpha, float pa, float pb, float pc, int tile_n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_H */
