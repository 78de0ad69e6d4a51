// bf16 products of the Newton-Schulz path on the 5th-generation tensor cores.
//
// Every product of the Muon update is a dense contraction: the Gram matrix
// XX^T, the square products of polynomials in G (G^2, PG, (PG)P, PQ), and the
// long apply QX ("MuonX" page, section 3.2 counts them: 6 long and 11 square
// for 2+2+1 Gram NS).  XX^T and the square products have symmetric results;
// the "DMuon" summary (section 2.2) computes only one triangle of them, and so
// does this kernel: symmetric launches enumerate lower-triangle tiles only and
// mirror on store.  Because every square operand is symmetric, both operands of
// every product except QX can be read K-major straight from row-major storage;
// QX reads X as an MN-major operand.
//
// Structure (one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: 3-D tensor maps (k, row, batch), 128-byte swizzle,
//               STAGES-deep ring of (A, B) tiles guarded by full/empty mbarriers
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer
//               (M = 128, N = BN, K = 16 per instruction, fp32 accumulator)
//   warps 2-9   epilogue: two warps per TMEM lane quarter, each draining half
//               of the tile's columns with tcgen05.ld 32 at a time, fused
//               epilogue from epilogue.cuh; while the main loop of a tile runs
//               they prefetch into L2 the caller data their epilogue will read
// Operand kinds: bf16 or fp16 (kind::f16, K = 16 per instruction, A and B of
// the same type) for the long products and the 16-bit Gram-space products,
// TF32 on fp32 storage (kind::tf32, K = 8) for the Gram-space products that
// need it and for the fp32 path's three-pass products; either way one k-block
// is 128 bytes of every operand row.  The three-pass products accumulate in
// chunks of k-blocks added in round-to-nearest fp32 (the CH instance, below).
// The accumulator is double-buffered in TMEM (2 x BN columns) so the epilogue
// of tile t overlaps the main loop of tile t+1.
// Paired launches (PAIR, 128 x 256 tiles per CTA): 2-CTA clusters run 2-SM
// products (tcgen05 cta_group::2).  The CTAs take row blocks 2p and 2p+1 of
// one 256-column tile; each loads its own A rows and its half of B, so a stage
// is 32 KB instead of 48 KB and six stages fit; the odd CTA relays each filled
// stage to the even CTA's full barrier, the even CTA issues M = 256 products
// and commits to both CTAs' barriers, and both epilogues report to the even
// CTA.  TMEM is allocated collectively by one warp of each CTA.  Same tiles
// and K order, so the results equal the unpaired kernel's bit for bit.  Every mbarrier wait is bounded:
// after WAIT_LIMIT_NS it sets an abort flag and the status word, waits (again
// bounded) for its own copies and products in flight, frees TMEM and returns.
#include "muon_internal.cuh"
#include "epilogue.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace muon {

namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;            // bf16 elements per k-block = 128 bytes: one swizzle row
constexpr int BK_BYTES = 128;
constexpr int NEPI = 8;                        // epilogue warps
constexpr int NTHREADS = 64 + 32 * NEPI;

// MIR: the launch may be symmetric and needs the mirror staging (K-major B);
// MN-major launches (the long applies) never are, and spend the 33 KB on one
// more pipeline stage where a stage is 32 KB.
template <int BN, bool PAIR = false, bool MIR = true>
struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;   // paired: this CTA's half of B
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (PAIR || BN == 128) ? (MIR ? 5 : 7) : 4;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    // per epilogue warp: one 32 x 33 fp32 chunk (staged stores), or 4 KB
    // tile-store buffers used in turn, two where they fit
    static constexpr int STORE_BUFS = (STAGES * STAGE_BYTES + NEPI * 8192 + 2048 <= 232448) ? 2 : 1;
    static constexpr int MIRROR_WARP_BYTES = STORE_BUFS == 2 ? 8192 : 32 * 33 * 4;
    static constexpr int MIRROR_BYTES = MIR ? NEPI * MIRROR_WARP_BYTES : 0;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + MIRROR_BYTES + NUM_BARS * 8 + 16 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// Bounded wait on phase `parity`.  Gives up when another role has aborted or
// after WAIT_LIMIT_NS, in which case it raises the abort flag and the status.
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > WAIT_LIMIT_NS) {
                *abort_flag = 1;
                atomicOr(status, STATUS_TIMEOUT);
                return false;
            }
        }
    }
}

// Bounded wait used while draining after an abort (ignores the abort flag).
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > WAIT_LIMIT_NS) return;
    }
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// Load delivered to the same shared-memory offset, and signalled on the
// mbarrier at the same offset, in every CTA of the cluster set in `mask`.
__device__ __forceinline__ void tma_load_3d_mc(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                               int c2, uint16_t mask) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "h"(mask)
        : "memory");
}

// Tile store shared -> global on the copy engine (bulk group of this thread).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of this thread's stores may be overwritten
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all but the most recent bulk-store group have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// this thread's stores are complete
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_idx() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of both CTAs of the cluster arrives and waits.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on the mbarrier at the same shared offset in CTA `rank` of the
// cluster, releasing this thread's earlier writes (epilogue: TMEM reads done).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar, uint32_t rank) {
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(bar), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr) : "memory");
}

// Relaxed remote arrive for the stage relay: it forwards a completion this
// thread observed on its own mbarrier (bulk copies the copy engine finished),
// and has no writes of its own to order, so it needs no cluster-scope fence
// (a release here cost about 0.4 us per stage, serialising the pipeline).
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t bar, uint32_t rank) {
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(bar), "r"(rank));
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr) : "memory");
}

// 2-SM forms (a CTA pair of the cluster): TMEM allocated collectively by one
// warp of each CTA at the same address; the even CTA issues M = 256 products
// whose A rows and B columns are split between the two CTAs' shared memory
// at the same offsets, each CTA's TMEM receiving its 128 rows; commits track
// them and arrive on the barrier at `bar`'s offset in every CTA of the mask.
__device__ __forceinline__ void tmem_alloc2(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_commit2(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void tc_mma2_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_mma2_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i gets its lane's 32 values.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    // The wait names every destination register so no use is scheduled before it.
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
          "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
          "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
          "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
          "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
        :
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 consecutive fp32 columns from this thread's 32 values; the
// store is complete after tmem_wait_st.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
          "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
          "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
          "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
          "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
          "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
          "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
          "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
          "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
          "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
          "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: start, leading/stride byte offsets, the
// fixed descriptor version of this MMA generation (bit 46) and 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B both bf16
// (format code 1) or both fp16 (code 0), A K-major, B K-major or MN-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, bool b_mn_major, bool fp16) {
    return (1u << 4) | (fp16 ? 0u : ((1u << 7) | (1u << 10))) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of kind::tf32: fp32 accumulator, TF32 A and B (format
// code 2), both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Tile order within one matrix.  sym == 0: all tiles, row blocks fastest.
// sym == 1: square 128 x 128 tiles with tn <= tm (lower triangle).
// sym == 2: 128 x 256 tiles that meet the lower triangle, tn <= tm / 2; row
// blocks 2p and 2p+1 both hold p + 1 tiles, so p(p+1) tiles precede block 2p.
// pair != 0 (sym 0 or 2): a unit is the two tiles (2p, tn) and (2p+1, tn),
// one per CTA of a cluster (rank selects the row block); tiles_m then counts
// row-block pairs, and in sym 2 pair p holds tn = 0 .. p.
struct TileSched {
    int tiles_m, tiles_n, per_batch, total, sym, pair, mc;

    // Units before pair row p of a symmetric multicast schedule: row i holds
    // floor(i / 2) + 1 units of two tiles (tn = 2j and 2j + 1, up to i).
    __host__ __device__ static int mc_sym_units(int p) { return p + (p / 2) * ((p - 1) / 2); }

    // rank: the CTA's rank in its cluster.  valid (multicast schedules only):
    // false when this pair's tile of the unit lies outside the matrix (odd
    // tile counts); the pair then repeats its partner's tile and stores nothing.
    __device__ __forceinline__ void decode(int t, int& b, int& tm, int& tn, int rank = 0, bool* valid = nullptr) const {
        b = t / per_batch;
        const int l = t - b * per_batch;
        if (mc) {
            // a unit is two pair tiles sharing pair row p (the same A rows):
            // pair c = rank >> 1 takes column tile 2j + c
            const int c = rank >> 1;
            int p, j, lim;
            if (sym) {
                p = (int)(2.0f * (sqrtf((float)l + 1.0f) - 1.0f));
                if (p < 0) p = 0;
                while (p > 0 && mc_sym_units(p) > l) --p;
                while (mc_sym_units(p + 1) <= l) ++p;
                j = l - mc_sym_units(p);
                lim = p;                       // tn <= p
            } else {
                p = l % tiles_m;
                j = l / tiles_m;
                lim = tiles_n - 1;
            }
            tn = 2 * j + c;
            const bool ok = tn <= lim;
            if (!ok) tn = 2 * j;
            if (valid) *valid = ok;
            tm = 2 * p + (rank & 1);
            return;
        }
        if (valid) *valid = true;
        if (pair) {
            int p;
            if (sym) {
                p = (int)((sqrtf(8.0f * (float)l + 1.0f) - 1.0f) * 0.5f);
                while (p * (p + 1) / 2 > l) --p;
                while ((p + 1) * (p + 2) / 2 <= l) ++p;
                tn = l - p * (p + 1) / 2;
            } else {
                p = l % tiles_m;
                tn = l / tiles_m;
            }
            tm = 2 * p + rank;
        } else if (sym == 2) {
            int p = (int)((sqrtf(4.0f * (float)l + 1.0f) - 1.0f) * 0.5f);
            while (p * (p + 1) > l) --p;
            while ((p + 1) * (p + 2) <= l) ++p;
            const int off = l - p * (p + 1);
            tm = 2 * p + (off >= p + 1 ? 1 : 0);
            tn = off >= p + 1 ? off - (p + 1) : off;
        } else if (sym) {
            int r = (int)((sqrtf(8.0f * (float)l + 1.0f) - 1.0f) * 0.5f);
            while (r * (r + 1) / 2 > l) --r;
            while ((r + 1) * (r + 2) / 2 <= l) ++r;
            tm = r;
            tn = l - r * (r + 1) / 2;
        } else {
            tm = l % tiles_m;
            tn = l / tiles_m;
        }
    }
};

// 16-bit workspace products (EPI_STORE / EPI_POLY): one warp's 32 x 32 chunk
// (rows r0 + lane, columns c0..) is converted into one of the warp's two
// staging buffers (4 KB each: the chunk, then its transpose, 64-byte rows;
// chunks alternate between them, so one chunk's stores read shared memory
// while the next is converted) and leaves as tile stores on the copy engine,
// so the warp issues two instructions instead of sixteen row-piece stores.  Symmetric products: a chunk below the diagonal is stored
// at (r0, c0) and transposed at (c0, r0); the diagonal chunk (c0 == r0) is
// assembled symmetric (rows c <= r from v, the rest mirrored) and stored once,
// so no element is written twice.  The stores clip at the matrix edge.
template <int NB>
__device__ __forceinline__ void epi_store_tma(const GemmArgs& a, const CUtensorMap* tmC, int b, int r0, int c0,
                                              float (&v)[32], float s, const float (&g)[32], uint8_t* stg2,
                                              int& groups) {
    const int lane = threadIdx.x & 31;
    const int r = r0 + lane;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= s;
    if (a.epi == EPI_POLY) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = a.pc * v[j] + a.pb * g[j] + ((c0 + j) == r ? a.pa : 0.f);
    }
    const bool f16 = (a.c_dtype == MUON_F16);
    if (groups >= NB) {         // the stores that last used this buffer have read it
        if (lane == 0) {
            if (NB == 2) bulk_wait_read1();
            else bulk_wait_read0();
        }
        __syncwarp();
    }
    uint8_t* stg = stg2 + (groups % NB) * 4096;
    uint8_t* nrm = stg;
    uint8_t* trn = stg + 2048;
#pragma unroll
    for (int u = 0; u < 4; ++u) *reinterpret_cast<uint4*>(nrm + lane * 64 + 16 * u) = pack8_h(v + 8 * u, f16);
    const bool below = a.symmetric && c0 < r0;
    const bool diag = a.symmetric && c0 == r0;
    if (below || diag) {
        if (diag) __syncwarp();     // the mirrored entries replace the row stores' upper part
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            // element (j, lane) of the transpose, or of the diagonal chunk's upper part
            uint8_t* dst = (below ? trn : nrm) + j * 64 + lane * 2;
            if (below || j < lane) {
                if (f16) *reinterpret_cast<__half*>(dst) = __float2half_rn(v[j]);
                else *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(v[j]);
            }
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(tmC, smem_u32(nrm), c0, r0, b);
        if (below) tma_store_3d(tmC, smem_u32(trn), r0, c0, b);
        bulk_commit();
    }
    ++groups;
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

// CH (chunked accumulation, TF32): the k-blocks of a tile accumulate in
// chunks of args.kchunk, each from zero; the epilogue adds every chunk into a
// running-sum TMEM buffer with fp32 adds that round to nearest, and the last
// chunk's sum goes through the ordinary epilogue.  The tensor core's own fp32
// accumulation does not round to nearest, so over a long K its error grows
// with K; in chunks it is bounded by the chunk length.  Unpaired 128 x 128
// tiles keep two accumulators (a chunk accumulates while the previous one is
// added); a 2-SM pair's 128 x 256 half-tile leaves room for one accumulator
// beside the running sum, so its products wait for each chunk's addition.
template <int BN, bool B_KMAJOR, bool TF32, bool PAIR, bool MC, bool CH = false>
__global__ void __launch_bounds__(NTHREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ GemmArgs args, const TileSched sched) {
    using C = Cfg<BN, PAIR, B_KMAJOR>;
    constexpr int S = C::STAGES;
    constexpr int TCOLS = CH ? 512 : C::TMEM_COLS;     // chunked: the accumulators and the running sum
    constexpr int NBUF = (CH && PAIR) ? 1 : 2;         // TMEM accumulators that alternate
    constexpr int SUM_COL = NBUF * BN;                 // chunked: first column of the running sum
    static_assert(!TF32 || B_KMAJOR, "TF32 products read both operands K-major");
    static_assert(!CH || (TF32 && !MC && (PAIR ? BN == 256 : BN == 128)),
                  "chunked accumulation: TF32, unpaired 128-wide or paired 256-wide tiles");
    static_assert(!CH || SUM_COL + BN <= TCOLS, "running sum inside the TMEM allocation");
    static_assert(!PAIR || BN == 256, "paired products use 128 x 256 tiles per CTA");
    static_assert(!MC || PAIR, "multicast clusters are made of 2-SM pairs");
    constexpr int MM = PAIR ? 2 * BM : BM;      // rows of one product instruction
    const uint32_t IDESC = TF32 ? idesc_tf32(MM, BN) : idesc_f16kind(MM, BN, !B_KMAJOR, args.dtype == MUON_F16);
    constexpr int KE = TF32 ? 32 : 64;    // elements per 128-byte k-block

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + S * C::A_BYTES;
    float* mirror_stage = reinterpret_cast<float*>(sB + S * C::B_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + S * C::B_BYTES + C::MIRROR_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * S;
    const uint32_t accf0 = empty0 + 8 * S;
    const uint32_t acce0 = accf0 + 16;
    const uint32_t drain_bar = acce0 + 16;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Paired launches (2-SM products): the two CTAs of a pair take the two
    // row blocks of a 256 x BN tile.  Each loads its own A rows and its half
    // of B; the odd CTA relays "stage full" to the even CTA, which issues the
    // M = 256 products and commits to both; both epilogues report to the even
    // CTA's accumulator barrier.
    // Multicast launches (MC): a cluster of two pairs takes two tiles that
    // share their A rows (pair row p, column tiles 2j and 2j + 1).  CTA
    // (pair c, half h) loads rows c * 64 .. + 64 of its 128 A rows and
    // multicasts them to itself and to CTA (1 - c, h), so each A row leaves L2
    // once per cluster; a stage is refilled only after both pairs' products
    // have released it (the empty barriers count both pairs' commits).
    const int rank = PAIR ? (int)cluster_ctarank() : 0;
    const int lead = rank & ~1;             // the even CTA of this CTA's pair
    const int unit0 = PAIR ? (int)cluster_idx() : (int)blockIdx.x;
    const int ustep = PAIR ? (int)cluster_count() : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, (PAIR && (rank & 1) == 0) ? 2 : 1);   // own copies (+ the peer's relay)
            mbar_init(empty0 + 8 * s, MC ? 2 : 1);                        // one commit per pair
        }
        mbar_init(accf0, 1);
        mbar_init(accf0 + 8, 1);
        mbar_init(acce0, PAIR ? 2 * NEPI : NEPI);
        mbar_init(acce0 + 8, PAIR ? 2 * NEPI : NEPI);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        if (PAIR) {
            tmem_alloc2(smem_u32(tmem_slot), TCOLS);
            tmem_relinquish2();
        } else {
            tmem_alloc(smem_u32(tmem_slot), TCOLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();     // the peer's barriers exist before anything targets them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int kblocks = (args.K + KE - 1) / KE;
    const int kchunk = CH ? max(1, args.kchunk) : kblocks;     // k-blocks per accumulation chunk
    const int nchunks = CH ? (kblocks + kchunk - 1) / kchunk : 1;
    pdl_wait();          // operands, G, W and the scale come from earlier kernels
    pdl_trigger();

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            int issued[S];
#pragma unroll
            for (int s = 0; s < S; ++s) issued[s] = -1;
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = unit0; t < sched.total && ok; t += ustep) {
                int b, tm, tn;
                sched.decode(t, b, tm, tn, rank);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_bounded(empty0 + 8 * stage, phase ^ 1u, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    if (args.stall && kb == args.stall - 1 && t == unit0 && blockIdx.x == 0) {
                        // test hook: this stage is never filled, so the MMA
                        // issuer's bounded wait for it runs out; nothing is
                        // in flight for it (issued[] keeps its older phase)
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    mbar_expect_tx(fb, C::STAGE_BYTES);
                    if (MC) {
                        // half of the A rows, to this CTA and its counterpart in the other pair
                        const int c = rank >> 1, h = rank & 1;
                        tma_load_3d_mc(smem_u32(sA + stage * C::A_BYTES + c * (C::A_BYTES / 2)), &tmA, fb, kb * KE,
                                       tm * BM + c * (BM / 2), b, (uint16_t)((1u << h) | (1u << (2 + h))));
                    } else {
                        tma_load_3d(smem_u32(sA + stage * C::A_BYTES), &tmA, fb, kb * KE, tm * BM, b);
                    }
                    if (PAIR) {
                        // this CTA's half of B: rows (K-major) or columns (MN-major) (rank & 1) * BN / 2 ..
                        const int hb = (rank & 1) * (BN / 2);
                        if (B_KMAJOR) {
                            tma_load_3d(smem_u32(sB + stage * C::B_BYTES), &tmB, fb, kb * KE, tn * BN + hb, b);
                        } else {
#pragma unroll
                            for (int q = 0; q < BN / 128; ++q)
                                tma_load_3d(smem_u32(sB + stage * C::B_BYTES + q * (BK * 128)), &tmB, fb,
                                            tn * BN + hb + q * 64, kb * BK, b);
                        }
                    } else if (B_KMAJOR) {
                        tma_load_3d(smem_u32(sB + stage * C::B_BYTES), &tmB, fb, kb * KE, tn * BN, b);
                    } else {
#pragma unroll
                        for (int q = 0; q < BN / 64; ++q)
                            tma_load_3d(smem_u32(sB + stage * C::B_BYTES + q * (BK * 128)), &tmB, fb,
                                        tn * BN + q * 64, kb * BK, b);
                    }
                    issued[stage] = (int)phase;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // wait (bounded) for this CTA's copies still in flight: after an
            // abort the MMA issuer no longer consumes them, and even when this
            // loop ended normally the issuer may still give up on a stage
            // before the last copies land.  Without an abort the copies are
            // the issuer's next operands and land at once.
#pragma unroll
            for (int s = 0; s < S; ++s)
                if (issued[s] >= 0) wait_drain(full0 + 8 * s, (uint32_t)issued[s]);
        }
        __syncwarp();
    } else if (warp == 1 && PAIR && (rank & 1) == 1) {
        // ---------------- relay (odd CTA of a pair) ----------------
        // every completed stage of this CTA is reported to the even CTA's full
        // barrier; this CTA refills it only after the even CTA's commit
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = unit0; t < sched.total && ok; t += ustep) {
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!wait_bounded(full0 + 8 * stage, phase, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_remote_relaxed(full0 + 8 * stage, (uint32_t)lead);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t aphase = 0;
            bool ok = true;
            for (int t = unit0; t < sched.total && ok; t += ustep) {
              for (int c = 0; c < nchunks && ok; ++c) {
                const int kb0 = CH ? c * kchunk : 0;
                const int kb1 = CH ? min(kblocks, kb0 + kchunk) : kblocks;
                if (!wait_bounded(acce0 + 8 * acc, aphase ^ 1u, abort_flag, args.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(full0 + 8 * stage, phase, abort_flag, args.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + stage * C::A_BYTES);
                    const uint32_t b_base = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // one instruction consumes 32 bytes of K (16 bf16 or 8 TF32)
                        const uint64_t ad = sdesc(a_base + kk * 32, 16, 1024);
                        const uint64_t bd = B_KMAJOR ? sdesc(b_base + kk * 32, 16, 1024)
                                                     : sdesc(b_base + kk * 2048, BK * 128, 1024);
                        const uint32_t accum = (kb > kb0 || kk > 0) ? 1u : 0u;
                        if (PAIR) {
                            if (TF32) tc_mma2_tf32(d, ad, bd, IDESC, accum);
                            else tc_mma2_bf16(d, ad, bd, IDESC, accum);
                        } else {
                            if (TF32) tc_mma_tf32(d, ad, bd, IDESC, accum);
                            else tc_mma_bf16(d, ad, bd, IDESC, accum);
                        }
                    }
                    // release the stage in both CTAs of the pair (MC: of both pairs)
                    if (PAIR) tc_commit2(empty0 + 8 * stage, (uint16_t)(MC ? 0xF : (0x3u << lead)));
                    else tc_commit(empty0 + 8 * stage);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (PAIR) tc_commit2(accf0 + 8 * acc, (uint16_t)(0x3u << lead));
                else tc_commit(accf0 + 8 * acc);
                acc = (acc + 1) % NBUF;
                if (acc == 0) aphase ^= 1u;
              }
            }
            if (!ok) {
                // wait (bounded) for the products this thread issued
                if (PAIR) tc_commit2(drain_bar, (uint16_t)(0x1u << lead));
                else tc_commit(drain_bar);
                wait_drain(drain_bar, 0);
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..9) ----------------
        const int q = warp & 3;                    // TMEM lane quarter this warp may access
        float (*mstage)[33] =
            reinterpret_cast<float (*)[33]>(mirror_stage + (warp - 2) * (C::MIRROR_WARP_BYTES / 4));
        const int half = (warp - 2) / 4;           // which half of the tile's columns
        constexpr int HALF_COLS = BN / 2;
        int tma_groups = 0;                        // bulk-store groups this warp has issued
        int acc = 0;
        uint32_t aphase = 0;
        for (int t = unit0; t < sched.total; t += ustep) {
            int b, tm, tn;
            bool vtile = true;
            sched.decode(t, b, tm, tn, rank, &vtile);
            const bool valid = MC ? vtile : true;  // MC: a repeated tile is computed, not stored
            if (valid && args.epi == EPI_UPDATE) {
                // the update reads the caller's W: start pulling this tile's
                // part into L2 while the products are still accumulating
                const MatEntry e = args.mats[b];
                const int r = tm * BM + q * 32 + lane;
                const int cbeg = tn * BN + half * HALF_COLS;
                const int ob = args.out_dtype == MUON_BF16 ? 2 : 4;
                const char* wb = reinterpret_cast<const char*>(e.w);
                if (!e.trans) {
                    if (r < args.M)
                        for (int c = cbeg; c < min(cbeg + HALF_COLS, args.N); c += 128 / ob)
                            prefetch_l2(wb + ((int64_t)r * args.N + c) * ob);
                } else if (tm * BM + q * 32 < args.M) {
                    for (int c = cbeg + lane; c < min(cbeg + HALF_COLS, args.N); c += 32)
                        prefetch_l2(wb + ((int64_t)c * args.M + tm * BM + q * 32) * ob);
                }
            }
            if (CH && nchunks > 1) {
                // all chunks but the last: running sum (third TMEM buffer) += chunk,
                // this warp's 32 lanes x HALF_COLS columns, 32 at a time
                const uint32_t tl = tmem_base + ((uint32_t)(q * 32) << 16);
                bool cok = true;
                for (int c = 0; c + 1 < nchunks; ++c) {
                    const bool okw = wait_bounded(accf0 + 8 * acc, aphase, abort_flag, args.status);
                    if (!__all_sync(0xffffffffu, okw)) { cok = false; break; }
                    tc_fence_after();
#pragma unroll 1
                    for (int h = 0; h < HALF_COLS / 32; ++h) {
                        const uint32_t col = (uint32_t)(half * HALF_COLS + 32 * h);
                        float v[32];
                        tmem_ld32(tl + (uint32_t)(acc * BN) + col, v);
                        if (c > 0) {
                            float r[32];
                            tmem_ld32(tl + (uint32_t)SUM_COL + col, r);
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = __fadd_rn(r[j], v[j]);
                        }
                        tmem_st32(tl + (uint32_t)SUM_COL + col, v);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (PAIR && (rank & 1)) mbar_arrive_remote(acce0 + 8 * acc, (uint32_t)lead);
                        else mbar_arrive(acce0 + 8 * acc);
                    }
                    acc = (acc + 1) % NBUF;
                    if (acc == 0) aphase ^= 1u;
                }
                if (!cok) break;
            }
            // per-tile scalars and the first chunk's G / W loads are issued
            // before the wait, so their latency hides behind the main loop
            const float scale = epi_alpha(args, b);
            MatEntry ent{};
            if (args.epi == EPI_UPDATE || args.epi == EPI_OUT) ent = args.mats[b];
            const int row0 = tm * BM + q * 32;
            const int warp_row_max = row0 + 31;
            const int ch_beg = half * (HALF_COLS / 32), ch_end = valid ? (half + 1) * (HALF_COLS / 32) : ch_beg;
            const bool loads = valid && (args.epi == EPI_POLY || args.epi == EPI_UPDATE);
            float gcur[32], gnxt[32];
            if (loads) epi_load_chunk<32>(args, ent, b, row0 + lane, tn * BN + ch_beg * 32, gcur);
            // every lane observes the barrier itself; the warp proceeds only together
            const bool ok = wait_bounded(accf0 + 8 * acc, aphase, abort_flag, args.status);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
#pragma unroll 1
            for (int ch = ch_beg; ch < ch_end; ++ch) {
                const int col0 = tn * BN + ch * 32;
                if (col0 >= args.N) break;
                if (args.symmetric && col0 > warp_row_max) continue;
                if (loads && ch + 1 < ch_end)      // next chunk's loads fly while this one is processed
                    epi_load_chunk<32>(args, ent, b, row0 + lane, col0 + 32, gnxt);
                float v[32];
                tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + ch * 32), v);
                if (CH && nchunks > 1) {
                    float r[32];
                    tmem_ld32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(SUM_COL + ch * 32), r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __fadd_rn(r[j], v[j]);
                }
                if (B_KMAJOR && args.tma_c) {
                    // 16-bit workspace products: the chunk (and its mirror) leave on the copy engine
                    epi_store_tma<C::STORE_BUFS>(args, &tmC, b, row0, col0, v, scale, gcur,
                                  reinterpret_cast<uint8_t*>(&mstage[0][0]), tma_groups);
                } else if (B_KMAJOR && (args.epi == EPI_STORE || args.epi == EPI_POLY)) {
                    // workspace products: rows and mirrored rows through the staging area
                    epi_store_staged(args, b, row0, col0, v, scale, gcur, mstage);
                } else {
                    epi_row_chunk<32, false>(args, ent, b, row0 + lane, col0, v, scale, gcur);
                }
                if (loads) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) gcur[j] = gnxt[j];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && (rank & 1)) mbar_arrive_remote(acce0 + 8 * acc, (uint32_t)lead);
                else mbar_arrive(acce0 + 8 * acc);
            }
            acc = (acc + 1) % NBUF;
            if (acc == 0) aphase ^= 1u;
        }
        if (tma_groups > 0 && lane == 0) bulk_wait0();   // the stores are complete before the CTA exits
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (PAIR) cluster_sync();     // no product, commit or remote arrive targets this CTA any more
    if (warp == 1) {
        tc_fence_after();
        if (PAIR) tmem_dealloc2(tmem_base, TCOLS);
        else tmem_dealloc(tmem_base, TCOLS);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 3-D tensor map (fp32, bf16 or fp16 elements, by storage code) over `batch`
// matrices of `rows` x `inner` (row pitch ld, matrix pitch stride, in
// elements), box box_inner x box_rows x 1, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int dtype, uint64_t inner, uint64_t rows, uint64_t batch,
              uint64_t ld, uint64_t stride, uint32_t box_inner, uint32_t box_rows, bool swizzle = true) {
    auto fn = encode_fn();
    if (!fn) return false;
    if (batch <= 1) stride = ld * rows;
    const bool f32 = !is_half(dtype);
    const uint64_t eb = f32 ? 4 : 2;
    const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : (dtype == MUON_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {ld * eb, stride * eb};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t elem[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, elem,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// MUON_TMA_STORE=0 routes 16-bit workspace outputs through the staged row
// stores instead (both write the same values; the tests compare them)
bool tma_store_enabled() {
    const char* e = std::getenv("MUON_TMA_STORE");
    return !(e && e[0] == '0');
}

template <int BN, bool B_KMAJOR, bool TF32, bool PAIR, bool MC, bool CH = false>
cudaError_t launch_impl(const GemmArgs& a, int num_sms, cudaStream_t s) {
    using C = Cfg<BN, PAIR, B_KMAJOR>;
    auto kern = gemm_tc_kernel<BN, B_KMAJOR, TF32, PAIR, MC, CH>;
    constexpr int CL = MC ? 4 : 2;           // CTAs per cluster of a paired launch
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    static int max_clusters = 0;
    std::call_once(attr_once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (attr_err == cudaSuccess && PAIR) {
            // how many clusters of this kernel fit on the device at once
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(CL * (num_sms / CL));
            cfg.blockDim = dim3(NTHREADS);
            cfg.dynamicSmemBytes = C::SMEM_BYTES;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = CL;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
            if (attr_err == cudaSuccess && max_clusters < 1) attr_err = cudaErrorInvalidConfiguration;
        }
    });
    if (attr_err != cudaSuccess) return attr_err;

    CUtensorMap mA, mB;
    constexpr uint32_t KE = TF32 ? 32 : 64;   // elements per 128-byte k-block
    // multicast launches load A in halves of BM / 2 rows
    if (!make_map(&mA, a.A, a.dtype, (uint64_t)a.K, (uint64_t)a.M, (uint64_t)a.batch, (uint64_t)a.lda,
                  (uint64_t)a.strideA, KE, MC ? BM / 2 : BM))
        return cudaErrorInvalidValue;
    // a paired K-major B tile arrives as two halves of BN / 2 rows
    bool okB = B_KMAJOR ? make_map(&mB, a.B, a.dtype, (uint64_t)a.K, (uint64_t)a.N, (uint64_t)a.batch,
                                   (uint64_t)a.ldb, (uint64_t)a.strideB, KE, PAIR ? BN / 2 : BN)
                        : make_map(&mB, a.B, a.dtype, (uint64_t)a.N, (uint64_t)a.K, (uint64_t)a.batch,
                                   (uint64_t)a.ldb, (uint64_t)a.strideB, 64, BK);
    if (!okB) return cudaErrorInvalidValue;
    // 16-bit workspace outputs of K-major launches leave through tile stores
    CUtensorMap mC;
    std::memset(&mC, 0, sizeof mC);
    GemmArgs ga = a;
    ga.tma_c = 0;
    if (PAIR) ga.stall = 0;     // the wait test hook runs on unpaired launches only
    const bool c16 = is_half(a.c_dtype) && !a.round_tf32;
    const bool al = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && (a.ldc % 8 == 0) && (a.strideC % 8 == 0 || a.batch <= 1);
    if (B_KMAJOR && (a.epi == EPI_STORE || a.epi == EPI_POLY) && c16 && al && tma_store_enabled()) {
        if (make_map(&mC, a.C, a.c_dtype, (uint64_t)a.N, (uint64_t)a.M, (uint64_t)a.batch, (uint64_t)a.ldc,
                     (uint64_t)a.strideC, 32, 32, false))
            ga.tma_c = 1;
    }

    TileSched sc;
    sc.tiles_m = (a.M + BM - 1) / BM;
    sc.tiles_n = (a.N + BN - 1) / BN;
    sc.sym = a.symmetric ? (BN == 256 ? 2 : 1) : 0;
    sc.pair = PAIR ? 1 : 0;
    sc.mc = MC ? 1 : 0;
    if (PAIR) {
        const int pm = (sc.tiles_m + 1) / 2;
        sc.tiles_m = pm;
        if (MC) sc.per_batch = sc.sym ? TileSched::mc_sym_units(pm) : pm * ((sc.tiles_n + 1) / 2);
        else sc.per_batch = sc.sym ? pm * (pm + 1) / 2 : pm * sc.tiles_n;
    } else if (sc.sym == 2) {
        sc.per_batch = 0;
        for (int tm = 0; tm < sc.tiles_m; ++tm) sc.per_batch += tm / 2 + 1;
    } else {
        sc.per_batch = a.symmetric ? sc.tiles_m * (sc.tiles_m + 1) / 2 : sc.tiles_m * sc.tiles_n;
    }
    sc.total = sc.per_batch * a.batch;
    if (!PAIR) {
        const int grid = sc.total < num_sms ? sc.total : num_sms;
        return launch_pdl(kern, dim3(grid), dim3(NTHREADS), (size_t)C::SMEM_BYTES, s, mA, mB, mC, ga, sc);
    }
    int clusters = std::min(num_sms / CL, max_clusters);
    if (sc.total < clusters) clusters = sc.total;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL * clusters);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, mA, mB, mC, ga, sc);
}

}  // namespace tc

cudaError_t launch_gemm_tc(const GemmArgs& a, int num_sms, cudaStream_t s) {
    const bool tf32 = (a.dtype == DT_TF32);
    if (!is_half(a.dtype) && !tf32) return cudaErrorInvalidValue;
    if (tf32 && !a.b_kmajor) return cudaErrorInvalidValue;
    if (a.M < 1 || a.N < 1 || a.K < 1 || a.batch < 1) return cudaErrorInvalidValue;
    if (a.symmetric && (a.M != a.N || !a.b_kmajor)) return cudaErrorInvalidValue;
    // TMA: 16-byte aligned bases and pitches
    const int64_t epr = tf32 ? 4 : 8;   // elements per 16 bytes
    auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    if (!al16(a.A) || !al16(a.B) || (a.lda % epr) || (a.ldb % epr) || (a.strideA % epr) || (a.strideB % epr))
        return cudaErrorInvalidValue;
    if ((int64_t)a.batch * ((a.M + 127) / 128) * ((a.N + 127) / 128) > (int64_t)1 << 30)
        return cudaErrorInvalidValue;
    // symmetric products default to 128 x 128 tiles, the others to 128 x 256;
    // 128 x 256 tiles may run as 2-SM products on 2-CTA clusters (each CTA
    // loads its own operand tiles)
    const int bn = a.symmetric ? (a.tile_n == 256 ? 256 : 128) : (a.tile_n == 128 ? 128 : 256);
    const bool pair = (bn == 256) && a.pair != 0;
    const bool mc = pair && a.mc != 0;
    if (tf32) {
        // chunked accumulation: paired 256-wide tiles when asked for, else unpaired 128-wide
        if (a.kchunk > 0)
            return (bn == 256 && pair) ? tc::launch_impl<256, true, true, true, false, true>(a, num_sms, s)
                                       : tc::launch_impl<128, true, true, false, false, true>(a, num_sms, s);
        if (bn == 128) return tc::launch_impl<128, true, true, false, false>(a, num_sms, s);
        if (!pair) return tc::launch_impl<256, true, true, false, false>(a, num_sms, s);
        return mc ? tc::launch_impl<256, true, true, true, true>(a, num_sms, s)
                  : tc::launch_impl<256, true, true, true, false>(a, num_sms, s);
    }
    if (bn == 128) {
        return a.b_kmajor ? tc::launch_impl<128, true, false, false, false>(a, num_sms, s)
                          : tc::launch_impl<128, false, false, false, false>(a, num_sms, s);
    }
    if (pair) {
        if (mc)
            return a.b_kmajor ? tc::launch_impl<256, true, false, true, true>(a, num_sms, s)
                              : tc::launch_impl<256, false, false, true, true>(a, num_sms, s);
        return a.b_kmajor ? tc::launch_impl<256, true, false, true, false>(a, num_sms, s)
                          : tc::launch_impl<256, false, false, true, false>(a, num_sms, s);
    }
    return a.b_kmajor ? tc::launch_impl<256, true, false, false, false>(a, num_sms, s)
                      : tc::launch_impl<256, false, false, false, false>(a, num_sms, s);
}

}  // namespace muon
