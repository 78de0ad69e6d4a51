// Whole Muon update of one small matrix per CTA, for buckets of many small
// matrices ("DMuon" summary, section 2.2: matrices too small to fill the GPU
// are grouped by shape and their recursion runs jointly to amortise launch
// overhead).  One launch processes the whole bucket: CTAs loop over the
// bucket's matrices and each runs
//   momentum (+Nesterov) -> Frobenius norm -> NS -> fused update (or the ortho
//   output)
// without leaving the SM.  X (oriented m x n) lives in shared memory as bf16
// chunks of 64 columns in the 128-byte-swizzled K-major layout, the m x m
// matrices of the iteration in three 128 x 128 bf16 slots of the same layout,
// and every product accumulates in TMEM (512 columns).  Two forms share the
// 224 KB of shared memory:
//
//   ROWS = 128: m <= 128, n <= 512, plain or Gram NS with segments of length
//     <= 2 (eight chunks of 128 rows):
//       XX^T, G^2, PG, (PG)P, PQ : M = N = 128, both operands K-major
//       QX                       : M = 128, N <= 256 per instruction, X read
//                                  MN-major from the same chunks
//   ROWS = 256: 128 < m <= 256, n <= 256, plain NS (four chunks of 256 rows).
//     A = XX^T is symmetric, so it is kept as its three blocks A00, A10, A11
//     (A01 = A10^T is read through the transpose bits of the instruction
//     descriptor), then
//       A^2 blocks  C00 = A00 A00 + A10^T A10,  C10 = A10 A00 + A11 A10,
//                   C11 = A10 A10^T + A11 A11              (M = N = K = 128)
//       P = aI + bA + cA^2 block by block, in place of A
//       X <- P X    two M-halves, N = n, X read MN-major   (TMEM [0,256), [256,512))
//
// Rows m.. and columns n.. of X are zero, so the padding contributes nothing
// (a padded row i of P is a e_i and maps the zero row i of X to zero).  Eight
// warps: thread 0 issues the tcgen05.mma instructions; all warps run the
// prologue and drain TMEM (two warps per TMEM lane quarter, each half of the
// columns).
#include "muon_internal.cuh"
#include "epilogue.cuh"

namespace muon {
namespace small {

constexpr int NT = 256;
constexpr int SCHUNK = 128 * 128;           // bytes of one 128-row x 64-column bf16 chunk
constexpr int X_BYTES = 128 * 1024;         // eight 128-row or four 256-row chunks
constexpr int S_BYTES = 2 * SCHUNK;         // one 128 x 128 slot
constexpr int SMEM_BYTES = X_BYTES + 3 * S_BYTES + 256 + 1024;

// ---- PTX helpers (same instruction forms as the persistent product kernel) ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
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

// Bounded wait: false after WAIT_LIMIT_NS.
__device__ __noinline__ bool wait_limited(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > WAIT_LIMIT_NS) return false;
    }
    return true;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle.  K-major operands: LBO
// unused (16), SBO = 1024 (8-row groups).  MN-major operands: LBO = stride
// between 64-element chunks of the M/N extent, SBO = 1024 (8-row K groups).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16 with bf16 A and B, fp32 accumulate; bit 15
// reads A MN-major (transposed), bit 16 B.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

#define MUON_R32(r)                                                                                          \
    "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),        \
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),            \
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),          \
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),          \
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define MUON_RW32(r)                                                                                         \
    "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),        \
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),            \
        "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),          \
        "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),          \
        "+r"(r[29]), "+r"(r[30]), "+r"(r[31])

// 32 consecutive TMEM columns of this thread's lane (warp-collective; the
// registers are valid only after tmem_wait).
__device__ __forceinline__ void tmem_issue32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : MUON_R32(r)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : MUON_RW32(r) : : "memory");
}
// Orders later uses of r after a preceding tmem_wait (volatile asm keeps its place).
__device__ __forceinline__ void reg_after_wait(uint32_t (&r)[32]) { asm volatile("" : MUON_RW32(r)); }

// Two 32-column loads behind one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t t0, uint32_t t1, float (&v0)[32], float (&v1)[32]) {
    uint32_t r0[32], r1[32];
    tmem_issue32(t0, r0);
    tmem_issue32(t1, r1);
    tmem_wait(r0);
    reg_after_wait(r1);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v0[i] = __uint_as_float(r0[i]);
        v1[i] = __uint_as_float(r1[i]);
    }
}

// Byte offset of element (r, c) in a chunked K-major region of ROWS-row
// chunks: chunk c / 64, row r at 128 B, 16-byte unit (c % 64) / 8 XOR-swizzled
// by r % 8 (the layout a TMA load with 128-byte swizzle produces).
template <int ROWS>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    const int cc = c & 63;
    return (uint32_t)((c >> 6) * (ROWS * 128) + r * 128 + ((((cc >> 3) ^ (r & 7)) << 4) | ((cc & 7) << 1)));
}

__device__ __forceinline__ uint4 pack8(const float* v) {
    __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]);
    __nv_bfloat162 h1 = __floats2bfloat162_rn(v[2], v[3]);
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[4], v[5]);
    __nv_bfloat162 h3 = __floats2bfloat162_rn(v[6], v[7]);
    uint4 q;
    q.x = *reinterpret_cast<uint32_t*>(&h0);
    q.y = *reinterpret_cast<uint32_t*>(&h1);
    q.z = *reinterpret_cast<uint32_t*>(&h2);
    q.w = *reinterpret_cast<uint32_t*>(&h3);
    return q;
}

__device__ __forceinline__ void unpack8(const uint4 q, float* v) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        v[2 * k] = f.x;
        v[2 * k + 1] = f.y;
    }
}

// Stores 32 values (columns c0..c0+31, c0 % 32 == 0) of row r as bf16.
template <int ROWS>
__device__ __forceinline__ void st_row32(uint8_t* region, int r, int c0, const float (&v)[32]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) *reinterpret_cast<uint4*>(region + swz<ROWS>(r, c0 + 8 * u)) = pack8(v + 8 * u);
}

template <int ROWS>
__device__ __forceinline__ void ld_row32(const uint8_t* region, int r, int c0, float (&v)[32]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) unpack8(*reinterpret_cast<const uint4*>(region + swz<ROWS>(r, c0 + 8 * u)), v + 8 * u);
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Contiguous global -> shared copy on the bulk-copy engine, completion counted
// in bytes on the mbarrier (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

constexpr int PIECE = 8192;                 // elements per prologue piece
constexpr int STAGE_AREA = 3 * S_BYTES;     // the three slots, free during the prologue

// Pipeline state of the prologue's staged loads; every thread holds the same
// copy.  Piece k of the launch uses stage k % nst with parity (k / nst) & 1.
struct Stream {
    uint32_t bars;          // shared address of the first of three stage mbarriers
    uint32_t stage;         // shared address of the stage area
    uint32_t nst;           // stages in use (2 or 3, fixed for the launch)
    uint32_t consumed;      // pieces consumed so far in this launch
    uint32_t issued;        // pieces issued so far in this launch
};

// Stages of the prologue stream for this launch's momentum dtype.
__device__ __forceinline__ uint32_t stream_stages(const SmallArgs& a) {
    const uint32_t msz = a.mode == 0 ? (a.mom_dtype == MUON_F32 ? 4u : 2u) : 0u;
    return min(3u, (uint32_t)STAGE_AREA / (PIECE * (2u + msz)));
}

// Piece p of matrix e (total elements; gradient then, for a Muon step,
// momentum) as piece k of the launch: stage k % nst, its barrier expecting
// the bytes.  Thread 0 only; the stage must be free.
__device__ __forceinline__ void issue_piece(const SmallArgs& a, const MatEntry& e, int total, uint32_t k, int p,
                                            const Stream& st) {
    const bool step = (a.mode == 0);
    const uint32_t msz = step ? (a.mom_dtype == MUON_F32 ? 4u : 2u) : 0u;
    const uint32_t gbytes = PIECE * 2;
    const uint32_t sbytes = gbytes + PIECE * msz;
    const uint32_t s = k % st.nst;
    const uint32_t bar = st.bars + 8 * s;
    const uint32_t elems = (uint32_t)min(PIECE, total - p * PIECE);
    // test hook: CTA 0 issues no copy for this piece, so the wait for it runs out
    if (a.stall && k == (uint32_t)(a.stall - 1) && blockIdx.x == 0) return;
    mbar_expect_tx(bar, elems * (2 + msz));
    bulk_g2s(st.stage + s * sbytes, reinterpret_cast<const __nv_bfloat16*>(e.grad) + (int64_t)p * PIECE, elems * 2,
             bar);
    if (step)
        bulk_g2s(st.stage + s * sbytes + gbytes, reinterpret_cast<const char*>(e.mom) + (int64_t)p * PIECE * msz,
                 elems * msz, bar);
}

// U of one matrix (momentum update when a.mode == 0) into X; returns this
// thread's sum of squares of U.  Aligned inputs stream through the slot area
// in pieces of 8192 elements on the bulk-copy engine (two or three pieces in
// flight); the rest takes one element per thread at a time.  ok turns false
// if a piece does not arrive within the wait limit.
template <int ROWS>
__device__ float prologue(const SmallArgs& a, const SmallBucket& bk, const MatEntry& e, uint8_t* X,
                          uint8_t* stage_ptr, Stream& st, bool& ok) {
    const int tid = threadIdx.x;
    const int raw_rows = e.trans ? bk.n : bk.m;
    const int raw_cols = e.trans ? bk.m : bk.n;
    const int total = raw_rows * raw_cols;
    const bool step = (a.mode == 0);
    const float beta = a.hyper ? a.hyper[1] : a.beta;
    const int nesterov = a.hyper ? (a.hyper[3] != 0.f) : a.nesterov;
    float ss = 0.f;
    auto put = [&](int e0, const float* u, int cnt) {
        const int rr = e0 / raw_cols, cc = e0 - rr * raw_cols;
        if (!e.trans && cnt == 8) {
            *reinterpret_cast<uint4*>(X + swz<ROWS>(rr, cc)) = pack8(u);
        } else {
            for (int k = 0; k < cnt; ++k) {
                const int r = e.trans ? cc + k : rr;
                const int c = e.trans ? rr : cc + k;
                *reinterpret_cast<__nv_bfloat16*>(X + swz<ROWS>(r, c)) = __float2bfloat16_rn(u[k]);
            }
        }
    };
    if (!bk.vec_ok) {
        for (int i = tid; i < total; i += NT) {
            const float g = ld_elem(e.grad, i, a.param_dtype);
            float u = g;
            if (step) {
                const float mn = fmaf(beta, ld_elem(e.mom, i, a.mom_dtype), g);
                st_elem(e.mom, i, mn, a.mom_dtype);
                u = nesterov ? fmaf(beta, mn, g) : mn;
            }
            ss = fmaf(u, u, ss);
            put(i, &u, 1);
        }
        return ss;
    }
    const bool mf32 = (a.mom_dtype == MUON_F32);
    const int msz = step ? (mf32 ? 4 : 2) : 0;
    const uint32_t gbytes = PIECE * 2;
    const uint32_t sbytes = gbytes + PIECE * msz;           // one stage: gradient then momentum
    const uint32_t nst = st.nst;
    const int npieces = (total + PIECE - 1) / PIECE;
    const uint32_t first = st.consumed;
    auto issue = [&](int p) { issue_piece(a, e, total, first + (uint32_t)p, p, st); };
    if (tid == 0) {
        fence_async_smem();         // earlier generic accesses of the stage area come first
        for (int p = 0; p < npieces && p < (int)nst; ++p) issue(p);
    }
    st.issued = first + (uint32_t)min(npieces, (int)nst);
    for (int p = 0; p < npieces; ++p) {
        const uint32_t k = first + (uint32_t)p;
        const uint32_t s = k % nst;
        const bool arrived = wait_limited(st.bars + 8 * s, (k / nst) & 1u);
        if (__syncthreads_and(arrived ? 1 : 0) == 0) {
            ok = false;
            return ss;
        }
        st.consumed = k + 1;
        const uint8_t* sg = stage_ptr + s * sbytes;
        const uint8_t* sm = sg + gbytes;
        const int base = p * PIECE;
        const int elems = min(PIECE, total - base);
        for (int i = tid * 8; i < elems; i += NT * 8) {
            float g[8], u[8];
            unpack8(*reinterpret_cast<const uint4*>(sg + 2 * i), g);
            if (step) {
                float mo[8];
                if (mf32) {
                    const float4 f0 = *reinterpret_cast<const float4*>(sm + 4 * i);
                    const float4 f1 = *reinterpret_cast<const float4*>(sm + 4 * i + 16);
                    mo[0] = f0.x; mo[1] = f0.y; mo[2] = f0.z; mo[3] = f0.w;
                    mo[4] = f1.x; mo[5] = f1.y; mo[6] = f1.z; mo[7] = f1.w;
                } else {
                    unpack8(*reinterpret_cast<const uint4*>(sm + 2 * i), mo);
                }
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {
                    mo[k2] = fmaf(beta, mo[k2], g[k2]);
                    u[k2] = nesterov ? fmaf(beta, mo[k2], g[k2]) : mo[k2];
                }
                store_row_run<8>(e.mom, base + i, mo, a.mom_dtype);
            } else {
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) u[k2] = g[k2];
            }
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) ss = fmaf(u[k2], u[k2], ss);
            put(base + i, u, 8);
        }
        __syncthreads();            // every thread is done with stage s
        if (tid == 0 && p + (int)nst < npieces) {
            fence_async_smem();
            issue(p + (int)nst);
        }
        st.issued = first + (uint32_t)min(npieces, p + 1 + (int)nst);
    }
    return ss;
}

// Output of one M-half of O: rows row0 .. row0+127 in TMEM lanes, columns in
// TMEM [tl + c) for c < 64 nck, scaled by alpha; written to the caller as O
// (mode 1) or applied to W (mode 0).  Blocks of 256 columns pass through
// shared memory as fp32 so that the caller's rows are read and written whole
// by a warp, not one row per lane.  The stage fills X exactly (128 rows of
// 1024 B, not a byte past it): the 16-byte piece index of float column c of
// row i is XOR-ed with i & 7, so eight lanes writing one column to eight rows
// hit eight bank groups.
__device__ __forceinline__ int so_off(int i, int c) { return i * 1024 + ((((c >> 2) ^ (i & 7)) << 4) | ((c & 3) << 2)); }

__device__ __noinline__ void write_out(const SmallArgs& a, const SmallBucket& bk, const MatEntry& e, uint8_t* stage,
                                       uint32_t tl, int row0, float alpha, int nck) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hw = warp >> 2, r = 32 * (warp & 3) + lane;
    const float lr = a.hyper ? a.hyper[0] : a.lr;
    const float wd = a.hyper ? a.hyper[2] : a.wd;
    const float lrwd = lr * wd;
    const float stepc = lr * bk.scale;
    const int od = a.param_dtype;
    const bool upd = (a.mode == 0);
    for (int col0 = 0; col0 < nck * 64; col0 += 256) {
        const int bc = min(256, nck * 64 - col0);
        // TMEM -> stage: this thread's row r, 32-column chunks [k0, k1) of the block
        const int per = bc / 64, k0 = hw * per, k1 = k0 + per;
        for (int k = k0; k < k1; k += 2) {
            float v0[32], v1[32];
            tmem_ld64(tl + col0 + 32 * k, tl + col0 + 32 * (k + 1), v0, v1);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                *reinterpret_cast<float4*>(stage + so_off(r, 32 * k + 4 * u)) =
                    make_float4(v0[4 * u] * alpha, v0[4 * u + 1] * alpha, v0[4 * u + 2] * alpha, v0[4 * u + 3] * alpha);
            if (k + 1 < k1) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    *reinterpret_cast<float4*>(stage + so_off(r, 32 * (k + 1) + 4 * u)) = make_float4(
                        v1[4 * u] * alpha, v1[4 * u + 1] * alpha, v1[4 * u + 2] * alpha, v1[4 * u + 3] * alpha);
            }
        }
        __syncthreads();
        if (!e.trans) {
            // warp w: rows w, w+8, ...; lane l: columns 8l .. 8l+7 of the block
            const int c = 8 * lane, col = col0 + c;
            if (c < bc && col < bk.n) {
                if (bk.vec_ok) {
                    // all sixteen rows' W in flight before the first is used
                    __nv_bfloat16* wp = reinterpret_cast<__nv_bfloat16*>(e.w);
                    uint4 w[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const int row = row0 + warp + 8 * t;
                        w[t] = (upd && row < bk.m) ? *reinterpret_cast<const uint4*>(wp + (int64_t)row * bk.n + col)
                                                  : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const int i = warp + 8 * t, row = row0 + i;
                        if (row >= bk.m) continue;
                        const float4 o0 = *reinterpret_cast<const float4*>(stage + so_off(i, c));
                        const float4 o1 = *reinterpret_cast<const float4*>(stage + so_off(i, c + 4));
                        float o[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
                        if (upd) {
                            float wf[8];
                            unpack8(w[t], wf);
#pragma unroll
                            for (int j = 0; j < 8; ++j) o[j] = wf[j] - fmaf(lrwd, wf[j], stepc * o[j]);
                        }
                        *reinterpret_cast<uint4*>(wp + (int64_t)row * bk.n + col) = pack8(o);
                    }
                } else {
                    for (int i = warp; i < 128 && row0 + i < bk.m; i += 8) {
                        const int64_t off = (int64_t)(row0 + i) * bk.n + col;
                        for (int j = 0; j < 8 && col + j < bk.n; ++j) {
                            float o = *reinterpret_cast<const float*>(stage + so_off(i, c + j));
                            if (upd) {
                                const float w = ld_elem(e.w, off + j, od);
                                o = w - fmaf(lrwd, w, stepc * o);
                            }
                            st_elem(e.w, off + j, o, od);
                        }
                    }
                }
            }
        } else {
            // the caller's matrix is the transpose: its row j is column j of O;
            // warp w: caller rows col0 + w, + 8, ...; lane l: elements l + 32 t
            for (int jj = warp; jj < bc && col0 + jj < bk.n; jj += 8) {
                const int64_t rbase = (int64_t)(col0 + jj) * bk.m;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int i = lane + 32 * t, row = row0 + i;
                    if (row >= bk.m) continue;
                    float o = *reinterpret_cast<const float*>(stage + so_off(i, jj));
                    if (upd) {
                        const float w = ld_elem(e.w, rbase + row, od);
                        o = w - fmaf(lrwd, w, stepc * o);
                    }
                    st_elem(e.w, rbase + row, o, od);
                }
            }
        }
        __syncthreads();
    }
}

// Per-CTA state shared by the matrices a CTA processes.
struct Ctx {
    uint8_t *X, *S0, *S1, *S2;
    float* red;              // 8 warp partials
    float* inv_s;
    uint32_t barA, tmem, tlane;
    int tid, warp, lane, hw, r;
    uint32_t phase;          // parity of the product barrier
    Stream stream;
};

// The whole update of matrix b of bucket bk (ROWS: the X layout, 128 or 256
// rows); nx: the CTA's next matrix (or null) whose inputs are pulled into L2
// meanwhile.  Returns false when a bounded wait gave up.
template <int ROWS>
__device__ bool process(const SmallArgs& a, const SmallBucket& bk, int b, const MatEntry* nx, int64_t nx_elems,
                        Ctx& c) {
    constexpr bool BIG = (ROWS == 256);
    constexpr int XCH = ROWS * 128;             // bytes of one X chunk
    uint8_t* const X = c.X;
    uint8_t* const S0 = c.S0;
    uint8_t* const S1 = c.S1;
    uint8_t* const S2 = c.S2;
    const uint32_t barA = c.barA, tmem = c.tmem, tlane = c.tlane;
    const int tid = c.tid, warp = c.warp, lane = c.lane, hw = c.hw, r = c.r;
    uint32_t& phase = c.phase;
    const int nck = (bk.n + 63) / 64;           // X chunks in use
    const bool pad = (bk.m != ROWS) || (bk.n % 64 != 0);
    constexpr uint32_t ID_SQ = idesc_bf16(128, 128, false, false);
    bool ok = true;

    // One product round: make this thread's smem writes visible to the tensor
    // cores and let thread 0 issue (begin); wait for completion, bounded (finish).
    auto begin = [&](auto&& issue) {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            issue();
            tc_commit(barA);
        }
    };
    auto finish = [&]() -> bool {
        const bool done = wait_limited(barA, phase);
        phase ^= 1u;
        const bool all = __syncthreads_and(done ? 1 : 0) != 0;
        tc_fence_after();
        return all;
    };
    auto run = [&](auto&& issue) -> bool {
        begin(issue);
        return finish();
    };
    // K-major X rows row0.., k-step s (16 elements)
    auto kx = [&](int row0, int s) {
        return sdesc(smem_u32(X) + (s >> 2) * XCH + row0 * 128 + (s & 3) * 32, 16, 1024);
    };
    // K-major slot, k-step s
    auto ks = [&](const uint8_t* S, int s) { return sdesc(smem_u32(S) + (s >> 2) * SCHUNK + (s & 3) * 32, 16, 1024); };
    // slot read transposed (MN-major): K runs over its rows 16s..16s+15
    auto ms = [&](const uint8_t* S, int s) { return sdesc(smem_u32(S) + s * 2048, SCHUNK, 1024); };
    // X as the MN-major B operand: K over rows krow.., N over the chunks from chunk0
    auto mx = [&](int krow, int chunk0) { return sdesc(smem_u32(X) + chunk0 * XCH + krow * 128, XCH, 1024); };

    // slot <- scale * TMEM columns [src + 64 hw, +64) of this lane
    auto drain_store = [&](uint32_t src, uint8_t* dst, float scale) {
        const int c0 = 64 * hw;
        float v0[32], v1[32];
        tmem_ld64(tlane + src + c0, tlane + src + c0 + 32, v0, v1);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            v0[j] *= scale;
            v1[j] *= scale;
        }
        st_row32<128>(dst, r, c0, v0);
        st_row32<128>(dst, r, c0 + 32, v1);
    };
    // slot <- a I (diagonal blocks) + b G + c acc, G the bf16 slot the square
    // consumed (so both terms see the same rounded G: an fp32 linear term with
    // a bf16 G^2 loses the cancellation a + b s^2 + c s^4 relies on near s = 1);
    // dst may be gslot (each thread reads its elements before writing them)
    auto drain_poly = [&](uint32_t src, const uint8_t* gslot, uint8_t* dst, bool diag) {
        const int c0 = 64 * hw;
        float v0[32], v1[32], g0[32], g1[32];
        tmem_ld64(tlane + src + c0, tlane + src + c0 + 32, v0, v1);
        ld_row32<128>(gslot, r, c0, g0);
        ld_row32<128>(gslot, r, c0 + 32, g1);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            v0[j] = a.c * v0[j] + a.b * g0[j] + ((diag && c0 + j == r) ? a.a : 0.f);
            v1[j] = a.c * v1[j] + a.b * g1[j] + ((diag && c0 + 32 + j == r) ? a.a : 0.f);
        }
        st_row32<128>(dst, r, c0, v0);
        st_row32<128>(dst, r, c0 + 32, v1);
    };
    // X row (row0 + lane) <- alpha * TMEM columns [tcol + 32 k) of this thread's chunks
    auto drain_x = [&](uint32_t tcol, int row0, float alpha) {
        const int k0 = hw * nck, k1 = k0 + nck;
        for (int k = k0; k < k1; k += 2) {
            float v0[32], v1[32];
            tmem_ld64(tlane + tcol + 32 * k, tlane + tcol + 32 * (k + 1), v0, v1);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                v0[j] *= alpha;
                v1[j] *= alpha;
            }
            st_row32<ROWS>(X, row0 + r, 32 * k, v0);
            if (k + 1 < k1) st_row32<ROWS>(X, row0 + r, 32 * (k + 1), v1);
        }
    };

    const MatEntry e = bk.mats[b];
    // zero the padding of X (only when there is padding), and start pulling
    // this matrix's W into L2
    if (pad) {
        for (int i = tid; i < nck * (XCH / 16); i += NT) reinterpret_cast<uint4*>(X)[i] = make_uint4(0, 0, 0, 0);
        __syncthreads();
    }
    // W is pulled into L2 as the last segment starts, so that it is still
    // there when the write-out reads it
    auto prefetch_w = [&]() {
        if (a.mode != 0) return;
        const int64_t wbytes = (int64_t)bk.m * bk.n * 2;
        for (int64_t off = (int64_t)tid * 128; off < wbytes; off += (int64_t)NT * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(e.w) + off));
    };
    float ss = prologue<ROWS>(a, bk, e, X, S0, c.stream, ok);
    if (!ok) return false;
    // while this matrix iterates, pull the next one's inputs into L2
    if (nx) {
        const int64_t gbytes = nx_elems * (a.param_dtype == MUON_BF16 ? 2 : 4);
        const int64_t mbytes = nx_elems * (a.mom_dtype == MUON_BF16 ? 2 : 4);
        for (int64_t off = (int64_t)tid * 128; off < gbytes; off += (int64_t)NT * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(nx->grad) + off));
        if (a.mode == 0)
            for (int64_t off = (int64_t)tid * 128; off < mbytes; off += (int64_t)NT * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(nx->mom) + off));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) c.red[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        double t = 0.0;
        for (int w = 0; w < NT / 32; ++w) t += (double)c.red[w];
        if (!isfinite(t)) atomicOr(a.status, STATUS_NONFINITE);
        *c.inv_s = (float)(1.0 / (sqrt(t) + 1e-7));
    }
    __syncthreads();
    const float inv = *c.inv_s;

    if constexpr (!BIG) {
        for (int si = 0; si < bk.nseg && ok; ++si) {
            const int L = bk.segs[si];
            const bool first = (si == 0), last = (si == bk.nseg - 1);
            const float gs = first ? inv * inv : 1.0f;
            if (last) prefetch_w();
            auto square = [&](const uint8_t* A, const uint8_t* B, uint32_t col) {
                return run([&] {
                    for (int s = 0; s < 8; ++s) tc_mma(tmem + col, ks(A, s), ks(B, s), ID_SQ, s > 0 ? 1u : 0u);
                });
            };
            // G = X X^T -> TMEM [0, 128) -> S0
            ok = run([&] {
                for (int s = 0; s < nck * 4; ++s) tc_mma(tmem, kx(0, s), kx(0, s), ID_SQ, s > 0 ? 1u : 0u);
            });
            if (!ok) break;
            drain_store(0, S0, gs);
            // P1 = aI + bG + cG^2 -> S1
            if (!(ok = square(S0, S0, 128))) break;
            drain_poly(128, S0, S1, true);
            uint8_t* Q = S1;
            if (L == 2) {
                if (!(ok = square(S1, S0, 256))) break;       // P1 G -> S2
                drain_store(256, S2, 1.f);
                if (!(ok = square(S2, S1, 0))) break;         // (P1 G) P1 = G' -> S0
                drain_store(0, S0, 1.f);
                if (!(ok = square(S0, S0, 128))) break;       // P2 = aI + bG' + cG'^2 -> S2
                drain_poly(128, S0, S2, true);
                if (!(ok = square(S2, S1, 256))) break;       // Q = P2 P1 -> S0
                drain_store(256, S0, 1.f);
                Q = S0;
            }
            // X <- Q X : TMEM [0, 64 nck)
            ok = run([&] {
                for (int h = 0; h < 2; ++h) {
                    const int nh = min(256, nck * 64 - 256 * h);
                    if (nh <= 0) break;
                    const uint32_t id = idesc_bf16(128, nh, false, true);
                    for (int s = 0; s < 8; ++s) tc_mma(tmem + 256 * h, ks(Q, s), mx(16 * s, 4 * h), id, s > 0 ? 1u : 0u);
                }
            });
            if (!ok) break;
            const float alpha = first ? inv : 1.0f;
            if (!last) drain_x(0, 0, alpha);
            else write_out(a, bk, e, X, tlane, 0, alpha, nck);
        }
    } else {
        constexpr uint32_t ID_WIDE = idesc_bf16(128, 256, false, false);
        constexpr uint32_t ID_TT = idesc_bf16(128, 128, true, true);
        constexpr uint32_t ID_KT = idesc_bf16(128, 128, false, true);
        const uint32_t id_px = idesc_bf16(128, nck * 64, false, true);
        const uint32_t id_px_t = idesc_bf16(128, nck * 64, true, true);
        for (int it = 0; it < bk.nseg && ok; ++it) {
            const bool first = (it == 0), last = (it == bk.nseg - 1);
            const float gs = first ? inv * inv : 1.0f;
            if (last) prefetch_w();
            // A = X X^T: A00 -> TMEM [0, 128); rows 128.. (A10 | A11) -> [128, 384)
            ok = run([&] {
                for (int s = 0; s < nck * 4; ++s) {
                    tc_mma(tmem, kx(0, s), kx(0, s), ID_SQ, s > 0 ? 1u : 0u);
                    tc_mma(tmem + 128, kx(128, s), kx(0, s), ID_WIDE, s > 0 ? 1u : 0u);
                }
            });
            if (!ok) break;
            drain_store(0, S0, gs);
            drain_store(128, S1, gs);
            drain_store(256, S2, gs);
            // A^2 blocks: C00 -> [0,128), C10 -> [128,256), C11 -> [256,384)
            ok = run([&] {
                for (int s = 0; s < 8; ++s) tc_mma(tmem, ks(S0, s), ks(S0, s), ID_SQ, s > 0 ? 1u : 0u);
                for (int s = 0; s < 8; ++s) tc_mma(tmem, ms(S1, s), ms(S1, s), ID_TT, 1u);
                for (int s = 0; s < 8; ++s) tc_mma(tmem + 128, ks(S1, s), ks(S0, s), ID_SQ, s > 0 ? 1u : 0u);
                for (int s = 0; s < 8; ++s) tc_mma(tmem + 128, ks(S2, s), ms(S1, s), ID_KT, 1u);
                for (int s = 0; s < 8; ++s) tc_mma(tmem + 256, ks(S1, s), ks(S1, s), ID_SQ, s > 0 ? 1u : 0u);
                for (int s = 0; s < 8; ++s) tc_mma(tmem + 256, ks(S2, s), ks(S2, s), ID_SQ, 1u);
            });
            if (!ok) break;
            drain_poly(0, S0, S0, true);
            drain_poly(128, S1, S1, false);
            drain_poly(256, S2, S2, true);
            // X <- P X: M-half h -> TMEM [256 h, 256 h + 64 nck); P01 = P10^T
            ok = run([&] {
                for (int h = 0; h < 2; ++h)
                    for (int kb = 0; kb < 2; ++kb) {
                        const uint8_t* Pblk = (h == 0) ? (kb == 0 ? S0 : S1) : (kb == 0 ? S1 : S2);
                        const bool tr = (h == 0 && kb == 1);
                        for (int s = 0; s < 8; ++s)
                            tc_mma(tmem + 256 * h, tr ? ms(Pblk, s) : ks(Pblk, s), mx(128 * kb + 16 * s, 0),
                                   tr ? id_px_t : id_px, (kb | s) ? 1u : 0u);
                    }
            });
            if (!ok) break;
            const float alpha = first ? inv : 1.0f;
            if (!last) {
                drain_x(0, 0, alpha);
                drain_x(256, 128, alpha);
            } else {
                write_out(a, bk, e, X, tlane, 0, alpha, nck);
                write_out(a, bk, e, X, tlane + 256, 128, alpha, nck);
            }
        }
    }
    fence_async_smem();         // the next prologue refills the slots on the copy engine
    __syncthreads();
    return ok;
}

// Item k of this CTA: its bucket and matrix index.
__device__ __forceinline__ void item_at(const SmallArgs& a, int k, int& bi, int& b) {
    if (a.cta_ptr) {
        const int it = a.items[k];
        bi = it >> 24;
        b = it & 0xFFFFFF;
    } else {
        bi = 0;
        b = blockIdx.x + k * (int)gridDim.x;
    }
}

__global__ void __launch_bounds__(NT, 1) small_ns_kernel(const __grid_constant__ SmallArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Ctx c;
    c.X = base;
    c.S0 = base + X_BYTES;
    c.S1 = c.S0 + S_BYTES;
    c.S2 = c.S1 + S_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(c.S2 + S_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 4);     // bar[0] products, bar[1..3] stages
    c.red = reinterpret_cast<float*>(tmem_slot + 2);
    c.inv_s = c.red + 8;
    c.tid = threadIdx.x;
    c.warp = c.tid >> 5;
    c.lane = c.tid & 31;
    c.hw = c.warp >> 2;
    c.r = 32 * (c.warp & 3) + c.lane;                              // this thread's TMEM lane
    c.barA = smem_u32(bar);

    if (c.tid == 0) {
        for (int i = 0; i < 4; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(c.barA + 8 * i) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (c.warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem = *tmem_slot;
    c.tlane = c.tmem + ((uint32_t)(32 * (c.warp & 3)) << 16);
    c.phase = 0;
    c.stream = Stream{c.barA + 8, smem_u32(c.S0), stream_stages(a), 0u, 0u};
    pdl_wait();          // the caller's matrices may come from the previous kernel
    pdl_trigger();

    int k0, k1;
    if (a.cta_ptr) {
        k0 = a.cta_ptr[blockIdx.x];
        k1 = a.cta_ptr[blockIdx.x + 1];
    } else {
        k0 = 0;
        k1 = (a.bk[0].batch - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    }
    bool ok = true;
    for (int k = k0; k < k1 && ok; ++k) {
        int bi, b;
        item_at(a, k, bi, b);
        const MatEntry* nx = nullptr;
        int64_t nx_elems = 0;
        if (k + 1 < k1) {
            int nbi, nb;
            item_at(a, k + 1, nbi, nb);
            nx = a.bk[nbi].mats + nb;
            nx_elems = (int64_t)a.bk[nbi].m * a.bk[nbi].n;
        }
        const SmallBucket& bk = a.bk[bi];
        ok = bk.m > 128 ? process<256>(a, bk, b, nx, nx_elems, c) : process<128>(a, bk, b, nx, nx_elems, c);
    }

    if (!ok) {
        if (c.tid == 0) {
            atomicOr(a.status, STATUS_TIMEOUT);
            tc_commit(c.barA);              // wait (bounded) for the products in flight
            wait_limited(c.barA, c.phase);
            for (uint32_t k = c.stream.consumed; k < c.stream.issued; ++k) {   // and the staged loads
                if (a.stall && k == (uint32_t)(a.stall - 1) && blockIdx.x == 0) continue;   // never issued
                wait_limited(c.stream.bars + 8 * (k % c.stream.nst), (k / c.stream.nst) & 1u);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (c.warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(c.tmem) : "memory");
    }
}

}  // namespace small

bool small_ns_fits(int m, int n, int nseg, const int* segs) {
    if (m < 1 || n < m || nseg < 1 || nseg > 8) return false;
    if (m <= 128) {
        if (n > 512) return false;
        for (int i = 0; i < nseg; ++i)
            if (segs[i] < 1 || segs[i] > 2) return false;
        return true;
    }
    if (m <= 256) {                 // plain NS only
        if (n > 256) return false;
        for (int i = 0; i < nseg; ++i)
            if (segs[i] != 1) return false;
        return true;
    }
    return false;
}

cudaError_t launch_small_ns(const SmallArgs& a, int num_sms, cudaStream_t s) {
    static cudaError_t attr = cudaFuncSetAttribute(small::small_ns_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   small::SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    if (a.nb < 1 || a.nb > SMALL_MAX_BUCKETS || a.param_dtype != MUON_BF16) return cudaErrorInvalidValue;
    for (int i = 0; i < a.nb; ++i) {
        const SmallBucket& bk = a.bk[i];
        if (!small_ns_fits(bk.m, bk.n, bk.nseg, bk.segs) || bk.batch < 1 || bk.batch >= (1 << 24))
            return cudaErrorInvalidValue;
    }
    int grid;
    if (a.cta_ptr) {
        if (!a.items || a.grid < 1 || a.grid > num_sms) return cudaErrorInvalidValue;
        grid = a.grid;
    } else {
        if (a.nb != 1) return cudaErrorInvalidValue;
        grid = a.bk[0].batch < num_sms ? a.bk[0].batch : num_sms;
    }
    return launch_pdl(small::small_ns_kernel, dim3(grid), dim3(small::NT), (size_t)small::SMEM_BYTES, s, a);
}

}  // namespace muon
