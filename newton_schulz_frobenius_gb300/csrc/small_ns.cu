// Whole Muon update of one small matrix per CTA, for buckets of many small
// matrices ("DMuon" summary, section 2.2: matrices too small to fill the GPU
// are grouped by shape and their recursion runs jointly to amortise launch
// overhead).  One launch processes the whole bucket: CTAs loop over the
// bucket's matrices and each runs
//   momentum (+Nesterov) -> Frobenius norm -> NS (plain, or Gram with segments
//   of length <= 2) -> fused update (or the ortho output)
// without leaving the SM: X (oriented m x n, m <= 128, n <= 512) lives in
// shared memory as eight 128 x 64 bf16 chunks in the 128-byte-swizzled
// K-major layout, the m x m Gram-space matrices in three 128 x 128 bf16 slots
// of the same layout, and every product accumulates in TMEM (512 columns):
//   XX^T, G^2, PG, (PG)P, PQ : M = N = 128, both operands K-major
//   Q X                      : M = 128, N <= 256 per instruction, X read
//                              MN-major from the same chunks
// Rows m..127 and columns n.. of X are zero, so the padding contributes
// nothing.  Eight warps: thread 0 issues the tcgen05.mma instructions; all
// warps run the prologue and drain TMEM (two warps per TMEM lane quarter).
#include "muon_internal.cuh"
#include "epilogue.cuh"

namespace muon {
namespace small {

constexpr int NT = 256;
constexpr int CHUNK = 128 * 128;            // bytes of one 128-row x 64-column bf16 chunk
constexpr int X_BYTES = 8 * CHUNK;          // n <= 512
constexpr int S_BYTES = 2 * CHUNK;          // one 128 x 128 Gram-space slot
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

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

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

// Byte offset of element (r, c) in a chunked 128-row K-major region: chunk
// c / 64, row r at 128 B, 16-byte unit (c % 64) / 8 XOR-swizzled by r % 8 (the
// layout a TMA load with 128-byte swizzle produces).
__device__ __forceinline__ uint32_t swz(int r, int c) {
    const int cc = c & 63;
    return (uint32_t)((c >> 6) * CHUNK + r * 128 + ((((cc >> 3) ^ (r & 7)) << 4) | ((cc & 7) << 1)));
}

// Stores 32 values (columns c0..c0+31, c0 % 32 == 0) of row r as bf16.
__device__ __forceinline__ void st_row32(uint8_t* region, int r, int c0, const float (&v)[32]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        uint4 q;
        __nv_bfloat162 h0 = __floats2bfloat162_rn(v[8 * u + 0], v[8 * u + 1]);
        __nv_bfloat162 h1 = __floats2bfloat162_rn(v[8 * u + 2], v[8 * u + 3]);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * u + 4], v[8 * u + 5]);
        __nv_bfloat162 h3 = __floats2bfloat162_rn(v[8 * u + 6], v[8 * u + 7]);
        q.x = *reinterpret_cast<uint32_t*>(&h0);
        q.y = *reinterpret_cast<uint32_t*>(&h1);
        q.z = *reinterpret_cast<uint32_t*>(&h2);
        q.w = *reinterpret_cast<uint32_t*>(&h3);
        *reinterpret_cast<uint4*>(region + swz(r, c0 + 8 * u)) = q;
    }
}

}  // namespace small
}  // namespace muon

namespace muon {
namespace small {

__device__ __forceinline__ void load8(const void* p, int64_t off, int dtype, float (&v)[8]) {
    if (dtype == MUON_BF16) {
        const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p) + off);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
            v[2 * k] = f.x;
            v[2 * k + 1] = f.y;
        }
    } else {
        const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + off);
        const float4 f0 = q[0], f1 = q[1];
        v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w;
        v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
    }
}

__device__ __forceinline__ void store8(void* p, int64_t off, int dtype, const float (&v)[8]) {
    float t[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) t[k] = v[k];
    store_row_run<8>(p, off, t, dtype);
}

// U of one matrix (momentum update when a.mode == 0) into X; returns this
// thread's sum of squares of U.
__device__ float prologue(const SmallArgs& a, const MatEntry& e, uint8_t* X) {
    const int tid = threadIdx.x;
    const int raw_rows = e.trans ? a.n : a.m;
    const int raw_cols = e.trans ? a.m : a.n;
    const int64_t total = (int64_t)raw_rows * raw_cols;
    const bool step = (a.mode == 0);
    const float beta = a.hyper ? a.hyper[1] : a.beta;
    const int nesterov = a.hyper ? (a.hyper[3] != 0.f) : a.nesterov;
    float ss = 0.f;
    auto put = [&](int rr, int cc, const float (&u)[8], int cnt) {
        if (!e.trans && cnt == 8) {
            uint4 q;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(u[0], u[1]);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(u[2], u[3]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(u[4], u[5]);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(u[6], u[7]);
            q.x = *reinterpret_cast<uint32_t*>(&h0);
            q.y = *reinterpret_cast<uint32_t*>(&h1);
            q.z = *reinterpret_cast<uint32_t*>(&h2);
            q.w = *reinterpret_cast<uint32_t*>(&h3);
            *reinterpret_cast<uint4*>(X + swz(rr, cc)) = q;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (k < cnt) {
                    const int r = e.trans ? cc + k : rr;
                    const int c = e.trans ? rr : cc + k;
                    *reinterpret_cast<__nv_bfloat16*>(X + swz(r, c)) = __float2bfloat16_rn(u[k]);
                }
            }
        }
    };
    if (a.vec_ok) {
        constexpr int U = 4;
        for (int64_t base = (int64_t)tid * 8; base < total; base += (int64_t)NT * 8 * U) {
            float g[U][8], mo[U][8];
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                const int64_t e0 = base + (int64_t)uu * NT * 8;
                if (e0 < total) {
                    load8(e.grad, e0, a.param_dtype, g[uu]);
                    if (step) load8(e.mom, e0, a.mom_dtype, mo[uu]);
                }
            }
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                const int64_t e0 = base + (int64_t)uu * NT * 8;
                if (e0 >= total) break;
                float u[8];
                if (step) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float mn = fmaf(beta, mo[uu][k], g[uu][k]);
                        mo[uu][k] = mn;
                        u[k] = nesterov ? fmaf(beta, mn, g[uu][k]) : mn;
                    }
                    store8(e.mom, e0, a.mom_dtype, mo[uu]);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) u[k] = g[uu][k];
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) ss = fmaf(u[k], u[k], ss);
                put((int)(e0 / raw_cols), (int)(e0 % raw_cols), u, 8);
            }
        }
    } else {
        for (int64_t i = tid; i < total; i += NT) {
            const float g = ld_elem(e.grad, i, a.param_dtype);
            float u = g;
            if (step) {
                const float mn = fmaf(beta, ld_elem(e.mom, i, a.mom_dtype), g);
                st_elem(e.mom, i, mn, a.mom_dtype);
                u = nesterov ? fmaf(beta, mn, g) : mn;
            }
            ss = fmaf(u, u, ss);
            float uv[8] = {u, 0, 0, 0, 0, 0, 0, 0};
            put((int)(i / raw_cols), (int)(i % raw_cols), uv, 1);
        }
    }
    return ss;
}

__global__ void __launch_bounds__(NT, 1) small_ns_kernel(const __grid_constant__ SmallArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* X = base;
    uint8_t* S0 = base + X_BYTES;
    uint8_t* S1 = S0 + S_BYTES;
    uint8_t* S2 = S1 + S_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(S2 + S_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
    float* red = reinterpret_cast<float*>(tmem_slot + 2);     // 8 warp partials
    float* inv_s = red + 8;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, hw = warp >> 2;
    const int r = 32 * q + lane;                                // this thread's row (TMEM lane)
    const uint32_t barA = smem_u32(bar);

    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(barA) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tlane = tmem + ((uint32_t)(32 * q) << 16);
    pdl_wait();          // the caller's matrices may come from the previous kernel
    pdl_trigger();

    const int nck = (a.n + 63) / 64;            // X chunks in use
    constexpr uint32_t ID_SQ = idesc_bf16(128, 128, false);
    uint32_t phase = 0;
    bool ok = true;

    // One product round: make this thread's smem writes visible to the tensor
    // cores, let thread 0 issue, wait for completion (bounded).
    auto run = [&](auto&& issue) -> bool {
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            issue();
            tc_commit(barA);
        }
        const bool done = wait_limited(barA, phase);
        phase ^= 1u;
        const bool all = __syncthreads_and(done ? 1 : 0) != 0;
        tc_fence_after();
        return all;
    };
    auto kdesc = [&](const uint8_t* region, int s) {   // K-major operand, k-step s (16 elements)
        return sdesc(smem_u32(region) + (s >> 2) * CHUNK + (s & 3) * 32, 16, 1024);
    };
    auto square = [&](const uint8_t* A, const uint8_t* B, uint32_t col) {
        return run([&] {
            for (int s = 0; s < 8; ++s) tc_mma(tmem + col, kdesc(A, s), kdesc(B, s), ID_SQ, s > 0 ? 1u : 0u);
        });
    };
    // 128 x 128 result in TMEM columns [src, src+128) -> bf16 slot; poly: P = aI + b*gs*G + c*acc
    auto drain_sq = [&](uint32_t src, uint8_t* dst, float scale, bool poly, float gs) {
        for (int k = 0; k < 2; ++k) {
            const int c0 = 64 * hw + 32 * k;
            float v[32];
            tmem_ld32(tlane + src + c0, v);
            if (poly) {
                float g[32];
                tmem_ld32(tlane + 0 + c0, g);
                // the linear term uses the same bf16 G that the G^2 product
                // consumed: a P mixing an fp32 G with a bf16 G^2 loses the
                // cancellation a + b s^2 + c s^4 relies on near s = 1
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float gb = __bfloat162float(__float2bfloat16_rn(gs * g[j]));
                    v[j] = a.c * v[j] + a.b * gb + ((c0 + j) == r ? a.a : 0.f);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= scale;
            }
            st_row32(dst, r, c0, v);
        }
    };

    for (int b = blockIdx.x; b < a.batch && ok; b += gridDim.x) {
        const MatEntry e = a.mats[b];
        // zero the chunks of X in use, and start pulling this matrix's W into L2
        for (int i = tid; i < nck * (CHUNK / 16); i += NT) reinterpret_cast<uint4*>(X)[i] = make_uint4(0, 0, 0, 0);
        if (a.mode == 0) {
            const int64_t wbytes = (int64_t)a.m * a.n * 2;
            for (int64_t off = (int64_t)tid * 128; off < wbytes; off += (int64_t)NT * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(e.w) + off));
        }
        __syncthreads();
        float ss = prologue(a, e, X);
        // while this matrix iterates, pull the next one's inputs into L2
        if (b + (int)gridDim.x < a.batch) {
            const MatEntry nx = a.mats[b + gridDim.x];
            const int64_t elems = (int64_t)a.m * a.n;
            const int64_t gbytes = elems * (a.param_dtype == MUON_BF16 ? 2 : 4);
            const int64_t mbytes = elems * (a.mom_dtype == MUON_BF16 ? 2 : 4);
            for (int64_t off = (int64_t)tid * 128; off < gbytes; off += (int64_t)NT * 128)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(nx.grad) + off));
            if (a.mode == 0)
                for (int64_t off = (int64_t)tid * 128; off < mbytes; off += (int64_t)NT * 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(nx.mom) + off));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        if (tid == 0) {
            double t = 0.0;
            for (int w = 0; w < NT / 32; ++w) t += (double)red[w];
            if (!isfinite(t)) atomicOr(a.status, STATUS_NONFINITE);
            *inv_s = (float)(1.0 / (sqrt(t) + 1e-7));
        }
        __syncthreads();
        const float inv = *inv_s;

        for (int si = 0; si < a.nseg && ok; ++si) {
            const int L = a.segs[si];
            const bool first = (si == 0), last = (si == a.nseg - 1);
            const float gs = first ? inv * inv : 1.0f;
            // G = X X^T -> TMEM [0, 128) -> S0
            ok = run([&] {
                for (int s = 0; s < nck * 4; ++s) tc_mma(tmem, kdesc(X, s), kdesc(X, s), ID_SQ, s > 0 ? 1u : 0u);
            });
            if (!ok) break;
            drain_sq(0, S0, gs, false, 1.f);
            // P1 = aI + bG + cG^2 -> S1
            ok = square(S0, S0, 128);
            if (!ok) break;
            drain_sq(128, S1, 1.f, true, gs);
            uint8_t* Q = S1;
            if (L == 2) {
                ok = square(S1, S0, 256);                 // P1 G -> S2
                if (!ok) break;
                drain_sq(256, S2, 1.f, false, 1.f);
                ok = square(S2, S1, 0);                   // (P1 G) P1 = G' -> TMEM [0,128), S0
                if (!ok) break;
                drain_sq(0, S0, 1.f, false, 1.f);
                ok = square(S0, S0, 128);                 // P2 = aI + bG' + cG'^2 -> S2
                if (!ok) break;
                drain_sq(128, S2, 1.f, true, 1.f);
                ok = square(S2, S1, 256);                 // Q = P2 P1 -> S0
                if (!ok) break;
                drain_sq(256, S0, 1.f, false, 1.f);
                Q = S0;
            }
            // X <- Q X : TMEM [0, 64*nck)
            ok = run([&] {
                for (int h = 0; h < 2; ++h) {
                    const int nh = min(256, nck * 64 - 256 * h);
                    if (nh <= 0) break;
                    const uint32_t id = idesc_bf16(128, nh, true);
                    for (int s = 0; s < 8; ++s) {
                        const uint64_t bd =
                            sdesc(smem_u32(X) + (4 * h) * CHUNK + s * 2048, CHUNK, 1024);
                        tc_mma(tmem + 256 * h, kdesc(Q, s), bd, id, s > 0 ? 1u : 0u);
                    }
                }
            });
            if (!ok) break;
            const float alpha = first ? inv : 1.0f;
            if (!last) {
                for (int k = hw; k < nck * 2; k += 2) {
                    float v[32];
                    tmem_ld32(tlane + 32 * k, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= alpha;
                    st_row32(X, r, 32 * k, v);
                }
            } else {
                // O (rows < m, columns < n): update the caller's W or write O
                const float lr = a.hyper ? a.hyper[0] : a.lr;
                const float wd = a.hyper ? a.hyper[2] : a.wd;
                const float lrwd = lr * wd;
                const float stepc = lr * a.scale;
                const int od = a.param_dtype;
                for (int k = hw; k < nck * 2; k += 2) {
                    const int c0 = 32 * k;
                    float v[32];
                    tmem_ld32(tlane + c0, v);
                    if (r >= a.m || c0 >= a.n) continue;
                    const int nv = min(32, a.n - c0);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= alpha;
                    if (!e.trans) {
                        const int64_t off = (int64_t)r * a.n + c0;
                        if (a.mode == 0) {
                            float w[32];
                            if (nv == 32) load_row_run<32>(e.w, off, w, od);
                            else
                                for (int j = 0; j < 32; ++j) w[j] = j < nv ? ld_elem(e.w, off + j, od) : 0.f;
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = w[j] - fmaf(lrwd, w[j], stepc * v[j]);
                        }
                        if (nv == 32) store_row_run<32>(e.w, off, v, od);
                        else
                            for (int j = 0; j < nv; ++j) st_elem(e.w, off + j, v[j], od);
                    } else {
                        float w[32];
                        if (a.mode == 0) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                w[j] = j < nv ? ld_elem(e.w, (int64_t)(c0 + j) * a.m + r, od) : 0.f;
                        }
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (j < nv) {
                                const float o = a.mode == 0 ? w[j] - fmaf(lrwd, w[j], stepc * v[j]) : v[j];
                                st_elem(e.w, (int64_t)(c0 + j) * a.m + r, o, od);
                            }
                        }
                    }
                }
            }
        }
        __syncthreads();
    }

    if (!ok) {
        if (tid == 0) {
            atomicOr(a.status, STATUS_TIMEOUT);
            tc_commit(barA);                // wait (bounded) for the products in flight
            wait_limited(barA, phase);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

}  // namespace small

bool small_ns_fits(int m, int n, int nseg, const int* segs) {
    if (m < 1 || m > 128 || n < m || n > 512 || nseg < 1 || nseg > 16) return false;
    for (int i = 0; i < nseg; ++i)
        if (segs[i] < 1 || segs[i] > 2) return false;
    return true;
}

cudaError_t launch_small_ns(const SmallArgs& a, int num_sms, cudaStream_t s) {
    static cudaError_t attr = cudaFuncSetAttribute(small::small_ns_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   small::SMEM_BYTES);
    if (attr != cudaSuccess) return attr;
    if (!small_ns_fits(a.m, a.n, a.nseg, a.segs) || a.batch < 1) return cudaErrorInvalidValue;
    if (a.param_dtype != MUON_BF16) return cudaErrorInvalidValue;
    const int grid = a.batch < num_sms ? a.batch : num_sms;
    return launch_pdl(small::small_ns_kernel, dim3(grid), dim3(small::NT), (size_t)small::SMEM_BYTES, s, a);
}

}  // namespace muon
