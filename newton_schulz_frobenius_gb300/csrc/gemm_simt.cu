// fp32 products of the Newton-Schulz path on the FFMA pipe.
//
// The fp32 path must hold a 1e-4 relative error against the fp64 reference;
// TF32 tensor-core inputs (10-bit mantissa) give about 3e-3 on a 256 x 1024
// matrix, so these products use true fp32 multiply-adds.  Tile 64 x 64, k-steps
// of 64, 256 threads, 4 x 4 outputs per thread; symmetric products launch only
// the lower-triangle tiles and mirror on store (see epilogue.cuh).
//
// The fp32 workload's products have few tiles (10 to 64 for a 256 x 1024
// matrix) against 152 SMs, so a launch is bound by the serial k-loop of each
// tile, not by the FFMA rate.  Such products split K over a cluster of S CTAs
// (S = 2, 4 or 8): CTA q of a cluster sums its own contiguous k-range, leaves
// the 64 x 64 partial tile in its shared memory, and after a cluster barrier
// CTA r adds rows [64r/S, 64(r+1)/S) of the S partials, always in the order
// q = 0 .. S-1, read through distributed shared memory, and stores them.  The
// result depends on the shape alone, never on scheduling.  Within a k-range
// each output sums its terms in order, one fused multiply-add at a time; each
// thread holds the next k-step's operands in registers (16-byte loads where
// the rows allow) while the current one is multiplied out of shared memory.
//
// Products with at least one 128 x 128 tile per SM take a second kernel:
// tiles of 128 x 128, k-steps of 16, 8 x 8 outputs per thread (four 16-byte
// shared-memory reads per 64 multiply-adds instead of two per 16), the
// operand tiles double-buffered in shared memory with the next k-step held
// in registers, one block barrier per k-step, two CTAs per SM (128
// registers a thread).
#include "muon_internal.cuh"
#include "epilogue.cuh"

namespace muon {

namespace {

constexpr int ST = 64;
constexpr int SK = 64;
constexpr int MAX_SPLIT = 8;   // portable cluster size

__device__ __forceinline__ void tri_decode(int l, int& tm, int& tn) {
    int t = (int)((sqrtf(8.0f * (float)l + 1.0f) - 1.0f) * 0.5f);
    while (t * (t + 1) / 2 > l) --t;
    while ((t + 1) * (t + 2) / 2 <= l) ++t;
    tm = t;
    tn = l - t * (t + 1) / 2;
}

__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16 bytes of CTA `rank`'s shared memory at the address `local` has in this CTA.
__device__ __forceinline__ float4 ld_cluster_f4(const void* local, uint32_t rank) {
    const uint32_t addr = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t raddr;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(addr), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(raddr) : "memory");
    return v;
}

// Four consecutive fp32 values at p[0..3] of a row with `valid` elements left
// (zero beyond); one 16-byte load when all four exist and vec allows it,
// else one load per element.
__device__ __forceinline__ float4 load4(const float* p, int valid, bool vec) {
    if (vec && valid >= 4) return __ldg(reinterpret_cast<const float4*>(p));
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid > 0) v.x = __ldg(p);
    if (valid > 1) v.y = __ldg(p + 1);
    if (valid > 2) v.z = __ldg(p + 2);
    if (valid > 3) v.w = __ldg(p + 3);
    return v;
}

// This thread's four 16-byte pieces of the k-step at k0 (k < kend): A
// (row-major, K contiguous) and B (K-major: N x K; otherwise K x N) as 64 x 64
// tiles.  K-contiguous pieces: row (idx & 63), columns 4 (idx >> 6) ..;
// N-contiguous pieces (B stored K x N): row k = idx >> 4, columns 4 (idx & 15) ..
template <bool B_KMAJOR>
__device__ __forceinline__ void load_kstep(const GemmArgs& a, const float* A, const float* B, int row0, int col0,
                                           int k0, int kend, bool vecA, bool vecB, float4 (&ra)[4],
                                           float4 (&rb)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int idx = threadIdx.x + i * 256;
        const int r = idx & 63, k = k0 + 4 * (idx >> 6);
        const int gr = row0 + r;
        ra[i] = (gr < a.M) ? load4(A + (int64_t)gr * a.lda + k, kend - k, vecA) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (B_KMAJOR) {
            const int gc = col0 + r;
            rb[i] = (gc < a.N) ? load4(B + (int64_t)gc * a.ldb + k, kend - k, vecB) : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            const int kk = k0 + (idx >> 4), c = col0 + 4 * (idx & 15);
            rb[i] = (kk < kend) ? load4(B + (int64_t)kk * a.ldb + c, a.N - c, vecB) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

// grid.x = tiles x split (the split CTAs of a tile adjacent, one cluster),
// grid.y = batch; kc = k-range per CTA (a multiple of 4).
template <bool B_KMAJOR>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const __grid_constant__ GemmArgs a, int tiles_m, int split, int kc) {
    __shared__ __align__(16) float As[SK][ST + 4];
    __shared__ __align__(16) float Bs[SK][ST + 4];

    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y;
    const int q = blockIdx.x % split;         // this CTA's k-range (its rank in the cluster)
    const int tile = blockIdx.x / split;
    int tm, tn;
    if (a.symmetric) tri_decode(tile, tm, tn);
    else { tm = tile % tiles_m; tn = tile / tiles_m; }

    const float* A = reinterpret_cast<const float*>(a.A) + (int64_t)b * a.strideA;
    const float* B = reinterpret_cast<const float*>(a.B) + (int64_t)b * a.strideB;
    const bool vecA = (a.lda % 4 == 0) && (a.strideA % 4 == 0 || a.batch == 1) &&
                      (reinterpret_cast<uintptr_t>(a.A) & 15) == 0;
    const bool vecB = (a.ldb % 4 == 0) && (a.strideB % 4 == 0 || a.batch == 1) &&
                      (reinterpret_cast<uintptr_t>(a.B) & 15) == 0;
    const int row0 = tm * ST, col0 = tn * ST;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int kbeg = min(a.K, q * kc), kend = min(a.K, kbeg + kc);

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    float4 ra[4], rb[4];
    if (kbeg < kend) load_kstep<B_KMAJOR>(a, A, B, row0, col0, kbeg, kend, vecA, vecB, ra, rb);
    for (int k0 = kbeg; k0 < kend; k0 += SK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = threadIdx.x + i * 256;
            const int r = idx & 63, k = 4 * (idx >> 6);
            As[k][r] = ra[i].x; As[k + 1][r] = ra[i].y; As[k + 2][r] = ra[i].z; As[k + 3][r] = ra[i].w;
            if (B_KMAJOR) {
                Bs[k][r] = rb[i].x; Bs[k + 1][r] = rb[i].y; Bs[k + 2][r] = rb[i].z; Bs[k + 3][r] = rb[i].w;
            } else {
                *reinterpret_cast<float4*>(&Bs[idx >> 4][4 * (idx & 15)]) = rb[i];
            }
        }
        __syncthreads();
        // the next k-step's operands travel while this one is multiplied out
        if (k0 + SK < kend) load_kstep<B_KMAJOR>(a, A, B, row0, col0, k0 + SK, kend, vecA, vecB, ra, rb);
        // shared-memory fragments one k ahead of the multiply-adds
        float4 av = *reinterpret_cast<const float4*>(&As[0][ty * 4]);
        float4 bv = *reinterpret_cast<const float4*>(&Bs[0][tx * 4]);
#pragma unroll 16
        for (int kk = 0; kk < SK; ++kk) {
            const int kn = (kk + 1) & (SK - 1);
            const float4 an = *reinterpret_cast<const float4*>(&As[kn][ty * 4]);
            const float4 bn = *reinterpret_cast<const float4*>(&Bs[kn][tx * 4]);
            const float ar[4] = {av.x, av.y, av.z, av.w};
            const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
            av = an;
            bv = bn;
        }
        __syncthreads();
    }

    if (split == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v[4] = {acc[i][0], acc[i][1], acc[i][2], acc[i][3]};
            epi_row_chunk_once<4>(a, b, row0 + ty * 4 + i, col0 + tx * 4, v);
        }
        return;
    }

    // the partial tile goes to As (free after the loop's last barrier)
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(&As[ty * 4 + i][tx * 4]) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    cluster_barrier();
    const int rows = ST / split;              // rows of the tile this CTA finishes
    for (int t = threadIdx.x; t < rows * (ST / 4); t += blockDim.x) {
        const int r = q * rows + t / (ST / 4), c = 4 * (t % (ST / 4));
        float4 s = ld_cluster_f4(&As[r][c], 0);
        for (int p = 1; p < split; ++p) {
            const float4 t = ld_cluster_f4(&As[r][c], (uint32_t)p);
            s.x += t.x; s.y += t.y; s.z += t.z; s.w += t.w;
        }
        float v[4] = {s.x, s.y, s.z, s.w};
        epi_row_chunk_once<4>(a, b, row0 + r, col0 + c, v);
    }
    // no CTA leaves while the others may still read its partial tile
    cluster_barrier();
}


// ---- large products: 128 x 128 tiles, 8 x 8 outputs per thread ----

constexpr int BT = 128;
constexpr int BKS = 16;
constexpr int BIG_LOADS = BT * BKS / 4 / 256;                        // 16-byte pieces per thread per operand
// two buffers of A and B, as dynamic shared memory (the form ptxas allocates
// registers best for)
constexpr int BIG_SMEM = 2 * 2 * BKS * (BT + 4) * (int)sizeof(float);

template <bool B_KMAJOR>
__device__ __forceinline__ void big_load(const GemmArgs& a, const float* A, const float* B, int row0, int col0,
                                         int k0, bool vecA, bool vecB, float4 (&ra)[BIG_LOADS],
                                         float4 (&rb)[BIG_LOADS]) {
    constexpr int KQ = BKS / 4;                 // 16-byte pieces along K per row
#pragma unroll
    for (int i = 0; i < BIG_LOADS; ++i) {
        const int idx = threadIdx.x + 256 * i;
        const int r = idx / KQ, k = k0 + 4 * (idx % KQ);
        ra[i] = (row0 + r < a.M) ? load4(A + (int64_t)(row0 + r) * a.lda + k, a.K - k, vecA)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        if (B_KMAJOR) {
            rb[i] = (col0 + r < a.N) ? load4(B + (int64_t)(col0 + r) * a.ldb + k, a.K - k, vecB)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            const int kk = k0 + (idx >> 5), c = col0 + 4 * (idx & 31);
            rb[i] = (kk < a.K) ? load4(B + (int64_t)kk * a.ldb + c, a.N - c, vecB) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}

template <bool B_KMAJOR>
__device__ __forceinline__ void big_store(float (*As)[BT + 4], float (*Bs)[BT + 4], const float4 (&ra)[BIG_LOADS],
                                          const float4 (&rb)[BIG_LOADS]) {
    constexpr int KQ = BKS / 4;
#pragma unroll
    for (int i = 0; i < BIG_LOADS; ++i) {
        const int idx = threadIdx.x + 256 * i;
        const int r = idx / KQ, k = 4 * (idx % KQ);
        As[k][r] = ra[i].x; As[k + 1][r] = ra[i].y; As[k + 2][r] = ra[i].z; As[k + 3][r] = ra[i].w;
        if (B_KMAJOR) {
            Bs[k][r] = rb[i].x; Bs[k + 1][r] = rb[i].y; Bs[k + 2][r] = rb[i].z; Bs[k + 3][r] = rb[i].w;
        } else {
            *reinterpret_cast<float4*>(&Bs[idx >> 5][4 * (idx & 31)]) = rb[i];
        }
    }
}

template <bool B_KMAJOR>
__global__ void __launch_bounds__(256, 2)
gemm_simt_big_kernel(const __grid_constant__ GemmArgs a, int tiles_m) {
    extern __shared__ __align__(16) float big_smem[];
    auto As = reinterpret_cast<float (*)[BKS][BT + 4]>(big_smem);
    auto Bs = reinterpret_cast<float (*)[BKS][BT + 4]>(big_smem + 2 * BKS * (BT + 4));

    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y;
    int tm, tn;
    if (a.symmetric) tri_decode(blockIdx.x, tm, tn);
    else { tm = blockIdx.x % tiles_m; tn = blockIdx.x / tiles_m; }
    const float* A = reinterpret_cast<const float*>(a.A) + (int64_t)b * a.strideA;
    const float* B = reinterpret_cast<const float*>(a.B) + (int64_t)b * a.strideB;
    const bool vecA = (a.lda % 4 == 0) && (a.strideA % 4 == 0 || a.batch == 1) &&
                      (reinterpret_cast<uintptr_t>(a.A) & 15) == 0;
    const bool vecB = (a.ldb % 4 == 0) && (a.strideB % 4 == 0 || a.batch == 1) &&
                      (reinterpret_cast<uintptr_t>(a.B) & 15) == 0;
    const int row0 = tm * BT, col0 = tn * BT;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    float4 ra[BIG_LOADS], rb[BIG_LOADS];
    big_load<B_KMAJOR>(a, A, B, row0, col0, 0, vecA, vecB, ra, rb);
    big_store<B_KMAJOR>(As[0], Bs[0], ra, rb);
    __syncthreads();
    int buf = 0;
    for (int k0 = 0; k0 < a.K; k0 += BKS) {
        const bool more = k0 + BKS < a.K;
        if (more) big_load<B_KMAJOR>(a, A, B, row0, col0, k0 + BKS, vecA, vecB, ra, rb);
#pragma unroll
        for (int kk = 0; kk < BKS; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][64 + ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][64 + tx * 4]);
            const float ar[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float br[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
        }
        if (more) {
            // the other buffer was last read one k-step ago, before the barrier below it
            big_store<B_KMAJOR>(As[buf ^ 1], Bs[buf ^ 1], ra, rb);
            __syncthreads();
            buf ^= 1;
        }
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int r = row0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        float v0[4] = {acc[i][0], acc[i][1], acc[i][2], acc[i][3]};
        float v1[4] = {acc[i][4], acc[i][5], acc[i][6], acc[i][7]};
        epi_row_chunk_once<4>(a, b, r, col0 + tx * 4, v0);
        epi_row_chunk_once<4>(a, b, r, col0 + 64 + tx * 4, v1);
    }
}

}  // namespace

// Split of K for a launch of `tiles` output tiles: doubled while the CTAs fit
// twice over on the SMs (two 256-thread CTAs per SM) and every CTA keeps at
// least one full k-step.
int simt_split(int64_t tiles, int K, int num_sms) {
    int split = 1;
    while (split < MAX_SPLIT && tiles * 2 * split <= 2 * (int64_t)num_sms && K / (2 * split) >= SK) split *= 2;
    return split;
}

cudaError_t launch_gemm_simt(const GemmArgs& a, int num_sms, cudaStream_t s) {
    {
        const int bm = (a.M + BT - 1) / BT, bn = (a.N + BT - 1) / BT;
        const int per = a.symmetric ? bm * (bm + 1) / 2 : bm * bn;
        if ((int64_t)per * a.batch >= num_sms) {
            static_assert(BIG_SMEM <= 48 * 1024, "dynamic shared memory above the default limit");
            dim3 grid(per, a.batch);
            if (a.b_kmajor) launch_pdl(gemm_simt_big_kernel<true>, grid, dim3(256), (size_t)BIG_SMEM, s, a, bm);
            else launch_pdl(gemm_simt_big_kernel<false>, grid, dim3(256), (size_t)BIG_SMEM, s, a, bm);
            return cudaGetLastError();
        }
    }
    const int tiles_m = (a.M + ST - 1) / ST;
    const int tiles_n = (a.N + ST - 1) / ST;
    const int per_batch = a.symmetric ? tiles_m * (tiles_m + 1) / 2 : tiles_m * tiles_n;
    const int split = simt_split((int64_t)per_batch * a.batch, a.K, num_sms);
    const int kc = ((a.K + split - 1) / split + 3) & ~3;
    auto kern = a.b_kmajor ? gemm_simt_kernel<true> : gemm_simt_kernel<false>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(per_batch * split, a.batch);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = split;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, a, tiles_m, split, kc);
}

}  // namespace muon
