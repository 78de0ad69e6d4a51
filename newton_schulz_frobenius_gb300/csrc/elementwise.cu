// Elementwise kernels of the Muon update: momentum (+Nesterov), orientation
// into the workspace, Frobenius partial sums, and the norm finalisation (by
// the last CTA to finish each matrix).
//
// Momentum smooths the gradient before Newton-Schulz ("MuonX" page, section 2);
// the Frobenius normalisation places every singular value at or below 1 before
// the iteration.  On the bf16 and fp32 paths the scale 1/(||U||_F + eps) is not
// applied here: it is folded into the first XX^T (as its square) and the first
// Q X of the NS path, so U is read and written exactly once.  fp16 has too
// little range for an unscaled U (small gradients fall into its subnormals),
// so the fp16 path runs the kernel twice: a first pass that only sums U^2, and
// a second that updates the momentum and stores U / (||U||_F + eps).
//
// Layout: one CTA handles a 64 x 64 tile of the ORIENTED matrix (m <= n).  For
// a tall caller matrix (trans = 1) the CTA reads the matching transposed tile of
// the caller's rows (coalesced), writes momentum back in the caller's layout,
// and transposes through shared memory so the workspace write is coalesced too.
#include "muon_internal.cuh"
#include "epilogue.cuh"

#include <algorithm>

namespace muon {

namespace {

constexpr int PT = 64;          // tile edge

__host__ __device__ __forceinline__ int prep_tiles(int m, int n) { return ((m + PT - 1) / PT) * ((n + PT - 1) / PT); }
constexpr int PTHREADS = 256;   // 64 rows x 4 segments of 16 elements

__device__ __forceinline__ void load16(const void* p, int dtype, int64_t off, int valid, bool vec,
                                       float (&v)[16]) {
    if (vec && valid == 16) {
        if (dtype == MUON_F16) {
            const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(p) + off);
            unpack8_h(__ldg(q), v, true);
            unpack8_h(__ldg(q + 1), v + 8, true);
        } else if (dtype == MUON_BF16) {
            const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p) + off);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 u = __ldg(q + h);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&w[k]);
                    float2 f = __bfloat1622float2(b2);
                    v[h * 8 + 2 * k] = f.x;
                    v[h * 8 + 2 * k + 1] = f.y;
                }
            }
        } else {
            const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + off);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                float4 f = __ldg(q + h);
                v[4 * h] = f.x; v[4 * h + 1] = f.y; v[4 * h + 2] = f.z; v[4 * h + 3] = f.w;
            }
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = (j < valid) ? ld_elem(p, off + j, dtype) : 0.f;
}

__device__ __forceinline__ void store16(void* p, int dtype, int64_t off, int valid, bool vec,
                                        const float (&v)[16]) {
    if (vec && valid == 16) {
        store_row_run<16>(p, off, v, dtype);
        return;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (j < valid) st_elem(p, off + j, v[j], dtype);
}

// Sum of one matrix's nparts partial sums of squares by a 256-thread block, in
// double and in a fixed order (eight independent loads in flight per thread,
// then warp and block sums); the total is returned to thread 0.
__device__ double sum_partials_256(const float* pb, int nparts, double* red) {
    double s = 0.0;
    for (int i0 = threadIdx.x; i0 < nparts; i0 += 256 * 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + 256 * u;
            v[u] = i < nparts ? __ldcg(pb + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) s += (double)v[u];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0)
        for (int w = 0; w < 8; ++w) t += red[w];
    return t;
}

// One 64 x 64 tile of the oriented matrix b: momentum, U into X, and this
// thread's sum of squares of U added to ss.
__device__ __forceinline__ void prep_tile(const PrepArgs& a, const MatEntry& e, int b, int tile_idx, float beta,
                                          int nesterov, float (*tile)[PT + 1], float& ss) {
    const int tiles_c = (a.n + PT - 1) / PT;
    const int tr = tile_idx / tiles_c;
    const int tc = tile_idx % tiles_c;
    const int lr = threadIdx.x >> 2;          // row within the tile
    const int seg = (threadIdx.x & 3) * 16;   // first of 16 columns
    const bool vec = a.vec_ok != 0;
    // Raw (caller) coordinates of this thread's 16 elements.
    int raw_r, raw_c0, raw_rows, raw_cols;
    if (!e.trans) {
        raw_rows = a.m; raw_cols = a.n;
        raw_r = tr * PT + lr; raw_c0 = tc * PT + seg;
    } else {
        raw_rows = a.n; raw_cols = a.m;
        raw_r = tc * PT + lr; raw_c0 = tr * PT + seg;
    }
    int valid = 0;
    if (raw_r < raw_rows) valid = max(0, min(16, raw_cols - raw_c0));
    const int64_t off = (int64_t)raw_r * raw_cols + raw_c0;

    float u[16];
    if (valid > 0) {
        float g[16];
        load16(e.grad, a.in_dtype, off, valid, vec, g);
        if (a.with_momentum) {
            float mo[16];
            load16(e.mom, a.mom_dtype, off, valid, vec, mo);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float mn = fmaf(beta, mo[j], g[j]);            // M' = beta M + G
                mo[j] = mn;
                u[j] = nesterov ? fmaf(beta, mn, g[j]) : mn;         // U = G + beta M'
            }
            // momentum is stored in its own dtype; U continues from the fp32 M'
            if (a.write_mom) store16(e.mom, a.mom_dtype, off, valid, vec, mo);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) u[j] = g[j];
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j < valid) ss = fmaf(u[j], u[j], ss);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) u[j] = 0.f;
    }

    const int64_t xb = (int64_t)b * a.strideX;
    const bool xvec = (a.ldx % 8) == 0;
    if (a.x_scale) {
        const float xs = a.x_scale[b];
#pragma unroll
        for (int j = 0; j < 16; ++j) u[j] *= xs;
    }
    if (!a.write_x) {
        // first pass of the fp16 path: sums only
    } else if (!e.trans) {
        if (valid > 0) store16(a.X, a.x_dtype, xb + (int64_t)raw_r * a.ldx + raw_c0, valid, xvec, u);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) tile[lr][seg + j] = u[j];
        __syncthreads();
        // oriented row = tr*64 + lr2, columns tc*64 + seg2 .. +16  <- tile[col][row]
        const int orow = tr * PT + lr;
        const int ocol0 = tc * PT + seg;
        int ovalid = 0;
        if (orow < a.m) ovalid = max(0, min(16, a.n - ocol0));
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = tile[seg + j][lr];
        __syncthreads();        // the tile is read before the next one overwrites it
        if (ovalid > 0) store16(a.X, a.x_dtype, xb + (int64_t)orow * a.ldx + ocol0, ovalid, xvec, x);
    }
}


// Grid (parts, batch): CTA p of matrix b takes the tiles p, p + parts, ... and
// writes one partial sum of squares.
// Five CTAs per SM (46 registers, no spills) instead of the four 64 registers
// allowed: more loads in flight, 9% less time on the 24-layer stack's prologue.
__global__ void __launch_bounds__(PTHREADS, 5)
prep_kernel(const __grid_constant__ PrepArgs a) {
    __shared__ float tile[PT][PT + 1];
    __shared__ float red[PTHREADS / 32];

    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.y;
    const MatEntry e = a.mats[b];
    const float beta = a.hyper ? a.hyper[1] : a.beta;
    const int nesterov = a.hyper ? (a.hyper[3] != 0.f) : a.nesterov;
    const int ntiles = prep_tiles(a.m, a.n);
    float ss = 0.f;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) prep_tile(a, e, b, t, beta, nesterov, tile, ss);

    // Block sum of squares -> one partial per CTA.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < PTHREADS / 32; ++w) t += red[w];
        a.partials[(int64_t)b * a.nparts + blockIdx.x] = t;
    }
    if (!a.counter) return;
    // The CTA that completes matrix b's count turns its partials into the
    // scale 1/(||U||_F + eps) (summed in double in a fixed order) and resets
    // the count for the next launch.
    __shared__ int s_last;
    __shared__ double dred[PTHREADS / 32];
    if (threadIdx.x == 0) {
        __threadfence();
        s_last = (atomicAdd(a.counter + b, 1) == a.nparts - 1) ? 1 : 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const double t = sum_partials_256(a.partials + (int64_t)b * a.nparts, a.nparts, dred);
    if (threadIdx.x == 0) {
        if (!isfinite(t)) atomicOr(a.status, STATUS_NONFINITE);
        a.inv[b] = (float)(1.0 / (sqrt(t) + (double)a.eps));
        a.counter[b] = 0;
    }
}

__device__ __forceinline__ uint32_t hash32(uint32_t x) {
    x ^= x >> 16; x *= 0x7feb352du;
    x ^= x >> 15; x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

__global__ void fill_synthetic_kernel(void* X, int64_t count, int dtype, float scale, uint32_t seed) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * blockDim.x) {
        uint32_t h = hash32((uint32_t)i * 2654435761u ^ seed ^ (uint32_t)(i >> 32));
        float v = ((float)(h >> 8) * (1.0f / 16777216.0f) * 2.0f - 1.0f) * scale;
        st_elem(X, i, v, dtype);
    }
}

}  // namespace

int prep_num_parts(int m, int n) { return prep_tiles(m, n); }

int prep_grid_parts(int m, int n, int batch) {
    // 8 tiles per CTA, 16 when that still gives at least eight waves of five
    // CTAs per SM (152 SMs): long enough to amortise a CTA's set-up and its partial sum,
    // short enough that the last wave of a launch stays small.  Measured
    // against the earlier rule of about 2048 CTAs per launch: the 2560x9728
    // prologue 0.57 -> 0.60 of the HBM copy rate, the 7B stack's 0.76 -> 0.79.
    // Launches of fewer than 8 x 760 tiles take fewer tiles per CTA, down to
    // one, so that they still spread over the SMs: one 256x1024 fp32 matrix
    // (64 tiles) ran on 8 CTAs in 28 us.
    const int t = prep_tiles(m, n);
    const int64_t total = (int64_t)t * batch;
    int64_t tpc = total >= (int64_t)16 * 760 * 8 ? 16 : 8;
    if (total < (int64_t)8 * 760) tpc = std::max<int64_t>(1, total / 760);
    return (int)((t + tpc - 1) / tpc);
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
    dim3 grid(a.nparts, a.batch);
    return launch_pdl(prep_kernel, grid, dim3(PTHREADS), 0, s, a);
}

cudaError_t launch_fill_synthetic(void* X, int64_t count, int dtype, float scale, uint32_t seed,
                                  cudaStream_t s) {
    int64_t nb = (count + 255) / 256;
    int blocks = (int)(nb < 4096 ? nb : 4096);
    if (blocks < 1) blocks = 1;
    fill_synthetic_kernel<<<blocks, 256, 0, s>>>(X, count, dtype, scale, seed);
    return cudaGetLastError();
}

}  // namespace muon
