// fp32 products of the Newton-Schulz path on the FFMA pipe.
//
// The fp32 path must hold a 1e-4 relative error against the fp64 reference;
// TF32 tensor-core inputs (10-bit mantissa) give about 3e-3 on a 256 x 1024
// matrix, so these products use true fp32 multiply-adds.  Tile 64 x 64 x 16,
// 256 threads, 4 x 4 outputs per thread; symmetric products launch only the
// lower-triangle tiles and mirror on store (see epilogue.cuh).
#include "muon_internal.cuh"
#include "epilogue.cuh"

namespace muon {

namespace {

constexpr int ST = 64;
constexpr int SK = 16;

__device__ __forceinline__ void tri_decode(int l, int& tm, int& tn) {
    int t = (int)((sqrtf(8.0f * (float)l + 1.0f) - 1.0f) * 0.5f);
    while (t * (t + 1) / 2 > l) --t;
    while ((t + 1) * (t + 2) / 2 <= l) ++t;
    tm = t;
    tn = l - t * (t + 1) / 2;
}

template <bool B_KMAJOR>
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const __grid_constant__ GemmArgs a, int tiles_m) {
    __shared__ __align__(16) float As[SK][ST + 4];
    __shared__ __align__(16) float Bs[SK][ST + 4];

    const int b = blockIdx.y;
    int tm, tn;
    if (a.symmetric) tri_decode(blockIdx.x, tm, tn);
    else { tm = blockIdx.x % tiles_m; tn = blockIdx.x / tiles_m; }

    const float* A = reinterpret_cast<const float*>(a.A) + (int64_t)b * a.strideA;
    const float* B = reinterpret_cast<const float*>(a.B) + (int64_t)b * a.strideB;
    const int row0 = tm * ST, col0 = tn * ST;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < a.K; k0 += SK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int idx = threadIdx.x + i * 256;
            const int r = idx >> 4, k = idx & 15;
            const int gr = row0 + r, gk = k0 + k;
            As[k][r] = (gr < a.M && gk < a.K) ? A[(int64_t)gr * a.lda + gk] : 0.f;
            if (B_KMAJOR) {
                const int gc = col0 + r;
                Bs[k][r] = (gc < a.N && gk < a.K) ? B[(int64_t)gc * a.ldb + gk] : 0.f;
            }
        }
        if (!B_KMAJOR) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int idx = threadIdx.x + i * 256;
                const int k = idx >> 6, c = idx & 63;
                const int gk = k0 + k, gc = col0 + c;
                Bs[k][c] = (gk < a.K && gc < a.N) ? B[(int64_t)gk * a.ldb + gc] : 0.f;
            }
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SK; ++kk) {
            const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
            const float ar[4] = {av.x, av.y, av.z, av.w};
            const float br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float v[4] = {acc[i][0], acc[i][1], acc[i][2], acc[i][3]};
        epi_row_chunk_once<4>(a, b, row0 + ty * 4 + i, col0 + tx * 4, v);
    }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs& a, cudaStream_t s) {
    const int tiles_m = (a.M + ST - 1) / ST;
    const int tiles_n = (a.N + ST - 1) / ST;
    const int per_batch = a.symmetric ? tiles_m * (tiles_m + 1) / 2 : tiles_m * tiles_n;
    dim3 grid(per_batch, a.batch);
    if (a.b_kmajor) gemm_simt_kernel<true><<<grid, 256, 0, s>>>(a, tiles_m);
    else gemm_simt_kernel<false><<<grid, 256, 0, s>>>(a, tiles_m);
    return cudaGetLastError();
}

}  // namespace muon
