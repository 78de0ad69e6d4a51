// Operand split for fp32 products on the TF32 tensor path (three passes).
//
// An fp32 value x is written as hi + lo, hi the nearest TF32 value of x and lo
// the nearest TF32 value of the exact remainder x - hi, so |x - hi - lo| is at
// most 2^-22 |x|.  A product A op(B) is then hi_A hi_B + hi_A lo_B + lo_A hi_B
// up to the dropped lo_A lo_B term (2^-22 relative): three TF32 passes whose
// error stays near fp32's, against about 1e-3 for one TF32 pass.  The three
// passes run as ONE tensor-core product over a tripled K: this kernel writes
// A' = [hi_A | hi_A | lo_A] and B' = [hi_B | lo_B | hi_B], both K-major with
// each third padded to a multiple of 4 elements (16-byte rows), so that
// A' B'^T is the three-pass sum.  B given K x N (N contiguous) is transposed
// on the way, since the TF32 tensor path reads K-major operands only.
#include "muon_internal.cuh"
#include "epilogue.cuh"

namespace muon {

namespace {

__device__ __forceinline__ void split_store(float* row, int64_t Kp, int k, float x, int order) {
    const float hi = round_tf32(x);
    const float lo = round_tf32(x - hi);
    row[k] = hi;
    row[Kp + k] = order == SPLIT_HHL ? hi : lo;
    row[2 * Kp + k] = order == SPLIT_HHL ? lo : hi;
}

// Source rows x K, K contiguous: four consecutive k per thread.
__global__ void __launch_bounds__(256) split_rows_kernel(const __grid_constant__ SplitArgs p) {
    const float* src = reinterpret_cast<const float*>(p.src) + (int64_t)blockIdx.y * p.stride_src;
    float* dst = p.dst + (int64_t)blockIdx.y * p.stride_dst;
    const int64_t q4 = p.Kp / 4;
    const int64_t total = (int64_t)p.rows * q4;
    const bool vec = (p.ld_src % 4 == 0) && (p.stride_src % 4 == 0 || gridDim.y == 1) &&
                     (reinterpret_cast<uintptr_t>(p.src) & 15) == 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / q4);
        const int k = 4 * (int)(i % q4);
        const float* s = src + (int64_t)r * p.ld_src + k;
        float v[4];
        if (vec && k + 4 <= p.K) {
            const float4 t = __ldg(reinterpret_cast<const float4*>(s));
            v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = (k + j < p.K) ? __ldg(s + j) : 0.f;
        }
        float* row = dst + (int64_t)r * (3 * p.Kp);
        float hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hi[j] = round_tf32(v[j]);
            lo[j] = round_tf32(v[j] - hi[j]);
        }
        const float4 H = make_float4(hi[0], hi[1], hi[2], hi[3]);
        const float4 L = make_float4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<float4*>(row + k) = H;
        *reinterpret_cast<float4*>(row + p.Kp + k) = p.order == SPLIT_HHL ? H : L;
        *reinterpret_cast<float4*>(row + 2 * p.Kp + k) = p.order == SPLIT_HHL ? L : H;
    }
}

// Source K x rows, rows contiguous: 32 x 32 tiles transposed through shared
// memory, so both the reads and the writes are coalesced.
__global__ void __launch_bounds__(256) split_cols_kernel(const __grid_constant__ SplitArgs p) {
    __shared__ float tile[32][33];
    const float* src = reinterpret_cast<const float*>(p.src) + (int64_t)blockIdx.z * p.stride_src;
    float* dst = p.dst + (int64_t)blockIdx.z * p.stride_dst;
    const int k0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int k = k0 + ty + 8 * j, r = r0 + tx;
        tile[ty + 8 * j][tx] = (k < p.K && r < p.rows) ? __ldg(src + (int64_t)k * p.ld_src + r) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = r0 + ty + 8 * j, k = k0 + tx;
        if (r < p.rows && k < p.Kp) split_store(dst + (int64_t)r * (3 * p.Kp), p.Kp, k, tile[tx][ty + 8 * j], p.order);
    }
}

}  // namespace

cudaError_t launch_tf32_split(const SplitArgs& p, int num_sms, cudaStream_t s) {
    if (p.rows < 1 || p.K < 1 || p.batch < 1 || p.batch > 65535 || (p.Kp % 4) || p.Kp < p.K)
        return cudaErrorInvalidValue;
    if ((reinterpret_cast<uintptr_t>(p.dst) & 15) || (p.stride_dst % 4)) return cudaErrorInvalidValue;
    if (!p.transposed) {
        const int64_t chunks = (int64_t)p.rows * (p.Kp / 4);
        int64_t blocks = (chunks + 255) / 256;
        const int64_t cap = (int64_t)num_sms * 8 / p.batch + 1;
        if (blocks > cap) blocks = cap;
        split_rows_kernel<<<dim3((unsigned)blocks, p.batch), 256, 0, s>>>(p);
    } else {
        const int64_t gx = (p.Kp + 31) / 32, gy = ((int64_t)p.rows + 31) / 32;
        if (gy > 65535) return cudaErrorInvalidValue;
        split_cols_kernel<<<dim3((unsigned)gx, (unsigned)gy, p.batch), 256, 0, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace muon
