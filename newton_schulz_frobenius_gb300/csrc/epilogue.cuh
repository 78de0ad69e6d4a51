// Product epilogues shared by the tensor-core (bf16) and FFMA (fp32) kernels.
//
// A thread owns W consecutive accumulator columns c0 .. c0+W-1 of one row r of
// matrix b and hands them to epi_row_chunk, which applies the per-batch scale
// and one of the epilogues of the Newton-Schulz update:
//   EPI_STORE   workspace product (XX^T, P G, P Q, Q X ...)
//   EPI_POLY    P = aI + bG + cG^2 fused into the G^2 product
//   EPI_UPDATE  W' = W (1 - lr wd) - lr * s * O fused into the last Q X
//   EPI_OUT     O written to the caller's matrix (orthogonalize entry point)
// Symmetric products write only c <= r and mirror c < r to (c, r).
#pragma once

#include "muon_internal.cuh"

namespace muon {

__device__ __forceinline__ float ld_elem(const void* p, int64_t i, int dtype) {
    if (dtype == MUON_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
    return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ void st_elem(void* p, int64_t i, float v, int dtype) {
    if (dtype == MUON_BF16) reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    else reinterpret_cast<float*>(p)[i] = v;
}

// Nearest TF32 value (10 explicit mantissa bits), ties to even, on the fp32
// bit pattern; finite inputs only (the NS path keeps its values bounded).
__device__ __forceinline__ float round_tf32(float v) {
    uint32_t u = __float_as_uint(v);
    u = (u + 0xFFFu + ((u >> 13) & 1u)) & ~0x1FFFu;
    return __uint_as_float(u);
}

__device__ __forceinline__ float epi_alpha(const GemmArgs& a, int b) {
    float s = a.alpha;
    if (a.alpha_vec) {
        float v = a.alpha_vec[b];
        s *= a.alpha_sq ? v * v : v;
    }
    return s;
}

// Stores W contiguous values of row r starting at column c0 (all < N, row < M)
// with 16-byte vector stores when the address allows it.
template <int W>
__device__ __forceinline__ void store_row_run(void* base, int64_t off, const float (&v)[W], int dtype) {
    if (dtype == MUON_BF16) {
        __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(base) + off;
        if ((W % 8) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < W; j += 8) {
                __nv_bfloat162 q0 = __floats2bfloat162_rn(v[j + 0], v[j + 1]);
                __nv_bfloat162 q1 = __floats2bfloat162_rn(v[j + 2], v[j + 3]);
                __nv_bfloat162 q2 = __floats2bfloat162_rn(v[j + 4], v[j + 5]);
                __nv_bfloat162 q3 = __floats2bfloat162_rn(v[j + 6], v[j + 7]);
                uint4 u;
                u.x = *reinterpret_cast<uint32_t*>(&q0);
                u.y = *reinterpret_cast<uint32_t*>(&q1);
                u.z = *reinterpret_cast<uint32_t*>(&q2);
                u.w = *reinterpret_cast<uint32_t*>(&q3);
                *reinterpret_cast<uint4*>(p + j) = u;
            }
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) p[j] = __float2bfloat16_rn(v[j]);
        }
    } else {
        float* p = reinterpret_cast<float*>(base) + off;
        if ((W % 4) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < W; j += 4)
                *reinterpret_cast<float4*>(p + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) p[j] = v[j];
        }
    }
}

template <int W>
__device__ __forceinline__ void epi_row_chunk(const GemmArgs& a, int b, int r, int c0, float (&v)[W]) {
    if (r >= a.M) return;
    const float s = epi_alpha(a, b);
    const int nvalid = min(W, a.N - c0);
    if (nvalid <= 0) return;

    if (a.epi == EPI_STORE || a.epi == EPI_POLY) {
        const int64_t cbase = (int64_t)b * a.strideC;
        const int cd = a.c_dtype;
        if (a.epi == EPI_POLY) {
            const int64_t gbase = (int64_t)b * a.strideG + (int64_t)r * a.ldg + c0;
#pragma unroll
            for (int j = 0; j < W; ++j) {
                if (j < nvalid) {
                    float g = ld_elem(a.Gin, gbase + j, a.dtype);
                    v[j] = a.pc * (s * v[j]) + a.pb * g + ((c0 + j) == r ? a.pa : 0.f);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) v[j] *= s;
        }
        if (a.round_tf32) {
#pragma unroll
            for (int j = 0; j < W; ++j) v[j] = round_tf32(v[j]);
        }
        if (a.symmetric) {
#pragma unroll
            for (int j = 0; j < W; ++j) {
                const int c = c0 + j;
                if (j < nvalid && c <= r) {
                    st_elem(a.C, cbase + (int64_t)r * a.ldc + c, v[j], cd);
                    if (c < r) st_elem(a.C, cbase + (int64_t)c * a.ldc + r, v[j], cd);
                }
            }
        } else if (nvalid == W) {
            store_row_run<W>(a.C, cbase + (int64_t)r * a.ldc + c0, v, cd);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j)
                if (j < nvalid) st_elem(a.C, cbase + (int64_t)r * a.ldc + c0 + j, v[j], cd);
        }
        return;
    }

    // EPI_UPDATE / EPI_OUT: caller matrices through the table.
    const MatEntry e = a.mats[b];
    const int od = a.out_dtype;
    if (a.epi == EPI_OUT) {
        if (!e.trans) {
#pragma unroll
            for (int j = 0; j < W; ++j) v[j] *= s;
            if (nvalid == W) {
                store_row_run<W>(e.w, (int64_t)r * a.N + c0, v, od);
            } else {
#pragma unroll
                for (int j = 0; j < W; ++j)
                    if (j < nvalid) st_elem(e.w, (int64_t)r * a.N + c0 + j, v[j], od);
            }
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j)
                if (j < nvalid) st_elem(e.w, (int64_t)(c0 + j) * a.M + r, s * v[j], od);
        }
        return;
    }
    // EPI_UPDATE: W' = W (1 - lr wd) - lr * scale * O
    const float keep = 1.0f - a.lr * a.wd;
    const float step = a.lr * a.scale * s;
    if (!e.trans) {
        const int64_t off = (int64_t)r * a.N + c0;
        float w[W];
#pragma unroll
        for (int j = 0; j < W; ++j) w[j] = (j < nvalid) ? ld_elem(e.w, off + j, od) : 0.f;
#pragma unroll
        for (int j = 0; j < W; ++j) w[j] = fmaf(-step, v[j], keep * w[j]);
        if (nvalid == W) {
            store_row_run<W>(e.w, off, w, od);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j)
                if (j < nvalid) st_elem(e.w, off + j, w[j], od);
        }
    } else {
#pragma unroll
        for (int j = 0; j < W; ++j) {
            if (j < nvalid) {
                const int64_t off = (int64_t)(c0 + j) * a.M + r;
                const float w = ld_elem(e.w, off, od);
                st_elem(e.w, off, fmaf(-step, v[j], keep * w), od);
            }
        }
    }
}

}  // namespace muon

namespace muon {

// Tensor-core epilogue for one warp and one 32 x 32 chunk: lane l holds row
// r0 + l, columns c0 .. c0+31 (one tcgen05.ld).  The chunk is staged through
// shared memory (stage: 32 x 33 floats owned by this warp) so that every
// global access is a 32-lane run along a row of its matrix:
//   row phase     lane l handles column c0 + l of rows r0 .. r0+31
//                 (row-major stores, the polynomial's G reads, the caller's
//                 W / O in their own orientation)
//   column phase  lane l handles row r0 + l of columns c0 .. c0+31
//                 (the mirrored half of a symmetric product, and the caller's
//                 W / O of a transposed (tall) matrix)
__device__ __forceinline__ void epi_chunk_staged(const GemmArgs& a, int b, int r0, int c0, const float (&v)[32],
                                                 float (*stage)[33]) {
    const int lane = threadIdx.x & 31;
    const float s = epi_alpha(a, b);
#pragma unroll
    for (int j = 0; j < 32; ++j) stage[lane][j] = s * v[j];
    __syncwarp();

    const int col = c0 + lane;
    const bool col_ok = col < a.N;
    const int epi = a.epi;
    if (epi == EPI_STORE || epi == EPI_POLY) {
        const int64_t cbase = (int64_t)b * a.strideC;
        const int cd = a.c_dtype;
        for (int i = 0; i < 32; ++i) {
            const int row = r0 + i;
            if (row >= a.M) break;
            if (!col_ok) continue;
            float val = stage[i][lane];
            if (epi == EPI_POLY) {
                const float g = ld_elem(a.Gin, (int64_t)b * a.strideG + (int64_t)row * a.ldg + col, a.dtype);
                val = a.pc * val + a.pb * g + (row == col ? a.pa : 0.f);
            }
            if (a.round_tf32) val = round_tf32(val);
            stage[i][lane] = val;
            if (!a.symmetric || col <= row) st_elem(a.C, cbase + (int64_t)row * a.ldc + col, val, cd);
        }
        if (a.symmetric) {
            __syncwarp();
            const int r = r0 + lane;
            if (r < a.M) {
                for (int j = 0; j < 32; ++j) {
                    const int c = c0 + j;
                    if (c >= r || c >= a.N) break;   // only strictly below the diagonal
                    st_elem(a.C, cbase + (int64_t)c * a.ldc + r, stage[lane][j], cd);
                }
            }
        }
        __syncwarp();
        return;
    }

    const MatEntry e = a.mats[b];
    const int od = a.out_dtype;
    const float keep = 1.0f - a.lr * a.wd;
    const float step = a.lr * a.scale;
    if (!e.trans) {
        // caller matrix is m x n, row-major: row phase
        for (int i = 0; i < 32; ++i) {
            const int row = r0 + i;
            if (row >= a.M) break;
            if (!col_ok) continue;
            const int64_t off = (int64_t)row * a.N + col;
            const float o = stage[i][lane];
            if (epi == EPI_OUT) {
                st_elem(e.w, off, o, od);
            } else {
                const float w = ld_elem(e.w, off, od);
                st_elem(e.w, off, fmaf(-step, o, keep * w), od);
            }
        }
    } else {
        // caller matrix is n x m (tall): element (row, col) of the oriented
        // matrix lives at col * m + row; column phase keeps lanes on a run
        const int r = r0 + lane;
        if (r < a.M) {
            for (int j = 0; j < 32; ++j) {
                const int c = c0 + j;
                if (c >= a.N) break;
                const int64_t off = (int64_t)c * a.M + r;
                const float o = stage[lane][j];
                if (epi == EPI_OUT) {
                    st_elem(e.w, off, o, od);
                } else {
                    const float w = ld_elem(e.w, off, od);
                    st_elem(e.w, off, fmaf(-step, o, keep * w), od);
                }
            }
        }
    }
    __syncwarp();
}

}  // namespace muon
