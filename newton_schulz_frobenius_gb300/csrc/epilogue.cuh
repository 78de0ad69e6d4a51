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

// Storage codes: MUON_F32 (and DT_TF32, fp32 storage), MUON_BF16, MUON_F16.
__device__ __forceinline__ float ld_elem(const void* p, int64_t i, int dtype) {
    if (dtype == MUON_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p)[i]);
    if (dtype == MUON_F16) return __half2float(reinterpret_cast<const __half*>(p)[i]);
    return reinterpret_cast<const float*>(p)[i];
}

__device__ __forceinline__ void st_elem(void* p, int64_t i, float v, int dtype) {
    if (dtype == MUON_BF16) reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
    else if (dtype == MUON_F16) reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
    else reinterpret_cast<float*>(p)[i] = v;
}

// Eight 16-bit values (bf16 or fp16, round to nearest even) in one 16-byte word.
__device__ __forceinline__ uint4 pack8_h(const float* v, bool f16) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (f16) {
            __half2 h = __floats2half2_rn(v[2 * k], v[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        } else {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void unpack8_h(const uint4 q, float* v, bool f16) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = f16 ? __half22float2(*reinterpret_cast<const __half2*>(&w[k]))
                             : __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
        v[2 * k] = f.x;
        v[2 * k + 1] = f.y;
    }
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
    if (dtype == MUON_F16) {
        __half* p = reinterpret_cast<__half*>(base) + off;
        if ((W % 8) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < W; j += 8) *reinterpret_cast<uint4*>(p + j) = pack8_h(v + j, true);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) p[j] = __float2half_rn(v[j]);
        }
    } else if (dtype == MUON_BF16) {
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

// Loads W contiguous values (all < N, row < M) into v, with 16-byte vector
// loads when the address allows it.
template <int W>
__device__ __forceinline__ void load_row_run(const void* base, int64_t off, float (&v)[W], int dtype) {
    if (dtype == MUON_F16) {
        const __half* p = reinterpret_cast<const __half*>(base) + off;
        if ((W % 8) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < W; j += 8) unpack8_h(*reinterpret_cast<const uint4*>(p + j), v + j, true);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) v[j] = __half2float(p[j]);
        }
    } else if (dtype == MUON_BF16) {
        const __nv_bfloat16* p = reinterpret_cast<const __nv_bfloat16*>(base) + off;
        if ((W % 8) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < W; j += 8) {
                const uint4 u = *reinterpret_cast<const uint4*>(p + j);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[k]));
                    v[j + 2 * k] = f.x;
                    v[j + 2 * k + 1] = f.y;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) v[j] = __bfloat162float(p[j]);
        }
    } else {
        const float* p = reinterpret_cast<const float*>(base) + off;
        if ((W % 4) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < W; j += 4) {
                const float4 f = *reinterpret_cast<const float4*>(p + j);
                v[j] = f.x; v[j + 1] = f.y; v[j + 2] = f.z; v[j + 3] = f.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) v[j] = p[j];
        }
    }
}

// A tall caller matrix (stored n x m, oriented (r, c) at c m + r) is read and
// written a caller row per lane: the warp's 32 x 32 chunk (rows r0.., columns
// c0..) is handled in its transpose, lane j owning caller row c0 + j, elements
// r0 .. r0+31, as 64 contiguous bytes.  Only for whole chunks whose rows start
// on 16 bytes (the condition is the same for every lane of the warp).
__device__ __forceinline__ bool trans_vec_chunk(const GemmArgs& a, const MatEntry& e, int r0, int c0) {
    const int es = a.out_dtype == MUON_F32 ? 4 : 2;
    return e.trans && r0 + 32 <= a.M && c0 + 32 <= a.N && ((int64_t)a.M * es) % 16 == 0 &&
           (reinterpret_cast<uintptr_t>(e.w) & 15) == 0;
}

// In-register transpose of a warp's 32 x 32 tile (lane i holds row i on entry,
// column i on return): five rounds of exchanges with the lane whose index
// differs in bit k, swapping the k-wide blocks that are out of place.
__device__ __forceinline__ void warp_transpose32(float (&v)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 16; k >= 1; k >>= 1) {
        const bool up = (lane & k) != 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j & k) continue;
            const float x = __shfl_xor_sync(0xffffffffu, up ? v[j] : v[j + k], k);
            if (up) v[j] = x;
            else v[j + k] = x;
        }
    }
}

// Loads, for one thread's row r and columns c0 .. c0+W-1, the values the
// epilogue will combine with the product: G for EPI_POLY, the caller's W for
// EPI_UPDATE (nothing otherwise).  Split from epi_row_chunk so a caller can
// issue the next chunk's loads before it processes the current one.
template <int W>
__device__ __forceinline__ void epi_load_chunk(const GemmArgs& a, const MatEntry& e, int b, int r, int c0,
                                               float (&g)[W]) {
    if (r >= a.M) return;
    const int nvalid = min(W, a.N - c0);
    if (nvalid <= 0) return;
    if (a.epi == EPI_POLY) {
        const int64_t goff = (int64_t)b * a.strideG + (int64_t)r * a.ldg + c0;
        if (nvalid == W) {
            load_row_run<W>(a.Gin, goff, g, a.dtype);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) g[j] = (j < nvalid) ? ld_elem(a.Gin, goff + j, a.dtype) : 0.f;
        }
    } else if (a.epi == EPI_UPDATE) {
        const int od = a.out_dtype;
        if (!e.trans) {
            const int64_t off = (int64_t)r * a.N + c0;
            if (nvalid == W) {
                load_row_run<W>(e.w, off, g, od);
            } else {
#pragma unroll
                for (int j = 0; j < W; ++j) g[j] = (j < nvalid) ? ld_elem(e.w, off + j, od) : 0.f;
            }
        } else if (W == 32 && trans_vec_chunk(a, e, r - (threadIdx.x & 31), c0)) {
            // transposed chunk: this lane's caller row c0 + lane, elements r0 .. r0+31
            const int lane = threadIdx.x & 31;
            load_row_run<W>(e.w, (int64_t)(c0 + lane) * a.M + (r - lane), g, od);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j) g[j] = (j < nvalid) ? ld_elem(e.w, (int64_t)(c0 + j) * a.M + r, od) : 0.f;
        }
    }
}

// One thread, one row r, columns c0 .. c0+W-1, scale s (epi_alpha), table
// entry e (EPI_UPDATE / EPI_OUT) and the chunk's preloaded values g
// (epi_load_chunk).  Row runs use 16-byte vector stores; the mirrored half of
// a symmetric product and the caller's matrix of a tall (transposed) bucket
// are written column by column, which is coalesced across the 32 lanes of a
// warp because the lanes of a tensor-core epilogue warp own 32 consecutive rows.
template <int W, bool MIRROR = true>
__device__ __forceinline__ void epi_row_chunk(const GemmArgs& a, const MatEntry& e, int b, int r, int c0,
                                              float (&v)[W], float s, const float (&g)[W]) {
    if (r >= a.M) return;
    const int nvalid = min(W, a.N - c0);
    if (nvalid <= 0) return;
#pragma unroll
    for (int j = 0; j < W; ++j) v[j] *= s;

    if (a.epi == EPI_STORE || a.epi == EPI_POLY) {
        const int64_t cbase = (int64_t)b * a.strideC;
        const int cd = a.c_dtype;
        if (a.epi == EPI_POLY) {
#pragma unroll
            for (int j = 0; j < W; ++j) v[j] = a.pc * v[j] + a.pb * g[j] + ((c0 + j) == r ? a.pa : 0.f);
        }
        if (a.round_tf32) {
#pragma unroll
            for (int j = 0; j < W; ++j) v[j] = round_tf32(v[j]);
        }
        const int64_t roff = cbase + (int64_t)r * a.ldc + c0;
        const bool full_row = (nvalid == W) && (!a.symmetric || c0 + W - 1 <= r);
        if (full_row) {
            store_row_run<W>(a.C, roff, v, cd);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j)
                if (j < nvalid && (!a.symmetric || c0 + j <= r)) st_elem(a.C, roff + j, v[j], cd);
        }
        if (MIRROR && a.symmetric) {
#pragma unroll
            for (int j = 0; j < W; ++j)
                if (j < nvalid && c0 + j < r) st_elem(a.C, cbase + (int64_t)(c0 + j) * a.ldc + r, v[j], cd);
        }
        return;
    }

    // EPI_UPDATE / EPI_OUT: the caller's matrix through the table entry
    const int od = a.out_dtype;
    const float lr = a.hyper ? a.hyper[0] : a.lr;
    const float wd = a.hyper ? a.hyper[2] : a.wd;
    const float lrwd = lr * wd;
    const float step = lr * a.scale;
    if constexpr (W == 32) {
        if (trans_vec_chunk(a, e, r - (threadIdx.x & 31), c0)) {
            // tall caller matrix, whole chunk: transposed in registers, then one
            // caller row per lane (g was loaded in that layout by epi_load_chunk)
            const int lane = threadIdx.x & 31;
            warp_transpose32(v);
            if (a.epi == EPI_UPDATE) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = g[j] - fmaf(lrwd, g[j], step * v[j]);
            }
            store_row_run<32>(e.w, (int64_t)(c0 + lane) * a.M + (r - lane), v, od);
            return;
        }
    }
    if (a.epi == EPI_UPDATE) {
        // W - (lr wd W + step O): the decrement is formed first and subtracted
        // once, so an fp32-rounded factor (1 - lr wd) never scales every W
#pragma unroll
        for (int j = 0; j < W; ++j) v[j] = g[j] - fmaf(lrwd, g[j], step * v[j]);
    }
    if (!e.trans) {
        const int64_t off = (int64_t)r * a.N + c0;
        if (nvalid == W) {
            store_row_run<W>(e.w, off, v, od);
        } else {
#pragma unroll
            for (int j = 0; j < W; ++j)
                if (j < nvalid) st_elem(e.w, off + j, v[j], od);
        }
    } else {
        // caller matrix is n x m: oriented (r, c) lives at c * m + r
#pragma unroll
        for (int j = 0; j < W; ++j)
            if (j < nvalid) st_elem(e.w, (int64_t)(c0 + j) * a.M + r, v[j], od);
    }
}

// Mirrored half of a symmetric product for one warp's 32 x 32 chunk (rows
// r0.., columns c0..): element (r, c) with c < r is also written to (c, r).
// The warp's final values v (lane = row) go through a 32 x 33 fp32 staging
// area, then every lane writes one 8-column segment of a mirrored row, so a
// store instruction covers 8 rows x 64 bytes (bf16) instead of one column.
// The staging layout is bank-conflict-free for the row writes (bank
// lane + j) and for the column reads (bank 8s + k + i).
__device__ __forceinline__ void epi_mirror_staged(const GemmArgs& a, int b, int r0, int c0, const float (&v)[32],
                                                  float (*stage)[33]) {
    const int lane = threadIdx.x & 31;
    if (c0 >= r0 + 31) return;              // no element of the chunk lies strictly below the diagonal
#pragma unroll
    for (int j = 0; j < 32; ++j) stage[lane][j] = v[j];
    __syncwarp();
    const int64_t cbase = (int64_t)b * a.strideC;
    const int sg = lane & 3;
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
        const int i = pass * 8 + (lane >> 2);    // mirrored row c0 + i
        const int c = c0 + i;
        const int rb = r0 + 8 * sg;              // its columns rb .. rb+7 (rows of the chunk)
        float w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = stage[8 * sg + k][i];
        if (c < a.N) {
            const int64_t off = cbase + (int64_t)c * a.ldc + rb;
            if (c < rb && rb + 7 < a.M) {
                store_row_run<8>(a.C, off, w, a.c_dtype);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (rb + k < a.M && c < rb + k) st_elem(a.C, off + k, w[k], a.c_dtype);
            }
        }
    }
    __syncwarp();
}

// Workspace products (EPI_STORE / EPI_POLY) of one warp's 32 x 32 chunk
// (rows r0 + lane, columns c0..) through the 32 x 33 staging area: the final
// values are staged once, then both the rows and (symmetric) the mirrored
// rows leave as 8-column segments, four lanes per 64-byte row piece, so every
// store transaction is a whole 32-byte sector (a lane writing 16 bytes of its
// own row costs one half-sector transaction per lane).  Symmetric products
// keep (r, c) with c <= r and mirror c < r to (c, r).
__device__ __forceinline__ void epi_store_staged(const GemmArgs& a, int b, int r0, int c0, float (&v)[32], float s,
                                                 const float (&g)[32], float (*stage)[33]) {
    const int lane = threadIdx.x & 31;
    const int r = r0 + lane;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= s;
    if (a.epi == EPI_POLY) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = a.pc * v[j] + a.pb * g[j] + ((c0 + j) == r ? a.pa : 0.f);
    }
    if (a.round_tf32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = round_tf32(v[j]);
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) stage[lane][j] = v[j];
    __syncwarp();
    const int64_t cbase = (int64_t)b * a.strideC;
    const int sg = lane & 3;
    // rows: pass p writes rows r0 + 8p + lane / 4, columns c0 + 8 sg ..
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
        const int i = pass * 8 + (lane >> 2);
        const int rr = r0 + i, cc = c0 + 8 * sg;
        if (rr < a.M && cc < a.N) {
            float w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = stage[i][8 * sg + k];
            const int64_t off = cbase + (int64_t)rr * a.ldc + cc;
            if (cc + 7 < a.N && (!a.symmetric || cc + 7 <= rr)) {
                store_row_run<8>(a.C, off, w, a.c_dtype);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (cc + k < a.N && (!a.symmetric || cc + k <= rr)) st_elem(a.C, off + k, w[k], a.c_dtype);
            }
        }
    }
    // mirrored rows: pass p writes row c0 + 8p + lane / 4, columns r0 + 8 sg ..
    if (a.symmetric && c0 < r0 + 31) {
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
            const int i = pass * 8 + (lane >> 2);    // mirrored row c0 + i
            const int c = c0 + i;
            const int rb = r0 + 8 * sg;              // its columns rb .. rb+7 (rows of the chunk)
            float w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = stage[8 * sg + k][i];
            if (c < a.N) {
                const int64_t off = cbase + (int64_t)c * a.ldc + rb;
                if (c < rb && rb + 7 < a.M) {
                    store_row_run<8>(a.C, off, w, a.c_dtype);
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (rb + k < a.M && c < rb + k) st_elem(a.C, off + k, w[k], a.c_dtype);
                }
            }
        }
    }
    __syncwarp();
}

// Convenience for callers without pipelining: scale, table entry and loads
// for one chunk, then the epilogue.
template <int W>
__device__ __forceinline__ void epi_row_chunk_once(const GemmArgs& a, int b, int r, int c0, float (&v)[W]) {
    MatEntry e{};
    if (a.epi == EPI_UPDATE || a.epi == EPI_OUT) e = a.mats[b];
    float g[W];
    epi_load_chunk<W>(a, e, b, r, c0, g);
    epi_row_chunk<W>(a, e, b, r, c0, v, epi_alpha(a, b), g);
}

}  // namespace muon

