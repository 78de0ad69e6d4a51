// AdamW step for the parameters that stay off Muon ("MuonX" page, section 2:
// embeddings and biases keep AdamW), every tensor of the call in one launch.
//
// The host cuts the tensors into chunks of CHUNK_ELEMS elements; CTA k
// handles chunk k: 16-byte vector loads and stores where the tensor's
// pointers allow it, scalar otherwise.  Per element it reads p, g, m, v and
// writes p, m, v once, so the kernel is bound by HBM bandwidth.
//   m' = b1 m + (1 - b1) g,  v' = b2 v + (1 - b2) g^2
//   p' = p - [ lr wd p + (lr / bc1) m' / (sqrt(v') / sqrt(bc2) + eps) ]
// with bc1 = 1 - b1^t and bc2 = 1 - b2^t computed on the host in double.  The
// bracket is formed first and subtracted once: a factor (1 - lr wd) rounded to
// fp32 would carry an error of the same sign into every element, comparable
// to the update itself at small lr.
#include "host.h"
#include "epilogue.cuh"

namespace muon {

namespace {

constexpr int AT = 256;

__device__ __forceinline__ void adam8(const AdamArgs& a, float (&p)[8], const float (&g)[8], float (&m)[8],
                                      float (&v)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m[k] = fmaf(a.beta1, m[k], (1.0f - a.beta1) * g[k]);
        v[k] = fmaf(a.beta2, v[k], (1.0f - a.beta2) * g[k] * g[k]);
        const float denom = fmaf(sqrtf(v[k]), a.inv_sqrt_bc2, a.eps);
        p[k] -= fmaf(a.lr_wd, p[k], a.step_size * (m[k] / denom));
    }
}

// Five CTAs per SM (48 registers) instead of the four 60 registers allowed:
// more loads in flight, 0.91 -> 0.97 of the measured HBM copy bandwidth.
__global__ void __launch_bounds__(AT, 5) adamw_kernel(const __grid_constant__ AdamArgs a) {
    pdl_wait();
    pdl_trigger();
    const AdamChunk ch = a.chunks[blockIdx.x];
    const AdamTensor t = a.tensors[ch.tensor];
    const int pd = a.param_dtype, sd = a.state_dtype;
    const bool vec = t.vec_ok && (ch.start % 8 == 0);
    for (int i = threadIdx.x * 8; i < ch.len; i += AT * 8) {
        const int64_t off = ch.start + i;
        const int cnt = min(8, ch.len - i);
        float p[8], g[8], m[8], v[8];
        if (vec && cnt == 8) {
            load_row_run<8>(t.p, off, p, pd);
            load_row_run<8>(t.g, off, g, pd);
            load_row_run<8>(t.m, off, m, sd);
            load_row_run<8>(t.v, off, v, sd);
            adam8(a, p, g, m, v);
            store_row_run<8>(t.p, off, p, pd);
            store_row_run<8>(t.m, off, m, sd);
            store_row_run<8>(t.v, off, v, sd);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const bool in = k < cnt;
                p[k] = in ? ld_elem(t.p, off + k, pd) : 0.f;
                g[k] = in ? ld_elem(t.g, off + k, pd) : 0.f;
                m[k] = in ? ld_elem(t.m, off + k, sd) : 0.f;
                v[k] = in ? ld_elem(t.v, off + k, sd) : 0.f;
            }
            adam8(a, p, g, m, v);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (k < cnt) {
                    st_elem(t.p, off + k, p[k], pd);
                    st_elem(t.m, off + k, m[k], sd);
                    st_elem(t.v, off + k, v[k], sd);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_adamw(const AdamArgs& a, int nchunks, cudaStream_t s) {
    return launch_pdl(adamw_kernel, dim3(nchunks), dim3(AT), 0, s, a);
}

}  // namespace muon

// ---------------------------------------------------------------------------
// host entry point
// ---------------------------------------------------------------------------

using namespace muon;

// ---------------------------------------------------------------------------
// AdamW for the non-matrix parameters ("MuonX" page, section 2)
// ---------------------------------------------------------------------------

extern "C" int muon_adamw_step(void* const* params, const void* const* grads, void* const* exp_avg,
                               void* const* exp_avg_sq, const int64_t* numels, int64_t count, int param_dtype,
                               int state_dtype, float lr, float beta1, float beta2, float eps, float wd,
                               int64_t step, void* stream) try {
    if (count < 0) return fail(MUON_EINVAL, "count < 0");
    if (count == 0) return MUON_OK;
    if (!params || !grads || !exp_avg || !exp_avg_sq || !numels) return fail(MUON_EINVAL, "NULL array argument");
    if (!valid_dtype(param_dtype) || !(state_dtype == MUON_F32 || state_dtype == MUON_BF16))
        return fail(MUON_EDTYPE, "dtypes %d / %d (moments: fp32 or bf16)", param_dtype, state_dtype);
    if (step < 1) return fail(MUON_EINVAL, "step counts from 1");
    if (!std::isfinite(lr) || !std::isfinite(beta1) || !std::isfinite(beta2) || !std::isfinite(eps) ||
        !std::isfinite(wd) || beta1 < 0.f || beta1 >= 1.f || beta2 < 0.f || beta2 >= 1.f || eps < 0.f)
        return fail(MUON_EINVAL, "bad hyper-parameter");
    if (count > INT32_MAX) return fail(MUON_EINVAL, "more than 2^31 - 1 tensors");
    int64_t nchunks = 0;                        // checked before any table is built
    for (int64_t i = 0; i < count; ++i) {
        if (!params[i] || !grads[i] || !exp_avg[i] || !exp_avg_sq[i])
            return fail(MUON_EINVAL, "NULL tensor pointer at %lld", (long long)i);
        if (numels[i] < 0 || numels[i] > INT64_MAX / 16) return fail(MUON_EINVAL, "bad size at %lld", (long long)i);
        nchunks += (numels[i] + ADAM_CHUNK_ELEMS - 1) / ADAM_CHUNK_ELEMS;
        if (nchunks > INT32_MAX) return fail(MUON_EINVAL, "too many elements");
    }
    std::vector<AdamTensor> tens((size_t)count);
    std::vector<AdamChunk> chunks;
    chunks.reserve((size_t)nchunks);
    for (int64_t i = 0; i < count; ++i) {
        auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
        tens[(size_t)i] = AdamTensor{params[i], grads[i], exp_avg[i], exp_avg_sq[i],
                                     (a16(params[i]) && a16(grads[i]) && a16(exp_avg[i]) && a16(exp_avg_sq[i])) ? 1 : 0, 0};
        for (int64_t s0 = 0; s0 < numels[i]; s0 += ADAM_CHUNK_ELEMS)
            chunks.push_back(AdamChunk{s0, (int)i, (int)std::min<int64_t>(ADAM_CHUNK_ELEMS, numels[i] - s0)});
    }
    if (chunks.empty()) return MUON_OK;
    int r;
    DevCtx dc;
    if ((r = get_dev(dc))) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t tb = align_up(sizeof(AdamTensor) * tens.size(), 256);
    const size_t cb = align_up(sizeof(AdamChunk) * chunks.size(), 256);
    Workspace* w = nullptr;
    if ((r = ws_get(dc.device, s, tb + cb, &w))) return r;
    // both tables through the pinned staging ring, as one byte block (tb and cb
    // are multiples of 256, so the block is a whole number of ring rows)
    static_assert(256 % sizeof(MatEntry) == 0, "ring rows tile 256 bytes");
    std::vector<MatEntry> rows((tb + cb) / sizeof(MatEntry));
    std::memcpy(rows.data(), tens.data(), sizeof(AdamTensor) * tens.size());
    std::memcpy(reinterpret_cast<char*>(rows.data()) + tb, chunks.data(), sizeof(AdamChunk) * chunks.size());
    if ((r = upload_table(*w, rows, reinterpret_cast<MatEntry*>(w->base), s))) return r;
    AdamArgs a;
    a.tensors = reinterpret_cast<const AdamTensor*>(w->base);
    a.chunks = reinterpret_cast<const AdamChunk*>(w->base + tb);
    a.param_dtype = param_dtype;
    a.state_dtype = state_dtype;
    a.beta1 = beta1; a.beta2 = beta2; a.eps = eps;
    const double bc1 = 1.0 - std::pow((double)beta1, (double)step);
    const double bc2 = 1.0 - std::pow((double)beta2, (double)step);
    a.lr_wd = (float)((double)lr * (double)wd);
    a.step_size = (float)((double)lr / bc1);
    a.inv_sqrt_bc2 = (float)(1.0 / std::sqrt(bc2));
    double bytes = 0;
    for (int64_t i = 0; i < count; ++i) bytes += (double)numels[i] * (3.0 * esize(param_dtype) + 4.0 * esize(state_dtype));
    note_launch_begin(KC_ADAMW, s);
    cudaError_t e = launch_adamw(a, (int)chunks.size(), s);
    note_launch_end(KC_ADAMW, bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "adamw launch");
    return MUON_OK;
} MUON_CATCH_ALL
