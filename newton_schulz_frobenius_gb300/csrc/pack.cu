// Packed exchange buffers for an owner-centric step ("DMuon" summary, section
// 2.1: gradients are reduced into owner-contiguous buffers before the
// orthogonalisation and the updated parameters are published from them after;
// section 2.3: each matrix has one owner).  The host lays the matrices out
// rank by rank (muon_pack_plan); this kernel moves every matrix of a call
// between its caller storage and its place in the packed buffer in one
// launch: CTA k copies chunk k (up to PACK_CHUNK_ELEMS elements of one
// matrix), with 16-byte vectors where both sides are 16-byte aligned and one
// element at a time otherwise.  A pure copy: bound by HBM bandwidth.
#include "muon_internal.cuh"

namespace muon {

namespace {

constexpr int PT = 256;

__global__ void __launch_bounds__(PT) pack_kernel(const __grid_constant__ PackArgs a) {
    pdl_wait();
    pdl_trigger();
    const PackChunk ch = a.chunks[blockIdx.x];
    const PackMat mt = a.mats[ch.mat];
    char* mat = static_cast<char*>(mt.p) + (int64_t)ch.start * a.esize;
    char* pk = static_cast<char*>(a.packed) + (mt.off + ch.start) * a.esize;
    char* dst = a.to_packed ? pk : mat;
    const char* src = a.to_packed ? mat : pk;
    const int64_t bytes = (int64_t)ch.len * a.esize;
    if (mt.vec_ok) {
        // len is a multiple of 16 bytes except in a matrix's last chunk
        const int64_t nv = bytes / 16;
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        uint4* d4 = reinterpret_cast<uint4*>(dst);
        int64_t i = threadIdx.x;
        for (; i + 3 * PT < nv; i += 4 * PT) {        // four 16-byte loads in flight per thread
            const uint4 x0 = __ldcs(s4 + i), x1 = __ldcs(s4 + i + PT), x2 = __ldcs(s4 + i + 2 * PT),
                        x3 = __ldcs(s4 + i + 3 * PT);
            __stcs(d4 + i, x0);
            __stcs(d4 + i + PT, x1);
            __stcs(d4 + i + 2 * PT, x2);
            __stcs(d4 + i + 3 * PT, x3);
        }
        for (; i < nv; i += PT) __stcs(d4 + i, __ldcs(s4 + i));
        for (int64_t b = nv * 16 + threadIdx.x; b < bytes; b += PT) dst[b] = src[b];
    } else if (a.esize == 2) {
        const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src);
        uint16_t* d2 = reinterpret_cast<uint16_t*>(dst);
        for (int i = threadIdx.x; i < ch.len; i += PT) d2[i] = s2[i];
    } else {
        const uint32_t* s1 = reinterpret_cast<const uint32_t*>(src);
        uint32_t* d1 = reinterpret_cast<uint32_t*>(dst);
        for (int i = threadIdx.x; i < ch.len; i += PT) d1[i] = s1[i];
    }
}

}  // namespace

cudaError_t launch_pack(const PackArgs& a, int nchunks, cudaStream_t s) {
    if (nchunks <= 0) return cudaSuccess;
    return launch_pdl(pack_kernel, dim3(nchunks), dim3(PT), 0, s, a);
}

}  // namespace muon
