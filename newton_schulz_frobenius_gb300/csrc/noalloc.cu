// Allocation-free orthogonalisation entry point and its status accessor.

#include "host.h"

using namespace muon;

// ---------------------------------------------------------------------------
// Orthogonalisation without any allocation.
//
// Some callers may not allocate device memory at all: code running where the
// process's memory is owned by someone else's allocator (a framework's caching
// pool, a fixed per-job budget), or a real-time loop that forbids allocation
// after start-up.  muon_ns_orthogonalize grows a library workspace with
// cudaMalloc; this variant instead works inside one fixed array compiled into
// the library, so it calls no cudaMalloc, cudaFree, cudaMallocHost or other
// allocating routine.
//
// The array is NOALLOC_SCRATCH_BYTES long and every GPU that loads the library
// holds it until the process exits.  It holds, in order, a status word, the
// matrix table, and the NS buffers of the whole batch (no chunking), so a call
// whose batch does not fit is rejected with MUON_EINVAL.  All calls share the
// array and it keeps the last call's contents: the prep kernel's arrival
// counters are cleared on the caller's stream at the start of every call, and
// every other byte a call reads, except the status word, is written by that
// call first.
// Two calls that overlap on the GPU (different streams, or different host
// threads) race on the array; the next call after such a race starts clean.
// Device-detected errors of these calls (a bounded wait that gave up, a
// non-finite norm) accumulate in the array's status word (zero at load),
// which muon_noalloc_sync_status reads and clears without allocating.
// ---------------------------------------------------------------------------

namespace muon {

constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(64) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];
// the prep kernel's per-matrix arrival counters (cleared by every call)
constexpr int NOALLOC_MAX_BATCH = 65535;
static __device__ int g_noalloc_prep_cnt[NOALLOC_MAX_BATCH + 1];

struct NoallocDev {
    char* base = nullptr;   // device address of g_noalloc_scratch on this device
    int* pcnt = nullptr;    // device address of g_noalloc_prep_cnt
    int sms = 0;
};
static std::map<int, NoallocDev> g_noalloc_dev;

// Once per device, with that device current: the device address of the array
// (host code only sees a stand-in symbol) and the SM count.
static int noalloc_setup(NoallocDev& out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_noalloc_dev.find(dev);
    if (it == g_noalloc_dev.end()) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (!(major == 10 && minor == 3))
            return fail(MUON_ENOTSUP, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
        NoallocDev d;
        d.base = static_cast<char*>(p);
        e = cudaGetSymbolAddress(&p, g_noalloc_prep_cnt);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(counters)");
        d.pcnt = static_cast<int*>(p);
        d.sms = sms;
        it = g_noalloc_dev.emplace(dev, d).first;
    }
    out = it->second;
    return MUON_OK;
}

__global__ void noalloc_table_kernel(MatEntry* t, char* base, int64_t stride_bytes, int trans, int batch) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < batch) {
        char* p = base + (int64_t)b * stride_bytes;
        t[b] = MatEntry{p, nullptr, p, trans, 0};
    }
}

}  // namespace muon

extern "C" int muon_ns_orthogonalize_noalloc(void* ptr, int64_t m, int64_t n, int64_t batch, int dtype,
                                             const float coeffs[3], int steps, const int* segments,
                                             int num_segments, void* stream) try {
    if (!ptr) return fail(MUON_EINVAL, "ptr is NULL");
    if (m < 1 || n < 1 || batch < 1) return fail(MUON_EINVAL, "m, n, batch must be >= 1");
    if (m > (1 << 20) || n > (1 << 20) || batch > NOALLOC_MAX_BATCH) return fail(MUON_EINVAL, "size out of range");
    if (!valid_dtype(dtype)) return fail(MUON_EDTYPE, "dtype %d", dtype);
    if (!coeffs || !(std::isfinite(coeffs[0]) && std::isfinite(coeffs[1]) && std::isfinite(coeffs[2])))
        return fail(MUON_EINVAL, "coeffs missing or non-finite");
    int r = validate_segments(steps, segments, num_segments);
    if (r) return r;

    const int om = (int)std::min(m, n), on = (int)std::max(m, n);
    int nsd;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        nsd = ns_dtype(dtype, g_cfg);
    }
    const ChunkLayout L = chunk_layout(om, on, (int)batch, nsd);
    const size_t status_bytes = 256;
    const size_t table_bytes = align_up(sizeof(MatEntry) * (size_t)batch, 256);
    const size_t need = status_bytes + table_bytes + L.total;
    if (need > NOALLOC_SCRATCH_BYTES)
        return fail(MUON_EINVAL, "%lld matrices of %lld x %lld need %zu bytes of scratch; the fixed scratch holds %zu",
                    (long long)batch, (long long)m, (long long)n, need, NOALLOC_SCRATCH_BYTES);

    NoallocDev nd;
    if ((r = noalloc_setup(nd))) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DevCtx dc;
    dc.sms = nd.sms;
    dc.status = reinterpret_cast<int*>(nd.base);
    // the arrival counters start at zero: a call that raced with another one
    // (or was cut short) may have left them non-zero.  The status word is not
    // cleared here: it keeps every call's errors until it is read.
    MUON_CUDA(cudaMemsetAsync(nd.pcnt, 0, sizeof(int) * (size_t)batch, s));

    MatEntry* d_table = reinterpret_cast<MatEntry*>(nd.base + status_bytes);
    char* cbase = nd.base + status_bytes + table_bytes;
    const int64_t stride_bytes = m * n * (int64_t)esize(dtype);
    note_launch_begin(KC_OTHER, s);
    noalloc_table_kernel<<<(int)((batch + 127) / 128), 128, 0, s>>>(d_table, static_cast<char*>(ptr), stride_bytes,
                                                                     m > n ? 1 : 0, (int)batch);
    note_launch_end(KC_OTHER, 0.0, s);
    MUON_CUDA(cudaGetLastError());

    const int path = num_segments > 0 ? MUON_PATH_GRAM : MUON_PATH_PLAIN;
    std::vector<int> segs(segments, segments + num_segments);
    NsPlan plan = make_plan(coeffs, steps, segs, path, 256, om, on);
    const bool vec_ok = (reinterpret_cast<uintptr_t>(ptr) % 16 == 0) && (m % 8 == 0) && (n % 8 == 0);
    if ((r = run_prep(dc, s, cbase, L, om, on, (int)batch, d_table, dtype, dtype, nsd, false, 0, 0.f, vec_ok,
                      nd.pcnt)))
        return r;
    FinalEpi fin{EPI_OUT, d_table, dtype, 0.f, 0.f, 0.f};
    return run_ns(dc, s, cbase, L, om, on, (int)batch, nsd, plan, x_holds_u(nsd), fin);
} MUON_CATCH_ALL

extern "C" int muon_noalloc_sync_status(void* stream) try {
    NoallocDev nd;
    int r = noalloc_setup(nd);
    if (r) return r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MUON_CUDA(cudaStreamSynchronize(s));
    int v = 0;
    MUON_CUDA(cudaMemcpy(&v, nd.base, sizeof v, cudaMemcpyDeviceToHost));
    if (v) MUON_CUDA(cudaMemset(nd.base, 0, sizeof v));
    if (v & STATUS_TIMEOUT) return MUON_ETIMEOUT;
    if (v & STATUS_NONFINITE) return MUON_ENONFINITE;
    return MUON_OK;
} MUON_CATCH_ALL
