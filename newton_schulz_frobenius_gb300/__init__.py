"""Python binding of the GB300 Muon update library (``include/muon.h``).

Argument marshalling only: every step of the update runs in the library's CUDA
kernels.  The functions keep the C names; tensors are PyTorch CUDA tensors
(PyTorch supplies device memory and streams).  Loading fails loudly when the
shared library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libmuon_gb300.so")

MUON_OK = 0
MUON_EINVAL = -1
MUON_EDTYPE = -2
MUON_ENOMEM = -3
MUON_ECUDA = -4
MUON_ENONFINITE = -5
MUON_ETIMEOUT = -6
MUON_ENOTSUP = -7

MUON_F32 = 0
MUON_BF16 = 1
MUON_F16 = 2

MUON_PATH_AUTO = 0
MUON_PATH_PLAIN = 1
MUON_PATH_GRAM = 2

QUINTIC = (3.4445, -4.7750, 2.0315)

#: every entry point include/muon.h declares
EXPORTS = (
    "muon_ns_orthogonalize", "muon_ns_orthogonalize_noalloc", "muon_noalloc_sync_status", "muon_step",
    "muon_set_ns_config",
    "muon_set_ns_precision", "muon_autotune",
    "muon_tune_save", "muon_tune_load", "muon_last_path", "muon_sync_status",
    "muon_status_str", "muon_last_error_message", "muon_ns_flops", "muon_launch_count",
    "muon_set_kernel_timing", "muon_kernel_timing_read", "muon_debug_gemm", "muon_debug_arm_stall",
    "muon_group_create", "muon_group_step", "muon_group_destroy", "muon_group_set_host_io",
    "muon_owner_plan", "muon_adamw_step",
    "muon_pack_plan", "muon_pack",
)

_lib = None


class MuonError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({last_error_message()})")


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(nvcc, sm_103a); there is no CPU fallback")
    L = ctypes.CDLL(LIB_PATH)
    i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
    f3 = ctypes.POINTER(ctypes.c_float)
    ip = ctypes.POINTER(ctypes.c_int)
    i64p = ctypes.POINTER(ctypes.c_int64)
    dp = ctypes.POINTER(ctypes.c_double)
    sig = {
        "muon_ns_orthogonalize": (i32, [vp, i64, i64, i64, i32, f3, i32, ip, i32, vp]),
        "muon_ns_orthogonalize_noalloc": (i32, [vp, i64, i64, i64, i32, f3, i32, ip, i32, vp]),
        "muon_noalloc_sync_status": (i32, [vp]),
        "muon_step": (i32, [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), i64p, i64p, i64,
                            i32, i32, f32, f32, f32, i32, vp]),
        "muon_set_ns_config": (i32, [f3, i32, ip, i32, i32]),
        "muon_autotune": (i32, [i64p, i64p, i64, i32, vp]),
        "muon_tune_save": (i32, [ctypes.c_char_p]),
        "muon_tune_load": (i32, [ctypes.c_char_p]),
        "muon_last_path": (i32, [i64, i64, i32, ip]),
        "muon_sync_status": (i32, [vp]),
        "muon_status_str": (ctypes.c_char_p, [i32]),
        "muon_last_error_message": (ctypes.c_char_p, []),
        "muon_ns_flops": (i32, [i64, i64, i32, ip, i32, dp, dp]),
        "muon_launch_count": (i64, []),
        "muon_debug_arm_stall": (i32, [i32, i32]),
        "muon_set_kernel_timing": (i32, [i32]),
        "muon_kernel_timing_read": (i32, [ctypes.c_char_p, i64p, dp, dp, i32]),
        "muon_debug_gemm": (i32, [vp, vp, vp, i64, i64, i64, i64, i32, i32, i32, i32,
                                  f32, f32, f32, f32, i32, vp]),
        "muon_group_create": (i32, [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), i64p, i64p, i64,
                                    i32, i32, ctypes.POINTER(vp)]),
        "muon_group_step": (i32, [vp, f32, f32, f32, i32, vp]),
        "muon_group_destroy": (i32, [vp]),
        "muon_group_set_host_io": (i32, [vp, ctypes.POINTER(vp), ctypes.POINTER(vp)]),
        "muon_owner_plan": (i32, [i64p, i64p, i64, i32, i32, ip, dp, dp, ip]),
        "muon_adamw_step": (i32, [ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                  i64p, i64, i32, i32, f32, f32, f32, f32, f32, i64, vp]),
        "muon_pack_plan": (i32, [i64p, i64p, ip, i64, i32, i64, i64p, i64p]),
        "muon_pack": (i32, [ctypes.POINTER(vp), i64p, i64p, i64p, i64, i32, vp, i32, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def status_str(status: int) -> str:
    return lib().muon_status_str(int(status)).decode()


def last_error_message() -> str:
    return lib().muon_last_error_message().decode()


def _check(status: int, what: str) -> None:
    if status != MUON_OK:
        raise MuonError(status, what)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return MUON_F32
    if t.dtype == torch.bfloat16:
        return MUON_BF16
    if t.dtype == torch.float16:
        return MUON_F16
    raise TypeError(f"unsupported dtype {t.dtype}: float32, bfloat16 or float16")


def _stream_ptr(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ints(vals):
    vals = list(vals or [])
    return (ctypes.c_int * max(1, len(vals)))(*vals), len(vals)


def _cuda_contig(t, name):
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


# ---------------------------------------------------------------------------
# the entry points
# ---------------------------------------------------------------------------

def muon_ns_orthogonalize(x, coeffs=QUINTIC, steps: int = 5, segments=(2, 2, 1), stream=None):
    """In place: x (m x n or batch x m x n) <- NS(x / ||x||_F).  segments=None: plain NS."""
    _cuda_contig(x, "x")
    if x.dim() == 2:
        batch, m, n = 1, x.shape[0], x.shape[1]
    elif x.dim() == 3:
        batch, m, n = x.shape
    else:
        raise ValueError("x must be 2-D or 3-D")
    c = (ctypes.c_float * 3)(*coeffs)
    segs, nseg = _ints(segments)
    _check(lib().muon_ns_orthogonalize(x.data_ptr(), m, n, batch, _dtype_code(x), c, steps, segs, nseg,
                                       _stream_ptr(stream)), "muon_ns_orthogonalize")
    return x


def muon_ns_orthogonalize_noalloc(x, coeffs=QUINTIC, steps: int = 5, segments=(2, 2, 1), stream=None):
    """Same as muon_ns_orthogonalize, inside the library's fixed 64 MiB scratch
    array: no device memory is allocated (for callers that may not allocate)."""
    _cuda_contig(x, "x")
    if x.dim() == 2:
        batch, m, n = 1, x.shape[0], x.shape[1]
    elif x.dim() == 3:
        batch, m, n = x.shape
    else:
        raise ValueError("x must be 2-D or 3-D")
    c = (ctypes.c_float * 3)(*coeffs)
    segs, nseg = _ints(segments)
    _check(lib().muon_ns_orthogonalize_noalloc(x.data_ptr(), m, n, batch, _dtype_code(x), c, steps, segs, nseg,
                                               _stream_ptr(stream)), "muon_ns_orthogonalize_noalloc")
    return x


def muon_step(params, grads, moms, lr: float, beta: float, wd: float, nesterov: bool, stream=None):
    """One Muon step over lists of matrices (updated in place: params, moms)."""
    arr = _step_arrays(params, grads, moms)
    if arr is None:
        return
    _check(lib().muon_step(*arr, float(lr), float(beta), float(wd), 1 if nesterov else 0, _stream_ptr(stream)),
           "muon_step")


def _step_arrays(params, grads, moms):
    k = len(params)
    if not (len(grads) == k and len(moms) == k):
        raise ValueError("params, grads and moms must have the same length")
    if k == 0:
        return None
    pd = _dtype_code(params[0])
    md = _dtype_code(moms[0])
    for i in range(k):
        p, g, mo = params[i], grads[i], moms[i]
        for t, nm in ((p, "param"), (g, "grad"), (mo, "mom")):
            _cuda_contig(t, nm)
            if t.dim() != 2:
                raise ValueError(f"{nm} {i} must be 2-D")
        if p.shape != g.shape or p.shape != mo.shape:
            raise ValueError(f"shape mismatch at {i}")
        if _dtype_code(p) != pd or _dtype_code(g) != pd or _dtype_code(mo) != md:
            raise TypeError(f"dtype mismatch at {i}")
    VP = ctypes.c_void_p * k
    I64 = ctypes.c_int64 * k
    return (VP(*[p.data_ptr() for p in params]), VP(*[g.data_ptr() for g in grads]),
            VP(*[m.data_ptr() for m in moms]), I64(*[p.shape[0] for p in params]),
            I64(*[p.shape[1] for p in params]), k, pd, md)


def muon_group_create(params, grads, moms):
    """Registers a fixed set of matrices; returns an opaque group handle."""
    arr = _step_arrays(params, grads, moms)
    if arr is None:
        raise ValueError("a group needs at least one matrix")
    out = ctypes.c_void_p()
    _check(lib().muon_group_create(*arr, ctypes.byref(out)), "muon_group_create")
    return out.value


def muon_group_step(handle, lr: float, beta: float, wd: float, nesterov: bool, stream=None):
    _check(lib().muon_group_step(handle, float(lr), float(beta), float(wd), 1 if nesterov else 0,
                                 _stream_ptr(stream)), "muon_group_step")


def muon_group_destroy(handle):
    if handle:
        lib().muon_group_destroy(handle)


class MuonGroup:
    """The optimizer object of a training loop: a fixed set of (param, grad,
    momentum) CUDA tensors stepped many times.  The tensors must stay alive and
    at the same addresses for the group's lifetime (update them in place)."""

    def __init__(self, params, grads, moms):
        self._refs = (list(params), list(grads), list(moms))
        self.handle = muon_group_create(*self._refs)

    def step(self, lr: float, beta: float = 0.95, wd: float = 0.0, nesterov: bool = True, stream=None):
        muon_group_step(self.handle, lr, beta, wd, nesterov, stream)

    def set_host_io(self, host_grads=None, host_params=None):
        """Pinned CPU tensors (same shapes and dtypes as the group's gradients
        and parameters) that every step copies the gradients from and the
        updated parameters to, overlapped with the update; None turns a
        direction off."""
        k = len(self._refs[0])
        arrs = []
        for lst, nm in ((host_grads, "host_grads"), (host_params, "host_params")):
            if lst is None:
                arrs.append(None)
                continue
            lst = list(lst)
            if len(lst) != k:
                raise ValueError(f"{nm} must hold {k} tensors")
            for t, ref in zip(lst, self._refs[1] if nm == "host_grads" else self._refs[0]):
                if t.device.type != "cpu" or not t.is_contiguous() or t.shape != ref.shape or t.dtype != ref.dtype:
                    raise ValueError(f"{nm}: contiguous CPU tensors of the group's shapes and dtypes required")
            arrs.append((ctypes.c_void_p * k)(*[t.data_ptr() for t in lst]))
        self._host_refs = (host_grads, host_params)     # kept alive while the group uses them
        _check(lib().muon_group_set_host_io(self.handle, arrs[0], arrs[1]), "muon_group_set_host_io")

    def close(self):
        if self.handle:
            muon_group_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def muon_set_ns_precision(dtype: int = -1):
    """NS working precision for 16-bit parameters: -1 follows them, MUON_BF16
    or MUON_F16 forces that type."""
    _check(lib().muon_set_ns_precision(int(dtype)), "muon_set_ns_precision")


def muon_set_ns_config(coeffs=QUINTIC, steps: int = 5, segments=(2, 2, 1), path: int = MUON_PATH_AUTO):
    c = (ctypes.c_float * 3)(*coeffs) if coeffs is not None else None
    segs, nseg = _ints(segments)
    _check(lib().muon_set_ns_config(c, steps, segs, nseg, path), "muon_set_ns_config")


def muon_autotune(shapes, dtype: int = MUON_BF16, stream=None):
    shapes = list(shapes)
    k = len(shapes)
    I64 = ctypes.c_int64 * max(1, k)
    _check(lib().muon_autotune(I64(*[s[0] for s in shapes]), I64(*[s[1] for s in shapes]), k, dtype,
                               _stream_ptr(stream)), "muon_autotune")


def muon_tune_save(path: str):
    _check(lib().muon_tune_save(path.encode()), "muon_tune_save")


def muon_tune_load(path: str) -> int:
    r = lib().muon_tune_load(path.encode())
    if r < 0:
        raise MuonError(r, "muon_tune_load")
    return r


def muon_last_path(m: int, n: int, dtype: int):
    out = ctypes.c_int(-1)
    r = lib().muon_last_path(m, n, dtype, ctypes.byref(out))
    return out.value if r == MUON_OK else None


def muon_sync_status(stream=None) -> int:
    return lib().muon_sync_status(_stream_ptr(stream))


def muon_noalloc_sync_status(stream=None) -> int:
    """Status word of the allocation-free calls (read and cleared; allocates nothing)."""
    return lib().muon_noalloc_sync_status(_stream_ptr(stream))


def muon_ns_flops(m: int, n: int, path: int, segments=(2, 2, 1)):
    segs, nseg = _ints(segments)
    nom, alg = ctypes.c_double(), ctypes.c_double()
    _check(lib().muon_ns_flops(m, n, path, segs, nseg, ctypes.byref(nom), ctypes.byref(alg)), "muon_ns_flops")
    return nom.value, alg.value


def muon_launch_count() -> int:
    return lib().muon_launch_count()


#: kernels the bounded-wait test hook can stall
STALL_PRODUCT = 1
STALL_SMALL = 2


def muon_debug_arm_stall(kernel: int, stage: int = 0) -> None:
    """Test hook: the next launch of `kernel` leaves one stage unfilled, so its
    bounded wait runs out and muon_sync_status reports MUON_ETIMEOUT."""
    _check(lib().muon_debug_arm_stall(int(kernel), int(stage)), "muon_debug_arm_stall")


def muon_set_kernel_timing(enable: bool):
    lib().muon_set_kernel_timing(1 if enable else 0)


def muon_kernel_timing_read():
    """{class name: (launches, total_ms, algorithmic work)}; resets the record."""
    n = 16
    names = ctypes.create_string_buffer(32 * n)
    launches = (ctypes.c_int64 * n)()
    ms = (ctypes.c_double * n)()
    work = (ctypes.c_double * n)()
    k = lib().muon_kernel_timing_read(names, launches, ms, work, n)
    out = {}
    for i in range(k):
        nm = names.raw[32 * i:32 * i + 32].split(b"\0", 1)[0].decode()
        if launches[i]:
            out[nm] = (int(launches[i]), float(ms[i]), float(work[i]))
    return out


MUON_DEBUG_TF32 = 3
MUON_DEBUG_TF32_CHUNKED = 4


def muon_debug_gemm(A, B, C, b_kmajor=True, symmetric=False, poly=None, alpha=1.0, tile_n=0, stream=None,
                    tf32=False, tf32_chunked=False):
    """C[b] = alpha * A[b] op(B[b]) (or the fused polynomial when poly=(a, b, c)).
    tf32=True multiplies fp32 tensors on the TF32 tensor-core path;
    tf32_chunked=True does too, accumulating K in chunks summed in
    round-to-nearest fp32."""
    for t, nm in ((A, "A"), (B, "B"), (C, "C")):
        _cuda_contig(t, nm)
    batch = A.shape[0] if A.dim() == 3 else 1
    M, K = A.shape[-2], A.shape[-1]
    N = B.shape[-2] if b_kmajor else B.shape[-1]
    pa, pb, pc = poly if poly is not None else (0.0, 0.0, 0.0)
    code = MUON_DEBUG_TF32_CHUNKED if tf32_chunked else (MUON_DEBUG_TF32 if tf32 else _dtype_code(A))
    _check(lib().muon_debug_gemm(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, batch, code,
                                 1 if b_kmajor else 0, 1 if symmetric else 0, 1 if poly is not None else 0,
                                 float(alpha), float(pa), float(pb), float(pc), tile_n, _stream_ptr(stream)),
           "muon_debug_gemm")
    return C


def muon_owner_plan(shapes, ranks: int, dtype: int = MUON_BF16):
    """Owner rank per matrix for a multi-rank step (greedy longest-processing-
    time first on measured or modelled per-matrix costs).
    Returns (owners, per-rank loads, makespan, measured)."""
    shapes = list(shapes)
    k = len(shapes)
    I64 = ctypes.c_int64 * max(1, k)
    owners = (ctypes.c_int * max(1, k))()
    loads = (ctypes.c_double * max(1, ranks))()
    mk = ctypes.c_double()
    meas = ctypes.c_int()
    _check(lib().muon_owner_plan(I64(*[s[0] for s in shapes]), I64(*[s[1] for s in shapes]), k, dtype, ranks,
                                 owners, loads, ctypes.byref(mk), ctypes.byref(meas)), "muon_owner_plan")
    return list(owners)[:k], list(loads)[:ranks], mk.value, bool(meas.value)


def muon_pack_plan(shapes, owners, ranks: int, align_elems: int = 8):
    """Packed exchange layout: (element offset per matrix, segment length);
    rank r's owned matrices fill segment [r seg, (r+1) seg)."""
    shapes, owners = list(shapes), list(owners)
    k = len(shapes)
    if len(owners) != k:
        raise ValueError("one owner per matrix")
    I64 = ctypes.c_int64 * max(1, k)
    off = I64()
    seg = ctypes.c_int64()
    _check(lib().muon_pack_plan(I64(*[s[0] for s in shapes]), I64(*[s[1] for s in shapes]),
                                (ctypes.c_int * max(1, k))(*owners), k, int(ranks), int(align_elems), off,
                                ctypes.byref(seg)), "muon_pack_plan")
    return list(off)[:k], seg.value


def muon_pack(mats, offsets, packed, to_packed: bool = True, stream=None):
    """Copies CUDA matrices into (to_packed) or out of a packed CUDA buffer of
    the same dtype, matrix i at element offset offsets[i]."""
    k = len(mats)
    if len(offsets) != k:
        raise ValueError("one offset per matrix")
    if k == 0:
        return
    dt = _dtype_code(packed)
    _cuda_contig(packed, "packed")
    for i, t in enumerate(mats):
        _cuda_contig(t, f"matrix {i}")
        if _dtype_code(t) != dt:
            raise TypeError(f"matrix {i}: dtype differs from the packed buffer")
        if offsets[i] < 0 or offsets[i] + t.numel() > packed.numel():
            raise ValueError(f"matrix {i} does not fit the packed buffer at offset {offsets[i]}")
    shp = [(t.shape[0], t.numel() // t.shape[0]) if t.dim() >= 1 and t.shape[0] > 0 else (1, t.numel())
           for t in mats]
    VP = ctypes.c_void_p * k
    I64 = ctypes.c_int64 * k
    _check(lib().muon_pack(VP(*[t.data_ptr() for t in mats]), I64(*[s[0] for s in shp]), I64(*[s[1] for s in shp]),
                           I64(*offsets), k, dt, packed.data_ptr(), 1 if to_packed else 0, _stream_ptr(stream)),
           "muon_pack")


def muon_adamw_step(params, grads, exp_avgs, exp_avg_sqs, lr: float, beta1: float = 0.9, beta2: float = 0.999,
                    eps: float = 1e-8, wd: float = 0.0, step: int = 1, stream=None):
    """AdamW over lists of CUDA tensors of any shape (params, moments in place)."""
    k = len(params)
    if not (len(grads) == k and len(exp_avgs) == k and len(exp_avg_sqs) == k):
        raise ValueError("tensor lists must have the same length")
    if k == 0:
        return
    pd, sd = _dtype_code(params[0]), _dtype_code(exp_avgs[0])
    for i in range(k):
        for t, nm, dt in ((params[i], "param", pd), (grads[i], "grad", pd), (exp_avgs[i], "exp_avg", sd),
                          (exp_avg_sqs[i], "exp_avg_sq", sd)):
            _cuda_contig(t, nm)
            if _dtype_code(t) != dt or t.numel() != params[i].numel():
                raise TypeError(f"{nm} {i}: dtype or size mismatch")
    VP = ctypes.c_void_p * k
    _check(lib().muon_adamw_step(VP(*[t.data_ptr() for t in params]), VP(*[t.data_ptr() for t in grads]),
                                 VP(*[t.data_ptr() for t in exp_avgs]), VP(*[t.data_ptr() for t in exp_avg_sqs]),
                                 (ctypes.c_int64 * k)(*[t.numel() for t in params]), k, pd, sd, float(lr),
                                 float(beta1), float(beta2), float(eps), float(wd), int(step),
                                 _stream_ptr(stream)), "muon_adamw_step")
