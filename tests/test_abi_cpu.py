"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and its host-only logic (validation, FLOP accounting, status
strings, tune-cache parsing) behaves as documented.  No call here reaches a
CUDA device."""
import ctypes
import os
import re

import pytest

from oracle import muon_oracle as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def mg():
    from newton_schulz_frobenius_gb300 import _build
    _build.build()
    import newton_schulz_frobenius_gb300 as pkg
    pkg.lib()
    return pkg


def _declared():
    with open(os.path.join(ROOT, "include", "muon.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(muon_[a-z0-9_]+)\s*\(", src)))


def test_header_declarations_match_binding(mg):
    assert _declared() == sorted(mg.EXPORTS)


def test_library_exports_every_declared_symbol(mg):
    L = mg.lib()
    for name in _declared():
        assert hasattr(L, name), name


def test_plain_c_caller(mg, tmp_path):
    """The header compiles as strict C99 and a C program linked against the
    library runs its host-only entry points (tests/c_abi_host.c)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(mg.LIB_PATH)
    exe = str(tmp_path / "c_abi_host")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_abi_host.c"),
                    "-L", libdir, "-lmuon_gb300", "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "OK", r.stdout + r.stderr


def test_no_fallback_when_library_missing(monkeypatch):
    import newton_schulz_frobenius_gb300 as pkg
    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg, "LIB_PATH", "/nonexistent/libmuon_gb300.so")
    with pytest.raises(ImportError):
        pkg.lib()


def test_status_strings(mg):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert mg.status_str(code).startswith("MUON_")
    assert "unknown" in mg.status_str(12345)


@pytest.mark.parametrize("m,n", [(2560, 9728), (128, 512), (256, 256), (4096, 14336), (8192, 2048), (37, 200)])
def test_flop_accounting_matches_oracle_product_log(mg, m, n):
    om, on = min(m, n), max(m, n)
    for path, code, segs in (("plain", mg.MUON_PATH_PLAIN, ()), ("gram", mg.MUON_PATH_GRAM, (2, 2, 1)),
                             ("gram", mg.MUON_PATH_GRAM, (2, 3)), ("gram", mg.MUON_PATH_GRAM, (1, 1, 1, 1, 1))):
        nom, alg = mg.muon_ns_flops(m, n, code, segs)
        log = orc.ns_product_log(om, on, path, segments=segs if segs else (2, 2, 1))
        assert nom == log.nominal_flops()
        assert alg == log.algorithmic_flops()


def test_flop_accounting_pages_numbers(mg):
    nom_p, _ = mg.muon_ns_flops(2560, 9728, mg.MUON_PATH_PLAIN, ())
    nom_g, _ = mg.muon_ns_flops(2560, 9728, mg.MUON_PATH_GRAM, (2, 2, 1))
    assert round(nom_p / 1e12, 3) == 1.443 and round(nom_g / 1e12, 3) == 1.134


def test_flops_rejects_bad_arguments(mg):
    L = mg.lib()
    d = ctypes.c_double()
    assert L.muon_ns_flops(0, 5, 1, None, 0, ctypes.byref(d), ctypes.byref(d)) == mg.MUON_EINVAL
    assert L.muon_ns_flops(5, 5, 2, None, 0, ctypes.byref(d), ctypes.byref(d)) == mg.MUON_EINVAL
    assert L.muon_ns_flops(5, 5, 7, None, 0, ctypes.byref(d), ctypes.byref(d)) == mg.MUON_EINVAL
    huge = (ctypes.c_int * 2)(2 ** 31 - 1, 2 ** 31 - 1)
    for path in (1, 2):                                 # no overflowing step count, no endless loop
        assert L.muon_ns_flops(5, 9, path, huge, 2, ctypes.byref(d), ctypes.byref(d)) == mg.MUON_EINVAL
    neg = (ctypes.c_int * 2)(3, -1)
    assert L.muon_ns_flops(5, 9, 1, neg, 2, ctypes.byref(d), ctypes.byref(d)) == mg.MUON_EINVAL


def test_set_ns_config_validation(mg):
    L = mg.lib()
    c = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    bad = (ctypes.c_int * 3)(2, 2, 2)
    assert L.muon_set_ns_config(c, 5, bad, 3, 0) == mg.MUON_EINVAL        # sums to 6
    zero = (ctypes.c_int * 2)(5, 0)
    assert L.muon_set_ns_config(c, 5, zero, 2, 0) == mg.MUON_EINVAL       # empty segment
    huge = (ctypes.c_int * 2)(2 ** 31 - 1, 2 ** 31 - 1)
    assert L.muon_set_ns_config(c, 5, huge, 2, 0) == mg.MUON_EINVAL       # no int overflow in the sum
    over = (ctypes.c_int * 4)(3, 3, 3, -8)
    assert L.muon_set_ns_config(c, 5, over, 4, 0) == mg.MUON_EINVAL       # running sum past steps
    assert L.muon_set_ns_config(c, 0, None, 0, 0) == mg.MUON_EINVAL       # no steps
    assert L.muon_set_ns_config(c, 5, None, 0, 9) == mg.MUON_EINVAL       # bad path
    nanc = (ctypes.c_float * 3)(float("nan"), 0, 0)
    assert L.muon_set_ns_config(nanc, 5, None, 0, 0) == mg.MUON_EINVAL
    good = (ctypes.c_int * 3)(2, 2, 1)
    assert L.muon_set_ns_config(c, 5, good, 3, 0) == mg.MUON_OK
    assert "segments" in mg.last_error_message() or mg.last_error_message() != ""


def test_step_and_orthogonalize_validation_before_any_device_use(mg):
    L = mg.lib()
    vp = ctypes.c_void_p
    i64 = ctypes.c_int64
    assert L.muon_step(None, None, None, None, None, 0, 1, 1, 0.02, 0.95, 0.1, 0, None) == mg.MUON_OK
    assert L.muon_step(None, None, None, None, None, -1, 1, 1, 0.02, 0.95, 0.1, 0, None) == mg.MUON_EINVAL
    ptrs = (vp * 1)(None)
    ms = (i64 * 1)(4)
    ns = (i64 * 1)(8)
    assert L.muon_step(ptrs, ptrs, ptrs, ms, ns, 1, 1, 1, 0.02, 0.95, 0.1, 0, None) == mg.MUON_EINVAL
    assert L.muon_step(ptrs, ptrs, ptrs, ms, ns, 1, 7, 1, 0.02, 0.95, 0.1, 0, None) == mg.MUON_EDTYPE
    fake = (vp * 1)(0x1000)
    zero = (i64 * 1)(0)
    assert L.muon_step(fake, fake, fake, zero, ns, 1, 1, 1, 0.02, 0.95, 0.1, 0, None) == mg.MUON_EINVAL
    assert L.muon_step(fake, fake, fake, ms, ns, 1, 1, 1, float("inf"), 0.95, 0.1, 0, None) == mg.MUON_EINVAL
    c = (ctypes.c_float * 3)(3.4445, -4.775, 2.0315)
    segs = (ctypes.c_int * 3)(2, 2, 1)
    assert L.muon_ns_orthogonalize(None, 4, 8, 1, 1, c, 5, segs, 3, None) == mg.MUON_EINVAL
    assert L.muon_ns_orthogonalize(0x1000, 0, 8, 1, 1, c, 5, segs, 3, None) == mg.MUON_EINVAL
    assert L.muon_ns_orthogonalize(0x1000, 4, 8, 1, 5, c, 5, segs, 3, None) == mg.MUON_EDTYPE
    assert L.muon_ns_orthogonalize(0x1000, 4, 8, 1, 1, c, 4, segs, 3, None) == mg.MUON_EINVAL
    assert L.muon_ns_orthogonalize(0x1000, 4, 8, 1, 1, None, 5, segs, 3, None) == mg.MUON_EINVAL
    # a batch whose byte range overflows, or beyond the matrix table's index range
    assert L.muon_ns_orthogonalize(0x1000, 1 << 20, 1 << 20, 1 << 21, 1, c, 5, segs, 3, None) == mg.MUON_EINVAL
    assert "overflows" in mg.last_error_message()
    assert L.muon_ns_orthogonalize(0x1000, 1, 1, 1 << 31, 1, c, 5, segs, 3, None) == mg.MUON_EINVAL


def test_adamw_rejects_oversized_tables_before_device_use(mg):
    """Sizes whose chunk table would not fit the launch (or the byte range)
    are rejected before any table is built or any device is touched.  The
    pointers are placeholders, so this runs only without a CUDA device."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("placeholder pointers: host-only check")
    L = mg.lib()
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    fake = (vp * 1)(0x1000)
    for numel in (1 << 62, 1 << 50):
        r = L.muon_adamw_step(fake, fake, fake, fake, (i64 * 1)(numel), 1, mg.MUON_BF16, mg.MUON_F32,
                              1e-3, 0.9, 0.999, 1e-8, 0.0, 1, None)
        assert r == mg.MUON_EINVAL, (numel, r)
    # a size within range gets past validation and stops at the missing device
    r = L.muon_adamw_step(fake, fake, fake, fake, (i64 * 1)(1024), 1, mg.MUON_BF16, mg.MUON_F32,
                          1e-3, 0.9, 0.999, 1e-8, 0.0, 1, None)
    assert r not in (mg.MUON_OK, mg.MUON_EINVAL)


def test_autotune_validation_before_any_device_use(mg):
    L = mg.lib()
    i64 = ctypes.c_int64
    assert L.muon_autotune(None, None, -1, mg.MUON_BF16, None) == mg.MUON_EINVAL
    assert L.muon_autotune((i64 * 1)(4), (i64 * 1)(8), 1, 9, None) == mg.MUON_EDTYPE
    for m, n in ((0, 8), (8, (1 << 20) + 1), ((1 << 31) + 5, 8)):
        assert L.muon_autotune((i64 * 1)(m), (i64 * 1)(n), 1, mg.MUON_BF16, None) == mg.MUON_EINVAL, (m, n)
        assert "2^20" in mg.last_error_message()


def test_debug_gemm_validation(mg):
    L = mg.lib()
    assert L.muon_debug_gemm(None, None, None, 4, 4, 4, 1, 1, 1, 0, 0, 1.0, 0, 0, 0, 0, None) == mg.MUON_EINVAL
    p = 0x1000
    assert L.muon_debug_gemm(p, p, p, 4, 8, 4, 1, 1, 1, 1, 0, 1.0, 0, 0, 0, 0, None) == mg.MUON_EINVAL
    assert L.muon_debug_gemm(p, p, p, 8, 8, 8, 1, 1, 1, 1, 0, 1.0, 0, 0, 0, 100, None) == mg.MUON_EINVAL
    assert L.muon_debug_gemm(p, p, p, 8, 8, 12, 1, 1, 1, 0, 0, 1.0, 0, 0, 0, 0, None) == mg.MUON_EINVAL


def test_last_path_unknown_shape(mg):
    assert mg.muon_last_path(3, 7, mg.MUON_BF16) is None


def test_tune_load_missing_or_foreign_file(mg, tmp_path):
    assert mg.muon_tune_load(str(tmp_path / "missing.tsv")) == 0
    p = tmp_path / "junk.tsv"
    p.write_text("not a tune cache\n1\t2\t3\n")
    assert mg.muon_tune_load(str(p)) == 0


def test_kernel_timing_read_empty(mg):
    mg.muon_set_kernel_timing(False)
    assert mg.muon_kernel_timing_read() == {}
    assert mg.muon_launch_count() >= 0


def test_arm_stall_validation(mg):
    """The bounded-wait test hook is host state only: bad kernels or stages
    are refused, and disarming always succeeds."""
    for kernel, stage in ((3, 0), (1, -1), (2, 1 << 21)):
        with pytest.raises(mg.MuonError) as ei:
            mg.muon_debug_arm_stall(kernel, stage)
        assert ei.value.status == mg.MUON_EINVAL
    mg.muon_debug_arm_stall(mg.STALL_PRODUCT, 2)
    mg.muon_debug_arm_stall(0)
