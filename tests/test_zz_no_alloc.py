"""The allocation-free orthogonalisation entry point.

muon_ns_orthogonalize_noalloc serves callers that may not allocate device
memory (memory owned by another allocator, or no allocation allowed after
start-up).  It must give the same result as muon_ns_orthogonalize while working
only inside the library's fixed scratch array.  Each case calls it twice in a
row with different inputs, through the C ABI, and compares with the ordinary
entry point within the tolerance of the parity tests; the device status of
these calls is read through muon_noalloc_sync_status, which allocates nothing
either.  One test shows that nothing is allocated: with the library's
allocator hook failing every allocation (MUON_FAIL_ALLOC=1) the calls still
succeed, and the device's free memory is the same before and after them.
This file is collected last so a run that stops at the first failure has run
everything else first.
"""
import ctypes

import pytest

from tests.gpu_util import TOL

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    return pkg


def _call_noalloc(mg, x, segments):
    L = mg.lib()
    batch, m, n = (1, *x.shape) if x.dim() == 2 else x.shape
    c = (ctypes.c_float * 3)(*mg.QUINTIC)
    segs = (ctypes.c_int * max(1, len(segments or ())))(*(segments or ()))
    stream = torch.cuda.current_stream().cuda_stream
    return L.muon_ns_orthogonalize_noalloc(x.data_ptr(), m, n, batch, 1 if x.dtype == torch.bfloat16 else 0,
                                           c, 5, segs, len(segments or ()), stream)


def _noalloc_status(mg):
    return mg.lib().muon_noalloc_sync_status(torch.cuda.current_stream().cuda_stream)


def _rel(a, b):
    return ((a.double() - b.double()).norm() / b.double().norm()).item()


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, TOL["bf16"]), (torch.float32, TOL["f32"])])
def test_noalloc_matches_orthogonalize_twice(mg, dtype, tol):
    g = torch.Generator(device="cuda").manual_seed(1234)
    cases = [((3, 256, 1024), (2, 2, 1)), ((2, 640, 192), None)]   # second call: other shape, tall, plain
    for shape, segments in cases:
        x = (torch.randn(shape, generator=g, device="cuda") * 0.03).to(dtype)
        want = x.clone()
        got = x.clone()
        mg.muon_ns_orthogonalize(want, mg.QUINTIC, 5, segments)
        assert _call_noalloc(mg, got, segments) == mg.MUON_OK
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        assert _noalloc_status(mg) == mg.MUON_OK
        assert torch.isfinite(got.float()).all()
        assert _rel(got, want) <= tol


def test_noalloc_allocates_nothing(mg, monkeypatch):
    g = torch.Generator(device="cuda").manual_seed(77)
    xs = [(torch.randn(shape, generator=g, device="cuda") * 0.03).to(torch.bfloat16)
          for shape in ((4, 128, 512), (384, 1024))]
    segs = [(2, 2, 1), None]
    wants = [x.clone() for x in xs]
    for w, s in zip(wants, segs):
        mg.muon_ns_orthogonalize(w, mg.QUINTIC, 5, s)
    # one call before measuring: the first call on a device looks up the
    # fixed array (and may load the library's device code)
    warm = xs[0].clone()
    assert _call_noalloc(mg, warm, segs[0]) == mg.MUON_OK
    assert _noalloc_status(mg) == mg.MUON_OK
    gots = [x.clone() for x in xs]
    torch.cuda.synchronize()
    monkeypatch.setenv("MUON_FAIL_ALLOC", "1")       # every allocation of the library fails
    free0 = torch.cuda.mem_get_info()[0]
    for got, s in zip(gots, segs):
        assert _call_noalloc(mg, got, s) == mg.MUON_OK
    assert _noalloc_status(mg) == mg.MUON_OK
    free1 = torch.cuda.mem_get_info()[0]
    monkeypatch.delenv("MUON_FAIL_ALLOC")
    assert free1 == free0
    for got, want in zip(gots, wants):
        assert _rel(got, want) <= TOL["bf16"]


def test_noalloc_reports_nonfinite_input(mg):
    g = torch.Generator(device="cuda").manual_seed(5)
    x = (torch.randn((256, 1024), generator=g, device="cuda") * 0.03).to(torch.bfloat16)
    bad = x.clone()
    bad[3, 7] = float("nan")
    assert _call_noalloc(mg, bad, (2, 2, 1)) == mg.MUON_OK     # detected on the device
    assert _noalloc_status(mg) == mg.MUON_ENONFINITE
    assert _noalloc_status(mg) == mg.MUON_OK                   # reading cleared it
    # the next call on the same stream is clean and right
    want = x.clone()
    mg.muon_ns_orthogonalize(want, mg.QUINTIC, 5, (2, 2, 1))
    assert _call_noalloc(mg, x, (2, 2, 1)) == mg.MUON_OK
    assert _noalloc_status(mg) == mg.MUON_OK
    assert _rel(x, want) <= TOL["bf16"]


def test_noalloc_rejects_batches_beyond_the_scratch(mg):
    x = torch.zeros((2048, 8192), dtype=torch.bfloat16, device="cuda")   # needs > 64 MiB
    assert _call_noalloc(mg, x, (2, 2, 1)) == mg.MUON_EINVAL
    assert "scratch" in mg.last_error_message()
