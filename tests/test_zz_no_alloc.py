"""The allocation-free orthogonalisation entry point.

muon_ns_orthogonalize_noalloc serves callers that may not allocate device
memory (memory owned by another allocator, or no allocation allowed after
start-up).  It must give the same result as muon_ns_orthogonalize while working
only inside the library's fixed scratch array.  Each case calls it twice in a
row with different inputs, through the C ABI, and compares with the ordinary
entry point within the tolerance of the parity tests.  This file is collected
last so a run that stops at the first failure has run everything else first.
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
        assert torch.isfinite(got.float()).all()
        assert _rel(got, want) <= tol


def test_noalloc_rejects_batches_beyond_the_scratch(mg):
    x = torch.zeros((2048, 8192), dtype=torch.bfloat16, device="cuda")   # needs > 64 MiB
    assert _call_noalloc(mg, x, (2, 2, 1)) == mg.MUON_EINVAL
    assert "scratch" in mg.last_error_message()
