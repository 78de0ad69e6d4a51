"""Bounded device waits that run out, with no GPU fault.

Every mbarrier wait in the library's kernels gives up after a limit of about
two seconds, raises MUON_ETIMEOUT in the device status word, waits (bounded)
for the copies and products it has in flight, frees its tensor memory and
returns.  The test hook muon_debug_arm_stall makes that happen on purpose: the
next launch of the chosen kernel leaves one pipeline stage unfilled (its
producer issues no copy for it, so nothing is in flight for that stage) and
the consumer's wait for it runs out.  Each test then checks that the status
reads MUON_ETIMEOUT once, and that an ordinary call on the same stream
succeeds and matches the fp64 oracle.
"""
import time

import numpy as np
import pytest

from oracle import muon_oracle as orc
from tests.gpu_util import SIGMA_TOL, TOL, rel_fro, sigma_dev, to_device, to_f64
from workloads import gen_matrix, zeros_matrix

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    yield pkg
    pkg.muon_debug_arm_stall(0)
    pkg.muon_set_ns_config(pkg.QUINTIC, 5, (2, 2, 1), pkg.MUON_PATH_AUTO)


def _ortho_matches_oracle(mg, rows, cols, seed):
    h = gen_matrix(seed, 0, rows, cols, 0.03, "bf16")
    x = to_device(h, torch)
    mg.muon_ns_orthogonalize(x, mg.QUINTIC, 5, (2, 2, 1))
    assert mg.muon_sync_status() == mg.MUON_OK
    ref = orc.orthogonalize(orc.to_f64(h.data, "bf16"), "gram", segments=(2, 2, 1))
    O = to_f64(x)
    assert rel_fro(O, ref) <= TOL["bf16"]
    assert sigma_dev(O, ref) <= SIGMA_TOL


@pytest.mark.parametrize("stage", [0, 3])
def test_product_kernel_wait_runs_out(mg, stage):
    """The tensor-core product kernel (128-column tiles, unpaired): CTA 0
    never fills k-block `stage` of its first tile."""
    g = torch.Generator(device="cuda").manual_seed(31)
    A = (torch.randn((1, 256, 512), generator=g, device="cuda") / 512 ** 0.5).to(torch.bfloat16)
    B = (torch.randn((1, 384, 512), generator=g, device="cuda") / 512 ** 0.5).to(torch.bfloat16)
    C = torch.empty((1, 256, 384), dtype=torch.bfloat16, device="cuda")
    ref = (A[0].double() @ B[0].double().T)
    assert mg.muon_sync_status() == mg.MUON_OK
    mg.muon_debug_arm_stall(mg.STALL_PRODUCT, stage)
    try:
        t0 = time.perf_counter()
        mg.muon_debug_gemm(A, B, C, b_kmajor=True, tile_n=128)
        st = mg.muon_sync_status()
        waited = time.perf_counter() - t0
    finally:
        mg.muon_debug_arm_stall(0)
    assert st == mg.MUON_ETIMEOUT, mg.status_str(st)
    assert 1.0 <= waited <= 60.0, waited
    assert mg.muon_sync_status() == mg.MUON_OK            # reading cleared it
    # the same product on the same stream, now whole
    mg.muon_debug_gemm(A, B, C, b_kmajor=True, tile_n=128)
    assert mg.muon_sync_status() == mg.MUON_OK
    err = ((C[0].double() - ref).norm() / ref.norm()).item()
    assert err < 1e-2, err
    # and a whole orthogonalisation through the product kernels
    _ortho_matches_oracle(mg, 256, 1024, 4100)


def test_small_kernel_wait_runs_out(mg, monkeypatch):
    """The fused small-matrix kernel: CTA 0 never issues the first piece of
    its first matrix's gradient and momentum."""
    monkeypatch.setenv("MUON_SMALL", "1")
    mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_GRAM)
    shapes = [(128, 512)] * 4
    Ws = [gen_matrix(4200 + i, 1, r, c, 0.02, "bf16") for i, (r, c) in enumerate(shapes)]
    Gs = [gen_matrix(4200 + i, 0, r, c, 0.0316, "bf16") for i, (r, c) in enumerate(shapes)]
    w = [to_device(h, torch) for h in Ws]
    gr = [to_device(h, torch) for h in Gs]
    mo = [torch.zeros_like(x) for x in w]
    assert mg.muon_sync_status() == mg.MUON_OK
    mg.muon_debug_arm_stall(mg.STALL_SMALL, 0)
    try:
        before = mg.muon_launch_count()
        mg.muon_step(w, gr, mo, lr=0.02, beta=0.95, wd=0.1, nesterov=False)
        st = mg.muon_sync_status()
        launched = mg.muon_launch_count() - before
    finally:
        mg.muon_debug_arm_stall(0)
    assert launched == 1                                   # the one fused launch took the stall
    assert st == mg.MUON_ETIMEOUT, mg.status_str(st)
    assert mg.muon_sync_status() == mg.MUON_OK
    # a fresh step on the same stream: succeeds and matches the oracle
    w = [to_device(h, torch) for h in Ws]
    mo = [torch.zeros_like(x) for x in w]
    mg.muon_step(w, gr, mo, lr=0.02, beta=0.95, wd=0.1, nesterov=False)
    assert mg.muon_sync_status() == mg.MUON_OK
    for i, (r, c) in enumerate(shapes):
        ref = orc.muon_step(Ws[i].data, zeros_matrix(r, c, "bf16").data, Gs[i].data, lr=0.02, beta=0.95,
                            wd=0.1, nesterov=False, path="gram", param_dtype="bf16", mom_dtype="bf16")
        delta = ref["W_exact"] - ref["W_old"]
        err = np.linalg.norm(to_f64(w[i]) - ref["W_exact"]) / np.linalg.norm(delta)
        q = np.linalg.norm(ref["W_new"] - ref["W_exact"]) / np.linalg.norm(delta)
        assert err <= TOL["bf16"] + q, (i, err, q)
