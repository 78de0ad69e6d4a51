"""fp32 path with its products as three TF32 tensor-core passes
(MUON_FP32_TC=1: A' = [hi | hi | lo], B' = [hi | lo | hi], one TF32 product
over a tripled K) against the fp64 CPU oracle on identical seeded bytes, at the
fp32 bar (1e-4 relative Frobenius error).  Shapes cover several tiles, K not a
multiple of 4 (padded thirds) and both operand layouts of the apply (QX reads
X transposed through the split).  The bar holds at these sizes (3.6e-5 at
256x1024); the error grows with K (1.0e-4 at 768x3072, 1.4e-4 at 2048x8192),
which is why the path is opt-in."""
import pytest

from tests.gpu_util import SIGMA_TOL, TOL
from tests.test_gpu_parity import _ortho_case, _step_case

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def mg():
    import __graft_entry__
    __graft_entry__.build()
    import newton_schulz_frobenius_gb300 as pkg
    yield pkg
    pkg.muon_set_ns_config(pkg.QUINTIC, 5, (2, 2, 1), pkg.MUON_PATH_AUTO)


@pytest.mark.parametrize("rows,cols,batch", [(256, 1024, 1), (200, 37, 2), (96, 300, 1), (64, 160, 3), (37, 101, 2)])
@pytest.mark.parametrize("segments", [None, (2, 2, 1)])
def test_orthogonalize_tf32x3(mg, monkeypatch, rows, cols, batch, segments):
    monkeypatch.setenv("MUON_FP32_TC", "1")
    f, s = _ortho_case(mg, rows, cols, batch, "f32", segments, 300)
    assert f <= TOL["f32"], f
    assert s <= SIGMA_TOL


@pytest.mark.parametrize("path", ["plain", "gram"])
def test_step_single_256x1024_tf32x3(mg, monkeypatch, path):
    monkeypatch.setenv("MUON_FP32_TC", "1")
    code = mg.MUON_PATH_PLAIN if path == "plain" else mg.MUON_PATH_GRAM
    for err, q, m_ok, pname in _step_case(mg, [(256, 1024)], "f32", "f32", code, False, 1000, 1.0, steps=2):
        assert pname == path
        assert err <= TOL["f32"] + q, (err, q)
        assert m_ok


def test_tf32x3_runs_on_the_tensor_path(mg, monkeypatch):
    """Each product becomes two split launches and one TF32 tensor-core
    product; the recorded product work stays the fp32 product's."""
    w = torch.randn((256, 1024), device="cuda")
    g, mo = torch.randn_like(w) * 0.01, torch.zeros_like(w)
    mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_PLAIN)
    counts, recs = {}, {}
    for env in ("0", "1"):
        monkeypatch.setenv("MUON_FP32_TC", env)
        mg.muon_kernel_timing_read()
        mg.muon_set_kernel_timing(True)
        before = mg.muon_launch_count()
        mg.muon_step([w], [g], [mo], lr=0.02, beta=0.95, wd=0.1, nesterov=False)
        counts[env] = mg.muon_launch_count() - before
        recs[env] = mg.muon_kernel_timing_read()
        mg.muon_set_kernel_timing(False)
    assert mg.muon_sync_status() == mg.MUON_OK
    products = 5 * 3
    assert counts["1"] == counts["0"] + 2 * products
    assert recs["0"]["gemm_fp32"][0] == products
    assert "gemm_fp32" not in recs["1"] or recs["1"]["gemm_fp32"][0] == 0
    tc = sum(v[0] for k, v in recs["1"].items() if k.startswith("gemm_tc"))
    assert tc == products
    work0 = recs["0"]["gemm_fp32"][2]
    work1 = sum(v[2] for k, v in recs["1"].items() if k.startswith("gemm_tc"))
    assert abs(work1 - work0) / work0 < 1e-12
