"""fp32 path with its products as three TF32 tensor-core passes
(MUON_FP32_TC=1 forces it; large buckets take it by default: A' = [hi | hi |
lo], B' = [hi | lo | hi], one TF32 product over a tripled K, accumulated in
chunks added in round-to-nearest fp32) against the fp64 CPU oracle on
identical seeded bytes, at the fp32 bar (1e-4 relative Frobenius error).
Shapes cover several tiles, K not a multiple of 4 (padded thirds), both
operand layouts of the apply (QX reads X transposed through the split) and
the long K where whole-K accumulation missed the bar (1.0e-4 at 768x3072,
1.4e-4 at 2048x8192)."""
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


def _tf32_rn(x):
    m, e = torch.frexp(x.double())
    return torch.ldexp(torch.round(torch.ldexp(m, torch.tensor(11, device=x.device))), e - 11).float()


@pytest.mark.parametrize("tile_n", [0, 128, 256])
@pytest.mark.parametrize("M,N,K,batch,sym", [
    (256, 256, 8192, 1, True), (200, 328, 5000, 2, False), (384, 384, 384, 1, True),
    (130, 130, 2500, 3, True), (64, 520, 700, 1, False), (520, 776, 1500, 1, False)])
def test_chunked_tf32_product(mg, M, N, K, batch, sym, tile_n):
    """The TF32 product with chunked accumulation on three-pass operands
    ([hi|hi|lo] against [hi|lo|hi], as the fp32 path builds them): its error
    against the exact product of the fp32 values stays at the chunk's level
    for any K, where whole-K accumulation grows with K (about 1.2e-4 at
    K = 8192).  Ragged M, N and K, several matrices, symmetric launches,
    unpaired 128-wide tiles and 2-SM pairs (tile_n 256; 0 is the launcher's
    choice)."""
    g = torch.Generator(device="cuda").manual_seed(M + K)
    X = torch.randn((batch, M, K), generator=g, device="cuda")
    Y = X if sym else torch.randn((batch, N, K), generator=g, device="cuda")
    K4 = -(-K // 4) * 4

    def split(Z, order):
        hi = _tf32_rn(Z)
        lo = _tf32_rn(Z - hi)
        pad = torch.zeros(Z.shape[:-1] + (K4 - K,), device="cuda")
        hi, lo = torch.cat([hi, pad], -1), torch.cat([lo, pad], -1)
        return torch.cat([hi, hi, lo] if order == "hhl" else [hi, lo, hi], dim=-1).contiguous()

    A3, B3 = split(X, "hhl"), split(Y, "hlh")
    C = torch.full((batch, M, N), float("nan"), device="cuda")
    mg.muon_debug_gemm(A3, B3, C, b_kmajor=True, symmetric=sym, tf32_chunked=True, tile_n=tile_n)
    torch.cuda.synchronize()
    assert mg.muon_sync_status() == mg.MUON_OK
    ref = torch.matmul(X.double(), Y.double().transpose(1, 2))
    assert not torch.isnan(C).any()
    if sym:
        assert torch.equal(C, C.transpose(1, 2))
    err = ((C.double() - ref).norm() / ref.norm()).item()
    assert err < 1e-5, err


@pytest.mark.parametrize("rows,cols", [(768, 3072), (1024, 4096), (2048, 8192)])
@pytest.mark.parametrize("segments", [None, (2, 2, 1)])
def test_orthogonalize_tf32x3_long_k(mg, monkeypatch, rows, cols, segments):
    """Three-pass TF32 NS at the sizes where whole-K accumulation missed the
    fp32 bar (1.0e-4 at 768x3072, 1.4e-4 at 2048x8192): with chunked
    accumulation it holds."""
    monkeypatch.setenv("MUON_FP32_TC", "1")
    f, s = _ortho_case(mg, rows, cols, 1, "f32", segments, 320)
    assert f <= TOL["f32"], f
    assert s <= SIGMA_TOL


def test_step_fp32_large_auto(mg, monkeypatch):
    """A large fp32 matrix through muon_step with the automatic choices (the
    tensor path is taken at this size), two steps against the oracle, and
    the persistent group giving the same bytes."""
    monkeypatch.delenv("MUON_FP32_TC", raising=False)
    mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_AUTO)
    for err, q, m_ok, _ in _step_case(mg, [(1024, 4096), (4096, 1024)], "f32", "f32", mg.MUON_PATH_AUTO, True,
                                      1500, 1.0, steps=2):
        assert err <= TOL["f32"] + q, (err, q)
        assert m_ok
    g = torch.Generator(device="cuda").manual_seed(9)
    Wa = [torch.randn((1024, 4096), generator=g, device="cuda") * 0.02]
    Ga = [torch.randn((1024, 4096), generator=g, device="cuda")]
    Ma = [torch.zeros((1024, 4096), device="cuda")]
    Wb, Gb, Mb = [Wa[0].clone()], [Ga[0].clone()], [Ma[0].clone()]
    group = mg.MuonGroup(Wb, Gb, Mb)
    try:
        for _ in range(2):
            mg.muon_step(Wa, Ga, Ma, lr=0.02, beta=0.95, wd=0.1, nesterov=True)
            group.step(lr=0.02, beta=0.95, wd=0.1, nesterov=True)
        torch.cuda.synchronize()
        assert mg.muon_sync_status() == mg.MUON_OK
        assert torch.equal(Wa[0], Wb[0]) and torch.equal(Ma[0], Mb[0])
    finally:
        group.close()
