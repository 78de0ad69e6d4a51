"""CUDA path vs the fp64 CPU oracle on identical seeded bytes.

Bars (relative Frobenius error of the ortho output; singular values sorted):
fp32 path 1e-4, bf16 path 2e-2, max singular-value deviation 0.05.  For
muon_step the updated weights are compared as
||W'_gpu - W'_exact|| / ||W'_exact - W|| <= tol + q, q being the oracle's own
storage-rounding term, and momentum within one storage ulp of round(beta M + G).
Sizes span several tiles and ragged tails; edge cases cover vectors, tiny and
unaligned shapes, mixed orientation in one bucket, zero and non-finite input.
"""
import math

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
    pkg.muon_set_ns_config(pkg.QUINTIC, 5, (2, 2, 1), pkg.MUON_PATH_AUTO)


def _ortho_case(mg, rows, cols, batch, dtype, segments, seed, std=1.0):
    mats = [gen_matrix(seed + b, 0, rows, cols, std, dtype) for b in range(batch)]
    x = torch.stack([to_device(h, torch) for h in mats]).contiguous()
    mg.muon_ns_orthogonalize(x, mg.QUINTIC, 5, segments)
    assert mg.muon_sync_status() == mg.MUON_OK
    path = "gram" if segments else "plain"
    worst_f, worst_s = 0.0, 0.0
    for b, h in enumerate(mats):
        O_ref = orc.orthogonalize(orc.to_f64(h.data, dtype), path, segments=segments or (2, 2, 1))
        O = to_f64(x[b])
        worst_f = max(worst_f, rel_fro(O, O_ref))
        worst_s = max(worst_s, sigma_dev(O, O_ref))
    return worst_f, worst_s


@pytest.mark.parametrize("rows,cols,batch", [(256, 1024, 1), (200, 37, 2), (96, 300, 1), (64, 160, 3)])
@pytest.mark.parametrize("segments", [None, (2, 2, 1)])
def test_orthogonalize_fp32(mg, rows, cols, batch, segments):
    f, s = _ortho_case(mg, rows, cols, batch, "f32", segments, 100)
    assert f <= TOL["f32"], f
    assert s <= SIGMA_TOL


@pytest.mark.parametrize("fp32_tc", ["0", "auto"])
@pytest.mark.parametrize("rows,cols", [(1100, 2200), (2200, 1100)])
@pytest.mark.parametrize("segments", [None, (2, 2, 1)])
def test_orthogonalize_fp32_large_tiles(mg, monkeypatch, fp32_tc, rows, cols, segments):
    """fp32 NS whose long products have more 128x128 tiles than SMs: on FFMA
    (the large-tile kernel for them, the split-K one for the m x m products),
    and as the automatic choice takes it at this size (three-pass TF32 with
    chunked accumulation)."""
    if fp32_tc == "0":
        monkeypatch.setenv("MUON_FP32_TC", "0")
    else:
        monkeypatch.delenv("MUON_FP32_TC", raising=False)
    f, s = _ortho_case(mg, rows, cols, 1, "f32", segments, 140)
    assert f <= TOL["f32"], f
    assert s <= SIGMA_TOL


@pytest.mark.parametrize("small", ["1", "0"])
@pytest.mark.parametrize("rows,cols,batch", [
    (256, 1024, 1), (128, 512, 4), (256, 256, 2), (300, 1000, 1), (1000, 296, 1), (8, 16, 2),
    (2, 3, 1), (1, 64, 1), (37, 200, 2), (130, 130, 1), (512, 128, 3), (96, 300, 2)])
@pytest.mark.parametrize("segments", [None, (2, 2, 1), (2, 3)])
def test_orthogonalize_bf16(mg, monkeypatch, rows, cols, batch, segments, small):
    """small=1: shapes that fit run the one-CTA-per-matrix kernel; small=0: the
    general product path for every shape."""
    monkeypatch.setenv("MUON_SMALL", small)
    f, s = _ortho_case(mg, rows, cols, batch, "bf16", segments, 200, std=0.03)
    assert f <= TOL["bf16"], f
    assert s <= SIGMA_TOL, s


def _step_case(mg, shapes, dtype, mom_dtype, path_code, nesterov, seed0, grad_std, steps=1):
    """Runs `steps` muon_step calls (fresh gradient each) and compares each step."""
    Ws = [gen_matrix(seed0 + i, 1, r, c, 0.02, dtype) for i, (r, c) in enumerate(shapes)]
    Ms = [zeros_matrix(r, c, mom_dtype) for (r, c) in shapes]
    w = [to_device(h, torch) for h in Ws]
    mo = [to_device(h, torch) for h in Ms]
    mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), path_code)
    results = []
    for st in range(steps):
        Gs = [gen_matrix(seed0 + i, 0 if st == 0 else 2, r, c, grad_std, dtype) for i, (r, c) in enumerate(shapes)]
        g = [to_device(h, torch) for h in Gs]
        W_host = [to_f64(t) for t in w]
        M_host = [to_f64(t) for t in mo]
        mg.muon_step(w, g, mo, lr=0.02, beta=0.95, wd=0.1, nesterov=nesterov)
        assert mg.muon_sync_status() == mg.MUON_OK
        for i, (r, c) in enumerate(shapes):
            path = mg.muon_last_path(r, c, mg.MUON_BF16 if dtype == "bf16" else mg.MUON_F32)
            pname = "gram" if path == mg.MUON_PATH_GRAM else "plain"
            # the library receives fp32 hyper-parameters; the oracle gets the same values
            ref = orc.muon_step(_store(W_host[i], dtype), _store(M_host[i], mom_dtype), Gs[i].data,
                                lr=F32(0.02), beta=F32(0.95), wd=F32(0.1), nesterov=nesterov, path=pname,
                                param_dtype=dtype, mom_dtype=mom_dtype)
            d = ref["W_exact"] - ref["W_old"]
            err = np.linalg.norm(to_f64(w[i]) - ref["W_exact"]) / np.linalg.norm(d)
            q = np.linalg.norm(ref["W_new"] - ref["W_exact"]) / np.linalg.norm(d)
            m_gpu = to_f64(mo[i])
            ulp = _ulp(ref["M_new"], mom_dtype)
            m_ok = bool(np.all(np.abs(m_gpu - ref["M_new"]) <= ulp))
            results.append((err, q, m_ok, pname))
    return results


def F32(x):
    return float(np.float32(x))


def _store(x64, dtype):
    if dtype == "f32":
        return x64.astype(np.float32)
    return orc.bf16_bits_from_f64(orc.round_bf16(x64))


def _ulp(x, dtype):
    bits = 8 if dtype == "bf16" else 24
    ax = np.maximum(np.abs(x), 1e-30)
    return np.ldexp(1.0, (np.floor(np.log2(ax)).astype(int) - (bits - 1)))


@pytest.mark.parametrize("path", ["plain", "gram"])
def test_step_single_256x1024_f32(mg, path):
    code = mg.MUON_PATH_PLAIN if path == "plain" else mg.MUON_PATH_GRAM
    for err, q, m_ok, pname in _step_case(mg, [(256, 1024)], "f32", "f32", code, False, 1000, 1.0, steps=2):
        assert pname == path
        assert err <= TOL["f32"] + q, (err, q)
        assert m_ok


@pytest.mark.parametrize("path", ["plain", "gram"])
def test_step_bf16_mixed_shapes_two_steps(mg, path):
    code = mg.MUON_PATH_PLAIN if path == "plain" else mg.MUON_PATH_GRAM
    shapes = [(192, 640), (640, 192), (192, 640), (96, 96), (37, 200), (1, 40)]
    for err, q, m_ok, _ in _step_case(mg, shapes, "bf16", "bf16", code, True, 3000, 0.02, steps=2):
        assert err <= TOL["bf16"] + q, (err, q)
        assert m_ok


def test_step_bf16_params_f32_momentum(mg):
    shapes = [(256, 896), (896, 256)]
    for err, q, m_ok, _ in _step_case(mg, shapes, "bf16", "f32", mg.MUON_PATH_AUTO, False, 5000, 0.0316, steps=2):
        assert err <= TOL["bf16"] + q, (err, q)
        assert m_ok


def test_zero_gradient_only_decays(mg):
    W = gen_matrix(7000, 1, 128, 384, 0.02, "bf16")
    w = to_device(W, torch)
    g = torch.zeros_like(w)
    mo = torch.zeros_like(w)
    mg.muon_step([w], [g], [mo], lr=0.02, beta=0.95, wd=0.1, nesterov=False)
    assert mg.muon_sync_status() == mg.MUON_OK
    expect = orc.round_bf16(orc.to_f64(W.data, "bf16") * (1 - 0.002))
    got = to_f64(w)
    assert np.max(np.abs(got - expect) / np.maximum(np.abs(expect), 1e-30)) <= 2.0 ** -8


def test_nonfinite_gradient_is_reported(mg):
    w = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros_like(w)
    g[3, 5] = float("inf")
    mo = torch.zeros_like(w)
    mg.muon_step([w], [g], [mo], lr=0.02, beta=0.95, wd=0.1, nesterov=False)
    assert mg.muon_sync_status() == mg.MUON_ENONFINITE
    assert mg.muon_sync_status() == mg.MUON_OK        # the word is cleared on read


def test_launch_count_matches_plan(mg, monkeypatch):
    monkeypatch.setenv("MUON_SMALL", "0")
    w = torch.randn((128, 512), device="cuda").to(torch.bfloat16)
    g, mo = torch.randn_like(w) * 0.01, torch.zeros_like(w)
    # one prep launch (it finalises the norm itself), then the NS products
    for path, expect in ((mg.MUON_PATH_GRAM, 1 + 3 + 5 + 2 + 4 + 3), (mg.MUON_PATH_PLAIN, 1 + 5 * 3)):
        mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), path)
        before = mg.muon_launch_count()
        mg.muon_step([w], [g], [mo], lr=0.02, beta=0.95, wd=0.1, nesterov=False)
        assert mg.muon_launch_count() - before == expect
    assert mg.muon_sync_status() == mg.MUON_OK


def test_kernel_timing_record(mg):
    w = torch.randn((256, 1024), device="cuda").to(torch.bfloat16)
    g, mo = torch.randn_like(w) * 0.01, torch.zeros_like(w)
    mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_GRAM)
    mg.muon_kernel_timing_read()
    mg.muon_set_kernel_timing(True)
    mg.muon_step([w], [g], [mo], lr=0.02, beta=0.95, wd=0.1, nesterov=False)
    rec = mg.muon_kernel_timing_read()
    mg.muon_set_kernel_timing(False)
    assert rec["gemm_tc_syrk"][0] == 3 and rec["gemm_tc_apply"][0] == 2 and rec["gemm_tc_apply_update"][0] == 1
    nom, alg = mg.muon_ns_flops(256, 1024, mg.MUON_PATH_GRAM, (2, 2, 1))
    tot = sum(v[2] for k, v in rec.items() if k.startswith("gemm"))
    assert abs(tot - alg) / alg < 1e-12
    assert all(v[1] > 0 for v in rec.values())


def test_autotune_and_cache_round_trip(mg, tmp_path):
    mg.muon_set_ns_config(mg.QUINTIC, 5, (2, 2, 1), mg.MUON_PATH_AUTO)
    mg.muon_autotune([(256, 768), (768, 256), (128, 128)], mg.MUON_BF16)
    p = tmp_path / "tune.tsv"
    mg.muon_tune_save(str(p))
    assert mg.muon_tune_load(str(p)) >= 2
    w = torch.randn((768, 256), device="cuda").to(torch.bfloat16)
    g, mo = torch.randn_like(w) * 0.01, torch.zeros_like(w)
    mg.muon_step([w], [g], [mo], lr=0.02, beta=0.95, wd=0.1, nesterov=False)
    assert mg.muon_last_path(256, 768, mg.MUON_BF16) in (mg.MUON_PATH_PLAIN, mg.MUON_PATH_GRAM)
    assert mg.muon_sync_status() == mg.MUON_OK
    text = p.read_text().splitlines()
    assert text[0] == "muon-tune v4" and len(text) >= 3
    # a corrupt line is skipped, the rest loads
    p.write_text("\n".join(text + ["garbage\tline"]) + "\n")
    assert mg.muon_tune_load(str(p)) == len(text) - 1


@pytest.mark.parametrize("path", ["plain", "gram"])
@pytest.mark.parametrize("mom_dtype", ["bf16", "f32"])
def test_small_bucket_fused_step(mg, monkeypatch, path, mom_dtype):
    """Buckets of small matrices (mixed orientation) run as one fused launch
    with per-CTA work lists and match the oracle on two consecutive steps."""
    monkeypatch.setenv("MUON_SMALL", "1")
    code = mg.MUON_PATH_PLAIN if path == "plain" else mg.MUON_PATH_GRAM
    shapes = [(128, 512), (512, 128), (128, 512), (128, 384)]
    before = mg.muon_launch_count()
    res = _step_case(mg, shapes, "bf16", mom_dtype, code, True, 8000, 0.0316, steps=2)
    # two buckets (128x512 and 128x384) share one launch per step
    assert mg.muon_launch_count() - before == 2
    for err, q, m_ok, pname in res:
        assert pname == path
        assert err <= TOL["bf16"] + q, (err, q)
        assert m_ok


@pytest.mark.parametrize("mom_dtype", ["bf16", "f32"])
def test_fused_256_rows_step(mg, monkeypatch, mom_dtype):
    """Plain NS of 128 < m <= 256, n <= 256 matrices in the 256-row form of the
    one-CTA-per-matrix kernel (A kept as three symmetric blocks, A01 read
    transposed): square, ragged and transposed shapes, two steps."""
    monkeypatch.setenv("MUON_SMALL", "1")
    shapes = [(256, 256), (192, 256), (256, 192), (256, 200), (130, 130), (256, 256)]
    before = mg.muon_launch_count()
    res = _step_case(mg, shapes, "bf16", mom_dtype, mg.MUON_PATH_PLAIN, True, 8600, 0.0316, steps=2)
    # buckets 256x256, 192x256, 200x256, 130x130 (both forms) share one launch per step
    assert mg.muon_launch_count() - before == 2
    for err, q, m_ok, pname in res:
        assert pname == "plain"
        assert err <= TOL["bf16"] + q, (err, q)
        assert m_ok


def test_small_fused_zero_and_tiny(mg, monkeypatch):
    monkeypatch.setenv("MUON_SMALL", "1")
    for shape in ((1, 8), (3, 5), (64, 64)):
        for err, q, m_ok, _ in _step_case(mg, [shape], "bf16", "bf16", mg.MUON_PATH_PLAIN, False, 9000, 0.02):
            assert err <= TOL["bf16"] + q, (shape, err, q)
            assert m_ok
    w = gen_matrix(9100, 1, 96, 200, 0.02, "bf16")
    wt = to_device(w, torch)
    g = torch.zeros_like(wt)
    mo = torch.zeros_like(wt)
    mg.muon_step([wt], [g], [mo], lr=0.02, beta=0.95, wd=0.1, nesterov=False)
    assert mg.muon_sync_status() == mg.MUON_OK
    expect = orc.round_bf16(orc.to_f64(w.data, "bf16") * (1 - 0.002))
    assert np.max(np.abs(to_f64(wt) - expect) / np.maximum(np.abs(expect), 1e-30)) <= 2.0 ** -8


@pytest.mark.parametrize("dense", ["0", "1"])
@pytest.mark.parametrize("path", ["plain", "gram"])
def test_symmetric_products_both_forms(mg, monkeypatch, dense, path):
    """The Gram-space products as lower-triangle tiles with mirroring, or as
    all tiles, give the same update within the bar."""
    monkeypatch.setenv("MUON_SYM_DENSE", dense)
    monkeypatch.setenv("MUON_SMALL", "0")
    code = mg.MUON_PATH_PLAIN if path == "plain" else mg.MUON_PATH_GRAM
    for err, q, m_ok, _ in _step_case(mg, [(256, 768), (768, 256), (200, 200)], "bf16", "bf16", code, True,
                                      9500, 0.02, steps=2):
        assert err <= TOL["bf16"] + q, (err, q)
        assert m_ok


def test_fused_many_matrices_per_cta(mg, monkeypatch):
    """More matrices than CTAs in one fused launch (both kernel forms): each
    CTA runs several in turn through the same shared memory (the write-out
    stage, the prologue's staged pieces, the slots); every matrix matches the
    oracle."""
    monkeypatch.setenv("MUON_SMALL", "1")
    shapes = [(128, 512)] * 160 + [(256, 256)] * 160
    for err, q, m_ok, _ in _step_case(mg, shapes, "bf16", "bf16", mg.MUON_PATH_AUTO, True, 8800, 0.0316):
        assert err <= TOL["bf16"] + q, (err, q)
        assert m_ok


def test_auto_path_few_rows_bf16(mg):
    """With bf16 X and fewer than 64 rows the automatic path choice takes the
    Gram path (the plain iteration errs by up to 4 % there), and the update
    meets the bf16 bar: matrices with 3, 4 and 32 rows in both orientations."""
    shapes = [(4, 549), (549, 4), (3, 168), (32, 1000), (1000, 32)]
    for err, q, m_ok, pname in _step_case(mg, shapes, "bf16", "bf16", mg.MUON_PATH_AUTO, True, 9400, 0.02):
        assert pname == "gram"
        assert err <= TOL["bf16"] + q, (err, q)
        assert m_ok


def test_fused_mixed_orientations_many_per_cta(mg, monkeypatch):
    """Wide and tall matrices of one oriented shape in the same bucket (the
    tall ones read and write the caller's transposed layout), both kernel
    forms and a 384-column shape in one launch, several matrices per CTA;
    then the ortho output (O written instead of a W update) for 400 matrices
    on 152 CTAs."""
    monkeypatch.setenv("MUON_SMALL", "1")
    shapes = [(128, 512), (512, 128), (256, 256), (128, 384)] * 60
    for err, q, m_ok, _ in _step_case(mg, shapes, "bf16", "bf16", mg.MUON_PATH_AUTO, False, 8600, 0.0316):
        assert err <= TOL["bf16"] + q, (err, q)
        assert m_ok
    f, s = _ortho_case(mg, 128, 512, 400, "bf16", (2, 2, 1), 8700)
    assert f <= TOL["bf16"], f
    assert s <= SIGMA_TOL


@pytest.mark.parametrize("side", [15, 17, 31, 33, 63])
def test_odd_squares_orthogonalize(mg, side):
    """Random odd squares in bf16, 12 per call, through the Gram path (the
    automatic choice for bf16 below 64 rows; TF32 Gram space): the oracle
    iterates on the same bf16 matrices, so the comparison holds the kernels
    to the bar without the rounding of U that a step adds (which alone can
    move a nearly singular square's output by more than 1%; pinned on the
    CPU in test_precision_policy.py)."""
    f, s = _ortho_case(mg, side, side, 12, "bf16", (2, 2, 1), 7300 + side)
    assert f <= TOL["bf16"], f
    assert s <= SIGMA_TOL


@pytest.mark.parametrize("mom_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("small", ["0", "1"])
def test_degenerate_shapes_step(mg, monkeypatch, small, mom_dtype):
    """The method's degenerate shapes: row and column vectors (a 1 x 1 Gram
    matrix), 2 x 2, odd widths that rule out 16-byte rows, and thin matrices,
    through both the product kernels and the fused one-CTA-per-matrix kernel,
    two steps each, against the oracle.  (Random odd squares are tested by
    test_odd_squares_orthogonalize on bf16 inputs: in a step, a nearly
    singular square can miss the bar through the rounding of U to bf16
    alone.)"""
    monkeypatch.setenv("MUON_SMALL", small)
    shapes = [(1, 4096), (4096, 1), (2, 2), (1, 7), (3, 1000), (17, 40), (8, 520)]
    for err, q, m_ok, _ in _step_case(mg, shapes, "bf16", mom_dtype, mg.MUON_PATH_AUTO, True, 9900, 0.02, steps=2):
        assert err <= TOL["bf16"] + q, (err, q)
        assert m_ok


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_maximum_side_step(mg, dtype):
    """Matrices at the largest accepted side (2^20): a row and a column
    vector and a few-row matrix, two steps against the oracle (one long
    k-loop in XX^T, thousands of tiles in the apply)."""
    side = 1 << 20
    shapes = [(1, side), (side, 1), (8, side)] if dtype == "bf16" else [(2, side), (side, 3)]
    for err, q, m_ok, _ in _step_case(mg, shapes, dtype, dtype, mg.MUON_PATH_AUTO, False, 9950, 0.02, steps=2):
        assert err <= TOL[dtype] + q, (err, q)
        assert m_ok
