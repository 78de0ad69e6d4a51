"""Pins of the CPU oracle to facts outside itself.

Each check compares the oracle with something it does not compute itself:
the pages' printed product counts, an SVD identity (numpy's LAPACK SVD), a
scalar recursion carried out in 60-digit decimal arithmetic, closed forms of
the momentum and update rules, and a library bf16 conversion.  The mutation
tests at the end plant a plausible mistake in the oracle (on the CPU) and show
that at least one pin catches it.
"""
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

from oracle import muon_oracle as orc
from workloads import normal_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _gauss(seed, m, n):
    return normal_f64(seed, 0, m * n).reshape(m, n)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _svd_closed_form(U, coeffs, steps, eps=orc.EPS):
    """NS acts on each singular value alone: O = Uu diag(phi(s / (||U||_F + eps))) V^T,
    with phi the scalar polynomial a s + b s^3 + c s^5 applied ``steps`` times."""
    a, b, c = coeffs
    Uu, s, Vt = np.linalg.svd(U, full_matrices=False)
    t = s / (math.sqrt(float(np.sum(U * U))) + eps)
    for _ in range(steps):
        t = a * t + b * t ** 3 + c * t ** 5
    return (Uu * t) @ Vt


# ---------------------------------------------------------------------------
# the checks (each returns an error figure; the tests bound it)
# ---------------------------------------------------------------------------

def check_gram_equals_plain(shapes=((256, 1024), (128, 512), (64, 256), (96, 300), (40, 40))):
    worst = 0.0
    for i, (m, n) in enumerate(shapes):
        U = _gauss(11 + i, m, n)
        worst = max(worst, _rel(orc.orthogonalize(U, "gram"), orc.orthogonalize(U, "plain")))
    return worst


def check_svd_closed_form():
    worst = 0.0
    cases = [((64, 256), "plain", orc.QUINTIC, 5, (2, 2, 1)),
             ((64, 256), "gram", orc.QUINTIC, 5, (2, 2, 1)),
             ((48, 48), "plain", orc.QUINTIC, 5, (2, 2, 1)),
             ((48, 48), "gram", orc.QUINTIC, 5, (2, 3)),
             ((200, 37), "gram", orc.QUINTIC, 5, (2, 2, 1)),     # tall: oriented
             ((200, 37), "plain", orc.QUINTIC, 5, (2, 2, 1)),
             ((30, 70), "gram", orc.CUBIC, 7, (3, 4)),
             ((30, 70), "plain", (2.0, -1.3, 0.4), 3, (1, 1, 1))]
    for i, ((m, n), path, coeffs, steps, segs) in enumerate(cases):
        U = _gauss(21 + i, m, n)
        O = orc.orthogonalize(U, path, coeffs, steps, segs)
        worst = max(worst, _rel(O, _svd_closed_form(U, coeffs, steps)))
    return worst


def check_ns_band(shapes=((256, 1024), (128, 512), (96, 300), (1024, 256))):
    """Singular values of the 5-step quintic output of a random rectangular
    Gaussian matrix (long side >= 2x short side) lie in the NS band."""
    lo, hi = 1.0, 0.0
    for i, (m, n) in enumerate(shapes):
        for path in ("plain", "gram"):
            s = np.linalg.svd(orc.orthogonalize(_gauss(31 + i, m, n), path), compute_uv=False)
            lo, hi = min(lo, s.min()), max(hi, s.max())
    return lo, hi


def check_polar_convergence(steps):
    """Cubic coefficients (1.5, -0.5, 0) drive O to the polar factor U V^T."""
    U = _gauss(41, 8, 16)
    Uu, _, Vt = np.linalg.svd(U, full_matrices=False)
    polar = Uu @ Vt
    segs = tuple([steps // 4] * 3 + [steps - 3 * (steps // 4)])
    return (_rel(orc.orthogonalize(U, "plain", orc.CUBIC, steps), polar),
            _rel(orc.orthogonalize(U, "gram", orc.CUBIC, steps, segs), polar))


def _decimal_trajectory(vals, steps):
    getcontext().prec = 60
    a, b, c = (Decimal(x) for x in orc.QUINTIC)
    nrm = Decimal(sum(v * v for v in vals)).sqrt() + Decimal(orc.EPS)
    t = [Decimal(v) / nrm for v in vals]
    out = [list(t)]
    for _ in range(steps):
        t = [a * s + b * s ** 3 + c * s ** 5 for s in t]
        out.append(list(t))
    return out


def check_hand_diag34():
    """X = diag(3, 4): each singular value follows the scalar recursion alone."""
    traj = _decimal_trajectory([3, 4], 5)
    worst = 0.0
    seg_for = {1: (1,), 2: (2,), 3: (2, 1), 4: (2, 2), 5: (2, 2, 1)}
    c, s = math.cos(0.7), math.sin(0.7)
    R1 = np.array([[c, -s], [s, c]])
    R2 = np.array([[c * c - s * s, -2 * s * c], [2 * s * c, c * c - s * s]])
    for k in range(1, 6):
        expect = np.diag([float(v) for v in traj[k]])
        for path in ("plain", "gram"):
            O = orc.orthogonalize(np.diag([3.0, 4.0]), path, steps=k, segments=seg_for[k])
            worst = max(worst, float(np.max(np.abs(O - expect))))
            Or = orc.orthogonalize(R1 @ np.diag([3.0, 4.0]) @ R2.T, path, steps=k, segments=seg_for[k])
            worst = max(worst, float(np.max(np.abs(Or - R1 @ expect @ R2.T))))
    return worst


def check_momentum_closed_form(beta=0.95, k=7):
    """Constant gradient g from zero state: M_k = g (1 - beta^k) / (1 - beta);
    Nesterov: U_k = g + beta M_k."""
    g = _gauss(51, 3, 5)
    M = np.zeros_like(g)
    worst = 0.0
    for step in range(1, k + 1):
        M, U = orc.momentum(M, g, beta, nesterov=True)
        Mk = g * (1 - beta ** step) / (1 - beta)
        worst = max(worst, _rel(M, Mk), _rel(U, g + beta * Mk))
    M = np.zeros_like(g)
    for step in range(1, k + 1):
        M, U = orc.momentum(M, g, beta, nesterov=False)
    worst = max(worst, _rel(U, g * (1 - beta ** k) / (1 - beta)))
    return worst


def check_update_special_cases():
    W = _gauss(61, 20, 50)
    O = _gauss(62, 20, 50)
    e1 = float(np.max(np.abs(orc.weight_update(W, O, lr=0.0, wd=0.1) - W)))
    e2 = _rel(orc.weight_update(W, O, lr=0.02, wd=0.0) - W, -0.02 * 0.2 * math.sqrt(50) * O)
    e3 = _rel(orc.weight_update(W, np.zeros_like(W), lr=0.02, wd=0.1), W * (1 - 0.002))
    Wt = _gauss(63, 50, 20)   # tall: scale uses max(rows, cols) = 50 as well
    e4 = _rel(orc.weight_update(Wt, O.T, lr=0.02, wd=0.0) - Wt, -0.02 * 0.2 * math.sqrt(50) * O.T)
    return max(e1, e2, e3, e4)


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


# ---------------------------------------------------------------------------
# tests
# ---------------------------------------------------------------------------

def test_gram_equals_plain_fp64():
    assert check_gram_equals_plain() <= 1e-10


def test_svd_closed_form():
    assert check_svd_closed_form() <= 1e-11


def test_ns_band_rectangular():
    lo, hi = check_ns_band()
    assert 0.68 <= lo and hi <= 1.135, (lo, hi)


def test_square_gaussian_is_outside_band_but_matches_svd():
    """Square Gaussian inputs keep tiny singular values below the band after 5
    steps; the closed form still holds for them."""
    U = _gauss(71, 128, 128)
    s = np.linalg.svd(orc.orthogonalize(U, "plain"), compute_uv=False)
    assert s.min() < 0.68
    assert _rel(orc.orthogonalize(U, "plain"), _svd_closed_form(U, orc.QUINTIC, 5)) < 1e-11


def test_polar_convergence_cubic():
    e5 = check_polar_convergence(5)
    e20 = check_polar_convergence(20)
    assert min(e5) > 1e-3              # not there after 5 cubic steps
    assert max(e20) < 1e-10, e20


def test_quintic_is_not_polar():
    """f(1) = a + b + c = 0.701: the quintic map does not fix sigma = 1."""
    a, b, c = orc.QUINTIC
    assert abs((a + b + c) - 0.701) < 1e-12
    U = _gauss(42, 8, 16)
    Uu, _, Vt = np.linalg.svd(U, full_matrices=False)
    O = orc.orthogonalize(U, "gram")
    assert _rel(O, Uu @ Vt) > 0.05
    D = Uu.T @ O @ Vt.T                  # same singular vectors: U^T O V is diagonal
    assert np.max(np.abs(D - np.diag(np.diag(D)))) < 1e-12


def test_hand_diag34():
    assert check_hand_diag34() < 1e-13


def test_hand_2x3():
    """X = [[1,2,0],[0,1,1]]: plain and Gram 2+2+1 agree with the SVD form."""
    X = np.array([[1.0, 2.0, 0.0], [0.0, 1.0, 1.0]])
    expect = _svd_closed_form(X, orc.QUINTIC, 5)
    for path in ("plain", "gram"):
        assert np.max(np.abs(orc.orthogonalize(X, path) - expect)) < 1e-13


def test_segments_all_ones_is_plain():
    U = _gauss(81, 64, 160)
    Ga = orc.orthogonalize(U, "gram", segments=(1, 1, 1, 1, 1))
    assert _rel(Ga, orc.orthogonalize(U, "plain")) < 1e-13
    la = orc.ns_product_log(64, 160, "gram", segments=(1, 1, 1, 1, 1))
    lp = orc.ns_product_log(64, 160, "plain")
    assert la.counts(64) == lp.counts(64)
    assert la.nominal_flops() == lp.nominal_flops()


def test_orientation_transpose_invariance():
    U = _gauss(91, 60, 170)
    for path in ("plain", "gram"):
        assert _rel(orc.orthogonalize(U.T, path), orc.orthogonalize(U, path).T) < 1e-13


def test_momentum_closed_form():
    assert check_momentum_closed_form() < 1e-14


def test_update_special_cases():
    assert check_update_special_cases() < 1e-14


def test_product_counts_match_pages():
    g = _read_golden("pages_ns_cost_2560x9728.txt")
    m, n = int(g["m"]), int(g["n"])
    lp = orc.ns_product_log(m, n, "plain")
    lg = orc.ns_product_log(m, n, "gram", segments=(2, 2, 1))
    assert lp.counts(m) == (g["plain_long"], g["plain_square"])
    assert lg.counts(m) == (g["gram_long"], g["gram_square"])
    assert round(lp.nominal_flops() / 1e12, 3) == g["plain_tflops"]
    assert round(lg.nominal_flops() / 1e12, 3) == g["gram_tflops"]
    red = 100.0 * (1 - lg.nominal_flops() / lp.nominal_flops())
    assert round(red, 1) == g["reduction_percent"]


def test_product_counts_closed_forms():
    """Plain: 20 m^2 n + 10 m^3 nominal; Gram 2+2+1: 12 m^2 n + 22 m^3.
    Algorithmic (symmetric results counted half): 15 m^2 n + 5 m^3 and
    9 m^2 n + 11 m^3."""
    for (m, n) in ((128, 512), (2560, 9728), (4096, 14336), (300, 300)):
        lp = orc.ns_product_log(m, n, "plain")
        lg = orc.ns_product_log(m, n, "gram")
        assert lp.nominal_flops() == 20 * m * m * n + 10 * m ** 3
        assert lg.nominal_flops() == 12 * m * m * n + 22 * m ** 3
        assert lp.algorithmic_flops() == 15 * m * m * n + 5 * m ** 3
        assert lg.algorithmic_flops() == 9 * m * m * n + 11 * m ** 3


def test_round_bf16_matches_library_conversion():
    torch = pytest.importorskip("torch")
    x = np.concatenate([
        normal_f64(5, 0, 20000) * 0.03,
        np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -100 * 1.5,
                  65504.0, 1e30, -3.0e-20]),
    ]).astype(np.float32).astype(np.float64)
    lib = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(orc.round_bf16(x), lib)
    assert np.array_equal(orc.round_bf16(np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8])),
                          np.array([1.0, 1 + 2.0 ** -6]))


def test_muon_step_composition():
    """muon_step = momentum -> orthogonalize -> update -> round, on stored bytes."""
    from workloads import gen_matrix
    W = gen_matrix(5, 1, 40, 90, 0.02, "bf16")
    G = gen_matrix(5, 0, 40, 90, 0.02, "bf16")
    M = gen_matrix(5, 3, 40, 90, 0.01, "bf16")
    r = orc.muon_step(W.data, M.data, G.data, lr=0.02, beta=0.95, wd=0.1, nesterov=True,
                      path="gram", param_dtype="bf16", mom_dtype="bf16")
    G64, M64, W64 = (orc.to_f64(a.data, "bf16") for a in (G, M, W))
    M1 = 0.95 * M64 + G64
    O = _svd_closed_form(G64 + 0.95 * M1, orc.QUINTIC, 5)
    assert _rel(r["O"], O) < 1e-12
    W1 = W64 * (1 - 0.002) - 0.02 * 0.2 * math.sqrt(90) * O
    assert _rel(r["W_exact"], W1) < 1e-12
    assert np.array_equal(r["M_new"], orc.round_bf16(M1))


# ---------------------------------------------------------------------------
# planted mistakes: each mutant must break at least one pin
# ---------------------------------------------------------------------------

def _mut_gram_skip_apply(X, coeffs=orc.QUINTIC, segments=(2, 2, 1), log=None):
    a, b, c = coeffs
    m = X.shape[0]
    for i, L in enumerate(segments):
        G = X @ X.T
        Q = None
        for j in range(1, L + 1):
            P = a * np.eye(m) + b * G + c * G @ G
            Q = P if j == 1 else P @ Q
            if j < L:
                G = P @ G @ P
        if i == len(segments) - 1:          # earlier segments' transforms dropped
            X = Q @ X
    return X


def _mut_gram_sign(X, coeffs=orc.QUINTIC, segments=(2, 2, 1), log=None):
    a, b, c = coeffs
    return _orig_gram(X, (a, b, -c), segments)


def _mut_gram_single_g(X, coeffs=orc.QUINTIC, segments=(2, 2, 1), log=None):
    a, b, c = coeffs
    m = X.shape[0]
    for L in segments:
        G = X @ X.T
        Q = None
        for j in range(1, L + 1):
            P = a * np.eye(m) + b * G + c * G @ G
            Q = P if j == 1 else P @ Q
            if j < L:
                G = P @ G                    # dropped the second P
        X = Q @ X
    return X


def _mut_plain_drop_a(X, coeffs=orc.QUINTIC, steps=5, log=None):
    a, b, c = coeffs
    for _ in range(steps):
        A = X @ X.T
        X = (b * A + c * A @ A) @ X + X      # a replaced by 1
    return X


def _mut_norm_max(X, eps=orc.EPS):
    return X / (np.max(np.abs(X)) + eps)


def _mut_momentum_lerp(M, G, beta, nesterov):
    M_new = beta * M + (1 - beta) * G
    return M_new, (G + beta * M_new if nesterov else M_new)


def _mut_nesterov_old(M, G, beta, nesterov):
    M_new = beta * M + G
    return M_new, (G + beta * M if nesterov else M_new)


def _mut_update_min(W, O, lr, wd):
    s = 0.2 * math.sqrt(min(W.shape))
    return W * (1.0 - lr * wd) - lr * s * O


_orig_gram = orc.ns_gram


def _all_pins_hold():
    with np.errstate(all="ignore"):
        return _all_pins_hold_inner()


def _all_pins_hold_inner():
    try:
        ok = (check_gram_equals_plain() <= 1e-10 and check_svd_closed_form() <= 1e-11
              and check_hand_diag34() < 1e-13 and check_momentum_closed_form() < 1e-14
              and check_update_special_cases() < 1e-14)
        lo, hi = check_ns_band(((96, 300),))
        return ok and 0.68 <= lo and hi <= 1.135
    except Exception:
        return False


@pytest.mark.parametrize("name,target,mutant", [
    ("gram_skip_apply", "ns_gram", _mut_gram_skip_apply),
    ("gram_sign", "ns_gram", _mut_gram_sign),
    ("gram_single_g", "ns_gram", _mut_gram_single_g),
    ("plain_drop_a", "ns_plain", _mut_plain_drop_a),
    ("norm_max", "frobenius_normalise", _mut_norm_max),
    ("momentum_lerp", "momentum", _mut_momentum_lerp),
    ("nesterov_old", "momentum", _mut_nesterov_old),
    ("update_min", "weight_update", _mut_update_min),
])
def test_planted_mistake_is_caught(monkeypatch, name, target, mutant):
    assert _all_pins_hold()
    monkeypatch.setattr(orc, target, mutant)
    assert not _all_pins_hold(), name


# ---------------------------------------------------------------------------
# binary16 storage (the fp16 working type): the decoder and the rounding are
# written from the IEEE format; numpy's own half conversions are independent
# implementations of the same definition.
# ---------------------------------------------------------------------------

def test_f16_decode_all_bit_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    mine = orc.f16_bits_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    assert np.array_equal(mine[finite], ref[finite])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[np.isinf(ref)], ref[np.isinf(ref)])


def test_f16_rounding_matches_ieee():
    r = orc.round_f16
    # ties to even at 1, above the largest finite value, and in the subnormals
    assert r(np.array(1.0 + 2.0 ** -11)) == 1.0
    assert r(np.array(1.0 + 3 * 2.0 ** -11)) == 1.0 + 2.0 ** -9
    assert r(np.array(65519.0)) == 65504.0
    assert np.isinf(r(np.array(65520.0))) and r(np.array(-65520.0)) < 0
    assert r(np.array(2.0 ** -25)) == 0.0
    assert r(np.array(3 * 2.0 ** -26)) == 2.0 ** -24
    assert r(np.array(2.0 ** -14 - 2.0 ** -25)) == 2.0 ** -14     # tie between the last subnormal and 2^-14
    # random values over the whole range against numpy's double -> half
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 17, 200000)),
        (rng.integers(-2048, 2048, 20000) + 0.5) * np.exp2(rng.integers(-24, 5, 20000)).astype(np.float64)])
    with np.errstate(over="ignore"):                                # values past 65520 become inf
        want = x.astype(np.float16).astype(np.float64)
    got = r(x)
    same = (got == want) | (np.isinf(got) & np.isinf(want) & (np.sign(got) == np.sign(want)))
    assert same.all(), x[~same][:5]


def test_f16_storage_roundtrip():
    x = orc.round_f16(np.linspace(-3, 3, 1001))
    assert np.array_equal(orc.to_f64(orc.f16_bits_from_f64(x), "f16"), x)
    assert np.array_equal(orc.round_to(x, "f16"), x)
