"""Pins of the AdamW oracle: the closed form for a constant gradient, special
cases, PyTorch's own CPU AdamW in fp64 (a library routine), and planted
mistakes that each break at least one pin."""
import numpy as np
import pytest

from oracle import adamw_oracle as ad
from workloads import normal_f64

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01)


def _vec(seed, n, scale=1.0):
    return normal_f64(seed, 0, n) * scale


def check_closed_form():
    p0, g = _vec(1, 257), _vec(2, 257, 0.1)
    p, m, v = p0.copy(), np.zeros(257), np.zeros(257)
    worst = 0.0
    for t in range(1, 9):
        p, m, v = ad.adamw_math(p, g, m, v, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, step=t)
        want = ad.constant_gradient_closed_form(p0, g, lr=1e-3, eps=1e-8, step=t)
        worst = max(worst, float(np.max(np.abs(p - want))))
    return worst


def check_special_cases():
    p, g = _vec(3, 100), _vec(4, 100)
    m, v = _vec(5, 100, 0.01), np.abs(_vec(6, 100, 0.01))
    p1, _, _ = ad.adamw_math(p, g, m, v, lr=0.0, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1, step=3)
    e1 = float(np.max(np.abs(p1 - p)))
    z = np.zeros(100)
    p2, m2, v2 = ad.adamw_math(p, z, z, z, lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.1, step=5)
    e2 = float(np.max(np.abs(p2 - p * (1 - 1e-3)))) + float(np.max(np.abs(m2))) + float(np.max(np.abs(v2)))
    return max(e1, e2)


def check_against_torch(steps=4):
    torch = pytest.importorskip("torch")
    n = 301
    p0 = _vec(7, n)
    p = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([p], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["wd"])
    q, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    worst = 0.0
    for t in range(1, steps + 1):
        g = _vec(100 + t, n, 0.3)
        p.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        q, m, v = ad.adamw_math(q, g, m, v, step=t, **HP)
        worst = max(worst, float(np.max(np.abs(p.detach().numpy() - q))))
    return worst


def test_closed_form():
    assert check_closed_form() < 1e-13


def test_special_cases():
    assert check_special_cases() < 1e-15


def test_matches_pytorch_adamw_fp64():
    assert check_against_torch() < 1e-14


def test_stored_step_rounding():
    from oracle import muon_oracle as orc
    from workloads import gen_matrix
    p = gen_matrix(9, 1, 4, 33, 0.02, "bf16")
    g = gen_matrix(9, 0, 4, 33, 0.1, "bf16")
    z = np.zeros((4, 33), np.float32)
    r = ad.adamw_step(p.data, g.data, z, z, step=1, param_dtype="bf16", state_dtype="f32", **HP)
    assert np.array_equal(r["p_new"], orc.round_bf16(r["p_exact"]))
    assert np.array_equal(r["m_new"], orc.round_f32(r["m_exact"]))


def _mut_no_bias_correction(p, g, m, v, *, lr, beta1, beta2, eps, wd, step):
    m1 = beta1 * m + (1 - beta1) * g
    v1 = beta2 * v + (1 - beta2) * g * g
    return p * (1 - lr * wd) - lr * m1 / (np.sqrt(v1) + eps), m1, v1


def _mut_coupled_decay(p, g, m, v, *, lr, beta1, beta2, eps, wd, step):
    g = g + wd * p
    m1 = beta1 * m + (1 - beta1) * g
    v1 = beta2 * v + (1 - beta2) * g * g
    mh, vh = m1 / (1 - beta1 ** step), v1 / (1 - beta2 ** step)
    return p - lr * mh / (np.sqrt(vh) + eps), m1, v1


def _mut_eps_inside(p, g, m, v, *, lr, beta1, beta2, eps, wd, step):
    m1 = beta1 * m + (1 - beta1) * g
    v1 = beta2 * v + (1 - beta2) * g * g
    mh, vh = m1 / (1 - beta1 ** step), v1 / (1 - beta2 ** step)
    return p * (1 - lr * wd) - lr * mh / np.sqrt(vh + eps), m1, v1


def _pins_hold():
    try:
        return (check_closed_form() < 1e-13 and check_special_cases() < 1e-15 and check_against_torch() < 1e-14)
    except Exception:
        return False


@pytest.mark.parametrize("mutant", [_mut_no_bias_correction, _mut_coupled_decay, _mut_eps_inside])
def test_planted_mistake_is_caught(monkeypatch, mutant):
    assert _pins_hold()
    monkeypatch.setattr(ad, "adamw_math", mutant)
    assert not _pins_hold()
