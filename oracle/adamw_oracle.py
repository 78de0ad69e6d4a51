"""Plain fp64 CPU oracle of the AdamW step for the parameters that stay off
Muon (embeddings, biases, norms).

TEST INFRASTRUCTURE ONLY.  Only ``tests/`` and the CPU-baseline and reference
legs of ``bench.py`` may import this module; the library never calls it and
shares no code with it.  Pinned by ``tests/test_adamw_oracle_pins.py``.

Source: "MuonX: DMuon 调整多卡分工, Gram NS 降低计算量" (CSDN), section 2 — the
hidden 2-D weight matrices are updated by Muon while embeddings and biases stay
on AdamW.  The pages do not print AdamW; the standard decoupled-weight-decay
Adam step is used:
    m' = b1 m + (1 - b1) g,   v' = b2 v + (1 - b2) g^2
    m_hat = m' / (1 - b1^t),  v_hat = v' / (1 - b2^t)
    p' = p (1 - lr wd) - lr m_hat / (sqrt(v_hat) + eps)
with t the 1-based step count, decay and update both on the old p.
"""
from __future__ import annotations

import math

import numpy as np

from oracle.muon_oracle import round_to, to_f64


def adamw_math(p, g, m, v, *, lr, beta1, beta2, eps, wd, step):
    """The step in fp64 on fp64 arrays; returns (p', m', v')."""
    m1 = beta1 * m + (1.0 - beta1) * g
    v1 = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m1 / (1.0 - beta1 ** step)
    v_hat = v1 / (1.0 - beta2 ** step)
    p1 = p * (1.0 - lr * wd) - lr * m_hat / (np.sqrt(v_hat) + eps)
    return p1, m1, v1


def adamw_step(p, g, m, v, *, lr, beta1, beta2, eps, wd, step, param_dtype, state_dtype):
    """From stored arrays (fp32, or bf16 as uint16 bits) to exact and stored results."""
    p64, g64 = to_f64(p, param_dtype), to_f64(g, param_dtype)
    m64, v64 = to_f64(m, state_dtype), to_f64(v, state_dtype)
    p1, m1, v1 = adamw_math(p64, g64, m64, v64, lr=lr, beta1=beta1, beta2=beta2, eps=eps, wd=wd, step=step)
    return {"p_exact": p1, "m_exact": m1, "v_exact": v1, "p_old": p64,
            "p_new": round_to(p1, param_dtype), "m_new": round_to(m1, state_dtype),
            "v_new": round_to(v1, state_dtype)}


def constant_gradient_closed_form(p0, g, *, lr, eps, step):
    """From zero moments with a constant gradient g and wd = 0, bias correction
    makes m_hat = g and v_hat = g^2 at every step, so each step moves p by
    -lr g / (|g| + eps)."""
    return p0 - step * lr * g / (np.abs(g) + eps)


__all__ = ["adamw_math", "adamw_step", "constant_gradient_closed_form", "math"]
