"""AdamW (and Adam + L2), fp64, elementwise.

Follows [P2] "Optimizers: AdamW, Muon and the distributed optimizer", section
"AdamW: decoupled weight decay": first and second moments m, v; update m / (sqrt(v) + eps);
AdamW applies w <- w - eta*lambda*w to the weights directly, outside the normalisation,
while Adam + L2 adds lambda*w to the gradient first.

Readings (the page prints no formula for these; its worked example reproduces only with
them, which the tests check): bias correction m_hat = m / (1 - beta1^t),
v_hat = v / (1 - beta2^t); eps added outside the square root; decay applied before the
moment update; t starts at 1; m and v start at zero.
"""
from __future__ import annotations

import numpy as np

from .bf16 import round_to


def adamw_update(p, g, m, v, t: int, *, lr: float, beta1: float, beta2: float, eps: float, weight_decay: float,
                 param_dtype: str = "f64"):
    """One AdamW step at step count t >= 1. Returns (p_new, m_new, v_new)."""
    if t < 1:
        raise ValueError("t starts at 1")
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    p = p * (1.0 - lr * weight_decay)                  # decoupled decay on the weight itself
    m_new = beta1 * m + (1.0 - beta1) * g
    v_new = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m_new / (1.0 - beta1 ** t)
    v_hat = v_new / (1.0 - beta2 ** t)
    p_new = p - lr * m_hat / (np.sqrt(v_hat) + eps)
    return round_to(p_new, param_dtype), m_new, v_new


def adam_l2_update(p, g, m, v, t: int, *, lr: float, beta1: float, beta2: float, eps: float, weight_decay: float,
                   param_dtype: str = "f64"):
    """One Adam step with L2 regularisation: lambda*w joins the gradient and is normalised with it."""
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64) + weight_decay * p
    m_new = beta1 * np.asarray(m, dtype=np.float64) + (1.0 - beta1) * g
    v_new = beta2 * np.asarray(v, dtype=np.float64) + (1.0 - beta2) * g * g
    m_hat = m_new / (1.0 - beta1 ** t)
    v_hat = v_new / (1.0 - beta2 ** t)
    p_new = p - lr * m_hat / (np.sqrt(v_hat) + eps)
    return round_to(p_new, param_dtype), m_new, v_new
