"""Muon update, fp64, one matrix at a time.

Follows [P2] "Optimizers: AdamW, Muon and the distributed optimizer", section
"Muon: orthogonalising the update" (the three-step update rule and the newton_schulz /
Muon.step example), with the options of [P3] "dtensor-muon 0.1.0", table "Key options"
(nesterov, use_cautious_wd, ns_steps, orthogonalization_strategy).

Readings where the pages are silent (the same readings the GPU path takes):
  * Nesterov input is the sum G + mu*M with the *updated* M; nesterov=False uses M.
  * eps = 1e-7 is added to the Frobenius norm of that one matrix.
  * Transposition happens only when rows > cols (squares are not transposed).
  * Weight decay uses the pre-update parameter and is multiplied by lr; it is applied
    before the orthogonalised update ([P2] Muon.step decays, then adds).
  * Cautious decay (u * p > 0, [P3] "Features" and "Key options") masks the decay only,
    with u the orthogonalised update and p the pre-update parameter; ties do not decay.
  * The per-step coefficient triple (a_t, b_t, c_t) is a parameter: the classic
    (3.4445, -4.7750, 2.0315) repeated, or a per-step Polar Express table.
"""
from __future__ import annotations

import math
from typing import Sequence, Tuple

import numpy as np

from .bf16 import round_to

Coeffs = Sequence[Tuple[float, float, float]]

CLASSIC = (3.4445, -4.7750, 2.0315)


def newton_schulz(G, coeffs: Coeffs, eps: float = 1e-7) -> np.ndarray:
    """[P2] "Muon: orthogonalising the update", newton_schulz: approximate the polar factor U V^T.

    X = G / (||G||_F + eps); work on X^T when G has more rows than columns, so that the
    Gram matrix X X^T is the smaller square; per step t:
        A = X X^T ;  X <- a_t X + (b_t A + c_t A A) X
    and transpose back at the end.
    """
    G = np.asarray(G, dtype=np.float64)
    X = G / (np.linalg.norm(G) + eps)          # Frobenius norm of the whole matrix
    transposed = G.shape[0] > G.shape[1]
    if transposed:
        X = X.T
    for a, b, c in coeffs:
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if transposed else X


def newton_schulz_gram(G, coeffs: Coeffs, eps: float = 1e-7) -> np.ndarray:
    """[P4] "DMuon", section 2.2 "Efficient Gram Newton-Schulz Iteration": the same iteration run in the
    m x m Gram space (m = the smaller side), which costs O(m^3) per step instead of O(m^2 n).

    The page names the recurrence but prints no formula. Reading taken (the plainest one that reaches the
    same X_N as newton_schulz): with X_0 the normalised wide matrix and A_0 = X_0 X_0^T, every iterate is
    X_t = R_t X_0 for an m x m matrix R_t, and X_t X_t^T = A_t; per step t
        Q_t = a_t I + b_t A_t + c_t A_t A_t ;  R_{t+1} = Q_t R_t ;  A_{t+1} = Q_t A_t Q_t
    (X_{t+1} = Q_t X_t is newton_schulz's step), and the output is X_N = R_N X_0, transposed back.
    """
    G = np.asarray(G, dtype=np.float64)
    X0 = G / (np.linalg.norm(G) + eps)         # Frobenius norm of the whole matrix
    transposed = G.shape[0] > G.shape[1]
    if transposed:
        X0 = X0.T
    m = X0.shape[0]
    I = np.eye(m)
    A = X0 @ X0.T
    R = I
    for a, b, c in coeffs:
        Q = a * I + b * A + c * (A @ A)
        R = Q @ R
        A = Q @ A @ Q
    X = R @ X0
    return X.T if transposed else X


def compose_phi(x, coeffs: Coeffs) -> np.ndarray:
    """The scalar map a singular value goes through: phi = p_{N-1} o ... o p_0, p_t(s) = a s + b s^3 + c s^5.

    Each Newton-Schulz step maps X = U S V^T to U p_t(S) V^T, because X X^T = U S^2 U^T,
    so the whole iteration acts on each normalised singular value separately.
    """
    s = np.asarray(x, dtype=np.float64)
    for a, b, c in coeffs:
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def ns_closed_form(G, coeffs: Coeffs, eps: float = 1e-7) -> np.ndarray:
    """U phi(Sigma / (||G||_F + eps)) V^T from an SVD: what newton_schulz computes, by another route."""
    G = np.asarray(G, dtype=np.float64)
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    return (U * compose_phi(S / (np.linalg.norm(G) + eps), coeffs)) @ Vt


def update_scale(A: int, B: int, scale_mode: int = 0) -> float:
    """0: 0.2*sqrt(max(A,B)) ([P2] Muon rule step 3); 1: sqrt(max(1, A/B)) ([P2], the alternative scaling noted
    after the orthogonalisation example)."""
    if scale_mode == 0:
        return 0.2 * math.sqrt(max(A, B))
    if scale_mode == 1:
        return math.sqrt(max(1.0, A / B))
    raise ValueError(scale_mode)


def muon_update(p, g, m, *, lr: float, momentum: float, weight_decay: float, nesterov: bool = True,
                cautious_wd: bool = False, coeffs: Coeffs = (CLASSIC,) * 5, eps: float = 1e-7,
                scale_mode: int = 0, param_dtype: str = "f64"):
    """One Muon step on one A x B matrix. Returns (p_new, m_new, u) with u the orthogonalised direction.

    [P2] Muon rule: M <- mu M + G; orthogonalise G + mu M (Nesterov) into U V^T;
    W <- W - eta * 0.2 sqrt(max(A,B)) * U V^T, with decoupled decay W <- W (1 - eta lambda) first.
    [P3] use_cautious_wd: decay only where u * p > 0. nesterov=False orthogonalises M itself.
    p_new is rounded to the parameter's storage dtype (no fp32 master copy).
    """
    p = np.asarray(p, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    A, B = p.shape
    m_new = momentum * m + g
    ns_in = g + momentum * m_new if nesterov else m_new
    u = newton_schulz(ns_in, coeffs, eps)
    if cautious_wd:
        mask = (u * p > 0).astype(np.float64)
    else:
        mask = 1.0
    decayed = p - lr * weight_decay * p * mask
    p_new = decayed - lr * update_scale(A, B, scale_mode) * u
    return round_to(p_new, param_dtype), m_new, u


def muon_trajectory(p0, grads, **hp):
    """Run muon_update over a list of gradients from zero momentum; returns the final (p, m) and per-step p."""
    p = np.asarray(p0, dtype=np.float64)
    m = np.zeros_like(p)
    history = []
    for g in grads:
        p, m, _ = muon_update(p, g, m, **hp)
        history.append(p)
    return p, m, history
