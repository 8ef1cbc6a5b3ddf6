"""Planted mistakes: each plausible error in the oracle must fail at least one pin.

The mutation is planted in the oracle (on the CPU) by monkeypatching one function; the listed pins
are then run and at least one must fail. This checks that the pins constrain the oracle, not that
the oracle is right (the pins do that).
"""
import numpy as np
import pytest

from oracle import adamw as oadamw
from oracle import muon as omuon
from tests import test_oracle_pins as pins


def _ns_drop_c(G, coeffs, eps=1e-7):
    G = np.asarray(G, dtype=np.float64)
    X = G / (np.linalg.norm(G) + eps)
    t = G.shape[0] > G.shape[1]
    if t:
        X = X.T
    for a, b, c in coeffs:
        A = X @ X.T
        X = a * X + (b * A) @ X
    return X.T if t else X


def _ns_spectral_norm(G, coeffs, eps=1e-7):
    G = np.asarray(G, dtype=np.float64)
    X = G / (np.linalg.norm(G, 2) + eps)
    t = G.shape[0] > G.shape[1]
    if t:
        X = X.T
    for a, b, c in coeffs:
        A = X @ X.T
        X = a * X + (b * A + c * A @ A) @ X
    return X.T if t else X


def _ns_wrong_sign(G, coeffs, eps=1e-7):
    return _ns_ref(G, [(a, -b, c) for a, b, c in coeffs], eps)


_ns_ref = omuon.newton_schulz


def _gram_parts(G, eps):
    G = np.asarray(G, dtype=np.float64)
    X0 = G / (np.linalg.norm(G) + eps)
    t = G.shape[0] > G.shape[1]
    return (X0.T if t else X0), t


def _gram_one_sided_update(G, coeffs, eps=1e-7):
    X0, t = _gram_parts(G, eps)
    I = np.eye(X0.shape[0])
    A, R = X0 @ X0.T, I
    for a, b, c in coeffs:
        Q = a * I + b * A + c * A @ A
        R = Q @ R
        A = Q @ A                      # planted: A_{t+1} = Q A instead of Q A Q
    X = R @ X0
    return X.T if t else X


def _gram_last_q_only(G, coeffs, eps=1e-7):
    X0, t = _gram_parts(G, eps)
    I = np.eye(X0.shape[0])
    A, R = X0 @ X0.T, I
    for a, b, c in coeffs:
        Q = a * I + b * A + c * A @ A
        R = Q                          # planted: R not accumulated
        A = Q @ A @ Q
    X = R @ X0
    return X.T if t else X


def _gram_drop_c(G, coeffs, eps=1e-7):
    X0, t = _gram_parts(G, eps)
    I = np.eye(X0.shape[0])
    A, R = X0 @ X0.T, I
    for a, b, c in coeffs:
        Q = a * I + b * A              # planted: no c A^2 term
        R = Q @ R
        A = Q @ A @ Q
    X = R @ X0
    return X.T if t else X


def _muon_decay_after(p, g, m, *, lr, momentum, weight_decay, nesterov=True, cautious_wd=False,
                      coeffs=(omuon.CLASSIC,) * 5, eps=1e-7, scale_mode=0, param_dtype="f64"):
    p = np.asarray(p, float)
    m_new = momentum * np.asarray(m, float) + g
    u = omuon.newton_schulz(g + momentum * m_new if nesterov else m_new, coeffs, eps)
    p_new = p - lr * omuon.update_scale(*p.shape, scale_mode) * u
    mask = (u * p > 0) if cautious_wd else 1.0
    return p_new - lr * weight_decay * p_new * mask, m_new, u


def _muon_old_momentum_nesterov(p, g, m, *, lr, momentum, weight_decay, nesterov=True, cautious_wd=False,
                                coeffs=(omuon.CLASSIC,) * 5, eps=1e-7, scale_mode=0, param_dtype="f64"):
    p = np.asarray(p, float)
    m = np.asarray(m, float)
    m_new = momentum * m + g
    u = omuon.newton_schulz(g + momentum * m if nesterov else m_new, coeffs, eps)
    mask = (u * p > 0) if cautious_wd else 1.0
    return p - lr * weight_decay * p * mask - lr * omuon.update_scale(*p.shape, scale_mode) * u, m_new, u


def _muon_min_scale(p, g, m, **kw):
    saved = omuon.update_scale
    try:
        omuon.update_scale = lambda A, B, mode=0: 0.2 * np.sqrt(min(A, B))
        return _muon_ref(p, g, m, **kw)
    finally:
        omuon.update_scale = saved


_muon_ref = omuon.muon_update


def _adamw_no_bias_correction(p, g, m, v, t, *, lr, beta1, beta2, eps, weight_decay, param_dtype="f64"):
    p = np.asarray(p, float) * (1 - lr * weight_decay)
    m = beta1 * np.asarray(m, float) + (1 - beta1) * g
    v = beta2 * np.asarray(v, float) + (1 - beta2) * np.asarray(g) ** 2
    return p - lr * m / (np.sqrt(v) + eps), m, v


def _adamw_eps_inside(p, g, m, v, t, *, lr, beta1, beta2, eps, weight_decay, param_dtype="f64"):
    p = np.asarray(p, float) * (1 - lr * weight_decay)
    m = beta1 * np.asarray(m, float) + (1 - beta1) * g
    v = beta2 * np.asarray(v, float) + (1 - beta2) * np.asarray(g) ** 2
    return p - lr * (m / (1 - beta1 ** t)) / np.sqrt(v / (1 - beta2 ** t) + eps), m, v


NS_PINS = [
    lambda: pins.test_ns_equals_svd_closed_form((8, 16), pins.CLASSIC5),
    lambda: pins.test_page_singular_value_example(pins.os.path.join(pins.os.path.dirname(pins.__file__), "golden")),
    lambda: pins.test_equal_singular_values_input(64),
]
GRAM_PINS = [
    lambda: pins.test_gram_ns_equals_svd_closed_form((8, 16), pins.CLASSIC5),
    lambda: pins.test_gram_ns_page_singular_value_example(pins.os.path.join(pins.os.path.dirname(pins.__file__),
                                                                            "golden")),
    lambda: pins.test_gram_ns_equal_singular_values_input(64),
]
MUON_PINS = [pins.test_cautious_decay_hand_case, pins.test_momentum_and_nesterov_second_step,
             lambda: pins.test_first_step_update_is_ns_of_gradient(True), pins.test_zero_gradient_only_decays]
ADAMW_PINS = [lambda: pins.test_page_adamw_decay_example(pins.os.path.join(pins.os.path.dirname(pins.__file__),
                                                                           "golden")),
              lambda: pins.test_adamw_matches_torch_optim_fp64("adamw"), pins.test_adamw_first_step_closed_form]


def _some_pin_fails(pin_list):
    for pin in pin_list:
        try:
            pin()
        except AssertionError:
            return True
    return False


@pytest.mark.parametrize("mutant", [_ns_drop_c, _ns_spectral_norm, _ns_wrong_sign])
def test_ns_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(omuon, "newton_schulz", mutant)
    assert _some_pin_fails(NS_PINS)


@pytest.mark.parametrize("mutant", [_gram_one_sided_update, _gram_last_q_only, _gram_drop_c])
def test_gram_ns_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(omuon, "newton_schulz_gram", mutant)
    assert _some_pin_fails(GRAM_PINS)


@pytest.mark.parametrize("mutant", [_muon_decay_after, _muon_old_momentum_nesterov, _muon_min_scale])
def test_muon_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(omuon, "muon_update", mutant)
    assert _some_pin_fails(MUON_PINS)


@pytest.mark.parametrize("mutant", [_adamw_no_bias_correction, _adamw_eps_inside])
def test_adamw_mutants_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(oadamw, "adamw_update", mutant)
    assert _some_pin_fails(ADAMW_PINS)


def test_unmutated_oracle_passes_the_same_pins():
    assert not _some_pin_fails(NS_PINS + GRAM_PINS + MUON_PINS + ADAMW_PINS)
