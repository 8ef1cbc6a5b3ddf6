"""Pins for the fp64 oracle: each test checks it against something other than itself.

Sources: the pages' printed worked examples (tests/golden), closed forms (the SVD form
of the Newton-Schulz iteration, AdamW's first step and constant-gradient form),
library routines (torch.optim.AdamW / Adam in float64, torch's bfloat16 conversion),
invariants (transpose symmetry, orthogonal equivariance, scale invariance), brute force
(shape bucketing) and the alternation theorem (Polar Express minimax steps).
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import adamw as oadamw
from oracle import buckets as obuckets
from oracle import muon as omuon
from oracle import polar_express as ope
from oracle.bf16 import round_bf16
from tests.conftest import read_golden
import workloads

CLASSIC5 = [omuon.CLASSIC] * 5
PE8 = ope.polar_express_table(8)


def _orth(n, k, rng):
    q, r = np.linalg.qr(rng.standard_normal((n, k)))
    return q * np.sign(np.diag(r))


# ------------------------------------------------------------------------------------------------ Newton-Schulz

@pytest.mark.parametrize("shape", [(8, 16), (16, 8), (12, 12), (5, 9), (33, 7)])
@pytest.mark.parametrize("coeffs", [CLASSIC5, PE8, [omuon.CLASSIC] * 1], ids=["classic5", "pe8", "classic1"])
def test_ns_equals_svd_closed_form(shape, coeffs):
    rng = np.random.default_rng(sum(shape))
    G = rng.standard_normal(shape)
    got = omuon.newton_schulz(G, coeffs)
    ref = omuon.ns_closed_form(G, coeffs)
    assert np.linalg.norm(got - ref) <= 1e-11 * max(1.0, np.linalg.norm(ref))


def test_ns_singular_values_in_band_of_composed_polynomial():
    rng = np.random.default_rng(1)
    G = rng.standard_normal((64, 128))
    s_in = np.linalg.svd(G, compute_uv=False) / (np.linalg.norm(G) + 1e-7)
    s_out = np.linalg.svd(omuon.newton_schulz(G, CLASSIC5), compute_uv=False)
    np.testing.assert_allclose(np.sort(s_out), np.sort(np.abs(omuon.compose_phi(s_in, CLASSIC5))), atol=1e-12)
    # band of the classic 5-step quintic over [0.0021, 1]: every output lands in [0.68, 1.2024]
    xs = np.linspace(0.0021, 1.0, 200001)
    phi = omuon.compose_phi(xs, CLASSIC5)
    assert phi.min() > 0.679 and phi.max() < 1.2025
    assert s_out.max() <= phi.max() + 1e-12 and s_out.min() >= 0.679


def test_page_singular_value_example(golden_dir):
    """Reproduces the printed output of the orthogonalisation example, section "Muon: orthogonalising the update"."""
    fx = read_golden(os.path.join(golden_dir, "ns_singular_value_example.txt"))
    rng = np.random.default_rng(0)
    U = _orth(256, 256, rng)
    V = _orth(1024, 256, rng)
    S = np.logspace(0, -2, 256)
    G = (U * S) @ V.T
    for steps in (1, 3, 5):
        s = np.linalg.svd(omuon.newton_schulz(G, [omuon.CLASSIC] * steps), compute_uv=False)
        lo, hi, share = fx[str(steps)]
        assert round(s.min(), 2) == lo and round(s.max(), 2) == hi
        assert round(100 * np.mean((s > 0.7) & (s < 1.2))) == share
    X = omuon.newton_schulz(G, CLASSIC5)
    assert round(100 * (S[:8] ** 2).sum() / (S ** 2).sum()) == fx["top8_energy_before"][0]
    top = np.linalg.norm(X @ V[:, :8]) ** 2 / np.linalg.norm(X) ** 2
    assert round(100 * top, 1) == fx["top8_energy_after"][0]
    assert round(float(np.sqrt(np.mean(X ** 2))), 4) == fx["rms_after"][0]
    assert round(float(np.sqrt(np.mean((X * 0.2 * math.sqrt(1024)) ** 2))), 2) == fx["rms_scaled"][0]


@pytest.mark.parametrize("m", [4, 64, 96])
def test_equal_singular_values_input(m):
    """[I_m | 0] has every normalised singular value 1/sqrt(m): the output is phi(1/sqrt(m)) [I_m | 0]."""
    G = np.hstack([np.eye(m), np.zeros((m, m))])
    out = omuon.newton_schulz(G, CLASSIC5, eps=0.0)
    expect = omuon.compose_phi(1.0 / math.sqrt(m), CLASSIC5) * G
    np.testing.assert_allclose(out, expect, atol=1e-12)
    # and written out by hand for one step: a s + b s^3 + c s^5 at s = 1/sqrt(m)
    s = 1.0 / math.sqrt(m)
    one = omuon.newton_schulz(G, [omuon.CLASSIC], eps=0.0)
    np.testing.assert_allclose(one[0, 0], 3.4445 * s - 4.7750 * s ** 3 + 2.0315 * s ** 5, rtol=1e-13)


@pytest.mark.parametrize("shape", [(6, 10), (10, 6)])
def test_ns_transpose_symmetry(shape):
    G = np.random.default_rng(3).standard_normal(shape)
    assert np.array_equal(omuon.newton_schulz(G.T, CLASSIC5), omuon.newton_schulz(G, CLASSIC5).T)


def test_ns_orthogonal_equivariance_and_scale_invariance():
    rng = np.random.default_rng(4)
    G = rng.standard_normal((12, 20))
    Q = _orth(12, 12, rng)
    P = _orth(20, 20, rng)
    base = omuon.newton_schulz(G, CLASSIC5, eps=0.0)
    np.testing.assert_allclose(omuon.newton_schulz(Q @ G, CLASSIC5, eps=0.0), Q @ base, atol=1e-12)
    np.testing.assert_allclose(omuon.newton_schulz(G @ P, CLASSIC5, eps=0.0), base @ P, atol=1e-12)
    for alpha in (1e-3, 7.0, 1e4):
        np.testing.assert_allclose(omuon.newton_schulz(alpha * G, CLASSIC5, eps=0.0), base, atol=1e-12)


def test_ns_of_row_slices_is_not_ns_of_matrix():
    """The distributed-Muon example's point: orthogonalising row blocks separately is a different result."""
    G = np.random.default_rng(5).standard_normal((16, 32))
    full = omuon.newton_schulz(G, CLASSIC5)
    parts = np.vstack([omuon.newton_schulz(G[i:i + 4], CLASSIC5) for i in range(0, 16, 4)])
    assert np.linalg.norm(parts - full) / np.linalg.norm(full) > 0.3


# ------------------------------------------------------------------------------------------------ Gram-space iteration

@pytest.mark.parametrize("shape", [(8, 16), (16, 8), (12, 12), (5, 9), (33, 7), (6, 40)])
@pytest.mark.parametrize("coeffs", [CLASSIC5, PE8, [omuon.CLASSIC] * 1], ids=["classic5", "pe8", "classic1"])
def test_gram_ns_equals_svd_closed_form(shape, coeffs):
    """The Gram-space recurrence reaches U phi(Sigma / ||G||) V^T, the SVD closed form (not newton_schulz)."""
    rng = np.random.default_rng(100 + sum(shape))
    G = rng.standard_normal(shape)
    got = omuon.newton_schulz_gram(G, coeffs)
    ref = omuon.ns_closed_form(G, coeffs)
    assert np.linalg.norm(got - ref) <= 1e-10 * max(1.0, np.linalg.norm(ref))


def test_gram_ns_page_singular_value_example(golden_dir):
    """The printed orthogonalisation example ("Muon: orthogonalising the update") through the Gram-space
    recurrence: the same singular-value ranges and shares after 1, 3 and 5 steps."""
    fx = read_golden(os.path.join(golden_dir, "ns_singular_value_example.txt"))
    rng = np.random.default_rng(0)
    U = _orth(256, 256, rng)
    V = _orth(1024, 256, rng)
    G = (U * np.logspace(0, -2, 256)) @ V.T
    for steps in (1, 3, 5):
        s = np.linalg.svd(omuon.newton_schulz_gram(G, [omuon.CLASSIC] * steps), compute_uv=False)
        lo, hi, share = fx[str(steps)]
        assert round(s.min(), 2) == lo and round(s.max(), 2) == hi
        assert round(100 * np.mean((s > 0.7) & (s < 1.2))) == share


@pytest.mark.parametrize("m", [4, 64])
def test_gram_ns_equal_singular_values_input(m):
    G = np.hstack([np.eye(m), np.zeros((m, 3 * m))])
    out = omuon.newton_schulz_gram(G, PE8, eps=0.0)
    np.testing.assert_allclose(out, omuon.compose_phi(1.0 / math.sqrt(m), PE8) * G, atol=1e-12)


@pytest.mark.parametrize("shape", [(6, 30), (30, 6)])
def test_gram_ns_transpose_symmetry(shape):
    G = np.random.default_rng(7).standard_normal(shape)
    assert np.array_equal(omuon.newton_schulz_gram(G.T, CLASSIC5), omuon.newton_schulz_gram(G, CLASSIC5).T)


# ------------------------------------------------------------------------------------------------ Muon step

HP = dict(lr=0.02, momentum=0.95, weight_decay=0.01)


def test_zero_gradient_only_decays():
    p = np.random.default_rng(6).standard_normal((8, 12))
    z = np.zeros_like(p)
    p_new, m_new, u = omuon.muon_update(p, z, z, **HP)
    np.testing.assert_array_equal(u, 0.0)
    np.testing.assert_array_equal(m_new, 0.0)
    np.testing.assert_allclose(p_new, p * (1 - 0.02 * 0.01), rtol=1e-15, atol=0)


@pytest.mark.parametrize("nesterov", [True, False])
def test_first_step_update_is_ns_of_gradient(nesterov):
    rng = np.random.default_rng(7)
    p = rng.standard_normal((16, 24))
    g = rng.standard_normal((16, 24))
    for mu in (0.0, 0.5, 0.95):
        p_new, m_new, u = omuon.muon_update(p, g, np.zeros_like(p), lr=0.02, momentum=mu, weight_decay=0.0,
                                            nesterov=nesterov, eps=0.0)
        np.testing.assert_array_equal(m_new, g)
        np.testing.assert_allclose(u, omuon.ns_closed_form(g, CLASSIC5, eps=0.0), atol=1e-10)
        np.testing.assert_allclose(p_new, p - 0.02 * 0.2 * math.sqrt(24) * u, atol=1e-14)


def test_momentum_and_nesterov_second_step():
    """Step 2 by hand: M2 = mu*G1 + G2; the orthogonalised input is G2 + mu*M2 (or M2 without Nesterov)."""
    rng = np.random.default_rng(8)
    p = rng.standard_normal((8, 8))
    g1, g2 = rng.standard_normal((2, 8, 8))
    mu = 0.9
    _, m1, _ = omuon.muon_update(p, g1, np.zeros_like(p), lr=0.0, momentum=mu, weight_decay=0.0, eps=0.0)
    _, m2, u2 = omuon.muon_update(p, g2, m1, lr=0.0, momentum=mu, weight_decay=0.0, eps=0.0)
    np.testing.assert_allclose(m2, mu * g1 + g2, atol=1e-15)
    np.testing.assert_allclose(u2, omuon.ns_closed_form(g2 + mu * (mu * g1 + g2), CLASSIC5, eps=0.0), atol=1e-10)
    _, _, u2n = omuon.muon_update(p, g2, m1, lr=0.0, momentum=mu, weight_decay=0.0, nesterov=False,
                                 eps=0.0)
    np.testing.assert_allclose(u2n, omuon.ns_closed_form(mu * g1 + g2, CLASSIC5, eps=0.0), atol=1e-10)


def test_cautious_decay_hand_case():
    """G = I (2x2): u = phi(1/sqrt 2) I > 0 on the diagonal. p = diag(1, -1) plus zeros: only p[0,0] shares u's sign."""
    p = np.array([[1.0, 0.0], [0.0, -1.0]])
    g = np.eye(2)
    lr, wd = 0.1, 0.5
    s = omuon.compose_phi(1 / math.sqrt(2), CLASSIC5)
    scale = 0.2 * math.sqrt(2)
    p_new, _, u = omuon.muon_update(p, g, np.zeros((2, 2)), lr=lr, momentum=0.0, weight_decay=wd,
                                    cautious_wd=True, eps=0.0)
    expect = np.array([[1.0 - lr * wd - lr * scale * s, 0.0], [0.0, -1.0 - lr * scale * s]])
    np.testing.assert_allclose(p_new, expect, atol=1e-14)
    p_plain, _, _ = omuon.muon_update(p, g, np.zeros((2, 2)), lr=lr, momentum=0.0, weight_decay=wd, eps=0.0)
    np.testing.assert_allclose(p_plain[1, 1], -1.0 * (1 - lr * wd) - lr * scale * s, atol=1e-14)


def test_update_rms_is_near_point_two():
    """After scaling by 0.2 sqrt(max(A,B)) the update's RMS is about 0.2 (section "Muon: orthogonalising the update")."""
    G = np.random.default_rng(9).standard_normal((192, 576))
    u = omuon.newton_schulz(G, CLASSIC5)
    rms = np.sqrt(np.mean((omuon.update_scale(192, 576) * u) ** 2))
    assert 0.14 < rms < 0.22


def test_scale_modes():
    assert omuon.update_scale(768, 3072) == pytest.approx(0.2 * math.sqrt(3072))
    assert omuon.update_scale(3072, 768) == pytest.approx(0.2 * math.sqrt(3072))
    assert omuon.update_scale(3072, 768, 1) == pytest.approx(2.0)
    assert omuon.update_scale(768, 3072, 1) == 1.0


# ------------------------------------------------------------------------------------------------ AdamW

def test_page_adamw_decay_example(golden_dir):
    """Reproduces the printed output of the decoupled-decay example, section "AdamW: decoupled weight decay"."""
    fx = read_golden(os.path.join(golden_dir, "adamw_decay_example.txt"))
    lr, wd, steps = 1e-2, 0.1, 1000
    scale = np.array([0.01, 10.0])
    hp = dict(lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=wd)
    for name, fn in (("adamw", oadamw.adamw_update), ("adam_l2", oadamw.adam_l2_update)):
        w, m, v = np.ones(2), np.zeros(2), np.zeros(2)
        for t in range(steps):
            w, m, v = fn(w, scale * (-1) ** t, m, v, t + 1, **hp)
        assert [round(x, 3) for x in w] == fx[name]
    assert round((1 - lr * wd) ** steps, 3) == fx["theory"][0]


@pytest.mark.parametrize("which", ["adamw", "adam_l2"])
def test_adamw_matches_torch_optim_fp64(which):
    rng = np.random.default_rng(10)
    p0 = rng.standard_normal(257)
    hp = dict(lr=3e-3, beta1=0.8, beta2=0.95, eps=1e-6, weight_decay=0.3)
    w = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    cls = torch.optim.AdamW if which == "adamw" else torch.optim.Adam
    opt = cls([w], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"], weight_decay=hp["weight_decay"],
              foreach=False)
    fn = oadamw.adamw_update if which == "adamw" else oadamw.adam_l2_update
    p, m, v = p0.copy(), np.zeros(257), np.zeros(257)
    for t in range(1, 8):
        g = rng.standard_normal(257) * 10 ** rng.uniform(-3, 1)
        w.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = fn(p, g, m, v, t, **hp)
        np.testing.assert_allclose(p, w.detach().numpy(), rtol=1e-13, atol=1e-14)
        st = opt.state[w]
        for ours, theirs in ((m, st["exp_avg"].numpy()), (v, st["exp_avg_sq"].numpy())):
            np.testing.assert_allclose(ours, theirs, rtol=1e-13, atol=1e-13 * np.abs(theirs).max())


def test_adamw_first_step_closed_form():
    rng = np.random.default_rng(11)
    p, g = rng.standard_normal((2, 100))
    lr, wd, eps = 1e-3, 0.1, 1e-8
    p1, _, _ = oadamw.adamw_update(p, g, 0 * p, 0 * p, 1, lr=lr, beta1=0.9, beta2=0.95, eps=eps, weight_decay=wd)
    np.testing.assert_allclose(p1, p * (1 - lr * wd) - lr * g / (np.abs(g) + eps), rtol=1e-14)
    assert np.all(np.abs(p1 - p * (1 - lr * wd)) <= lr * (1 + 1e-12))


def test_adamw_constant_gradient_bias_correction():
    rng = np.random.default_rng(12)
    p, g = rng.standard_normal((2, 50))
    lr, eps = 1e-3, 0.0
    m = v = np.zeros(50)
    for t in range(1, 20):
        expect = p * (1 - lr * 0.05) - lr * np.sign(g)
        p, m, v = oadamw.adamw_update(p, g, m, v, t, lr=lr, beta1=0.9, beta2=0.99, eps=eps, weight_decay=0.05)
        np.testing.assert_allclose(p, expect, rtol=1e-12)
        np.testing.assert_allclose(m / (1 - 0.9 ** t), g, rtol=1e-12)
        np.testing.assert_allclose(v / (1 - 0.99 ** t), g * g, rtol=1e-12)


# ------------------------------------------------------------------------------------------------ bf16 rounding

def test_round_bf16_matches_torch_on_float32_values():
    rng = np.random.default_rng(13)
    x32 = (rng.standard_normal(200000) * 10.0 ** rng.uniform(-40, 38, 200000)).astype(np.float32)
    got = round_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_ties_and_limits():
    one = 1.0
    assert round_bf16(one + 2.0 ** -8) == 1.0                           # tie, even stays
    assert round_bf16(one + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6           # tie, odd rounds up
    assert round_bf16(one + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7  # just above the tie (no double rounding)
    assert round_bf16(-(one + 2.0 ** -8 + 2.0 ** -40)) == -(1.0 + 2.0 ** -7)
    top = (2 - 2 ** -7) * 2.0 ** 127
    half_ulp = 2.0 ** 119
    assert round_bf16(top + 0.9 * half_ulp) == top and np.isinf(round_bf16(top + 1.1 * half_ulp))
    assert round_bf16(2.0 ** -133) == 2.0 ** -133 and round_bf16(2.0 ** -135) == 0.0
    assert round_bf16(0.0) == 0.0 and np.isnan(round_bf16(np.nan))


# ------------------------------------------------------------------------------------------------ bucketing

def _brute_force_plan(shapes):
    n = len(shapes)
    first = {}
    for i, s in enumerate(shapes):
        first.setdefault(tuple(s), i)
    keys = sorted(first, key=lambda k: first[k])
    bid = [keys.index(tuple(s)) for s in shapes]
    idx = [sum(1 for j in range(i) if tuple(shapes[j]) == tuple(shapes[i])) for i in range(n)]
    K = [sum(1 for s in shapes if tuple(s) == k) for k in keys]
    off = [sum(K[c] * keys[c][0] * keys[c][1] for c in range(b)) for b in range(len(keys))]
    return bid, idx, keys, K, off


def test_bucket_plan_brute_force():
    rng = np.random.default_rng(14)
    for trial in range(200):
        n = int(rng.integers(0, 12))
        shapes = [tuple(int(v) for v in rng.integers(1, 4, 2)) for _ in range(n)]
        plan = obuckets.plan_buckets(shapes)
        bid, idx, keys, K, off = _brute_force_plan(shapes)
        assert plan["bucket_id"] == bid and plan["index_in_bucket"] == idx
        assert plan["bucket_shapes"] == keys and plan["bucket_K"] == K and plan["momentum_offset"] == off


def test_bucket_plan_model_sets():
    g = obuckets.plan_buckets(workloads.shape_list(workloads.workload("gpt2s")))
    assert g["bucket_shapes"] == [(768, 2304), (768, 768), (768, 3072), (3072, 768)]
    assert g["bucket_K"] == [12, 12, 12, 12]
    ll = obuckets.plan_buckets(workloads.shape_list(workloads.workload("llama8b")))
    assert ll["bucket_shapes"] == [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)]
    assert ll["bucket_K"] == [64, 64, 64, 32]
    assert ll["total_momentum"] == 6_979_321_856


# ------------------------------------------------------------------------------------------------ Polar Express

@pytest.mark.parametrize("interval", [(1e-3, 1.0), (0.05, 1.0), (0.3, 1.7), (0.9, 1.1)])
def test_minimax_step_equioscillates(interval):
    """Alternation theorem: equal-magnitude, alternating-sign error on 4 points and no larger error anywhere."""
    lo, hi = interval
    (a, b, c), E, pts = ope.minimax_odd_quintic(lo, hi)
    err = lambda x: 1 - (a * x + b * x ** 3 + c * x ** 5)
    e = err(pts)
    np.testing.assert_allclose(np.abs(e), E, rtol=1e-9)
    assert np.all(np.sign(e[:-1]) != np.sign(e[1:]))
    xs = np.linspace(lo, hi, 400001)
    assert np.max(np.abs(err(xs))) <= E * (1 + 1e-9)


def test_minimax_beats_perturbations():
    (a, b, c), E, _ = ope.minimax_odd_quintic(0.05, 1.0)
    xs = np.linspace(0.05, 1.0, 20001)
    rng = np.random.default_rng(15)
    for _ in range(200):
        d = rng.standard_normal(3) * 1e-3
        p = (a + d[0]) * xs + (b + d[1]) * xs ** 3 + (c + d[2]) * xs ** 5
        assert np.max(np.abs(1 - p)) >= E * (1 - 1e-9)


def test_polar_express_table_band_and_stored_copy(golden_dir):
    import json
    table = ope.polar_express_table(8)
    with open(os.path.join(golden_dir, "polar_express_8step.json")) as f:
        stored = json.load(f)["coeffs"]
    np.testing.assert_allclose(np.array(stored), np.array(table), rtol=0, atol=0)
    xs = np.linspace(1e-3, 1.0, 100001)
    phi = omuon.compose_phi(xs, table)
    assert np.max(np.abs(phi - 1)) < 1e-5
    # a Frobenius-normalised Gaussian 64 x 1024 matrix has sigma_min/||G||_F well above 1e-3
    G = np.random.default_rng(16).standard_normal((64, 1024))
    s = np.linalg.svd(omuon.newton_schulz(G, table), compute_uv=False)
    assert np.max(np.abs(s - 1)) < 1e-5


def test_polar_express_safety_margin():
    """A 1% overshoot of the normalised input stays bounded; without the margin the same table explodes."""
    xs = np.linspace(0.0, 1.01, 200001)
    safe = omuon.compose_phi(xs, ope.polar_express_table(8))
    assert np.all(np.abs(safe) < 1.01)
    with np.errstate(over="ignore", invalid="ignore"):
        unsafe = omuon.compose_phi(xs, ope.polar_express_table(8, safety=1.0))
    assert not np.all(np.abs(unsafe) < 10.0)
    # every intermediate stays inside the interval the next step was designed for
    table = ope.polar_express_table(8)
    s = xs.copy()
    lo, hi = 1e-3, 1.0
    for a, b, c in table:
        (_, _, _), E, _ = ope.minimax_odd_quintic(lo, hi)
        s = a * s + b * s ** 3 + c * s ** 5
        lo, hi = a * lo + b * lo ** 3 + c * lo ** 5, 1.0 + E
        assert s.max() <= hi * (1 + 1e-9)
