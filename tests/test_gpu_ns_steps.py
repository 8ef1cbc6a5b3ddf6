"""GPU parity of the three tensor-core steps of one Newton-Schulz iteration, through the C ABI.

Each step is compared element by element with its definition evaluated in fp64 on the same bf16
inputs: G = alpha X X^T, H = a I + b G + c G G, out = H X (the loop body of newton_schulz in
"Optimizers: AdamW, Muon and the distributed optimizer", section "Muon: orthogonalising the update",
a X + (b G + c G G) X, with a folded into the polynomial).
Shapes span several 128 x 256 tiles, ragged edges in both dimensions, a single row, and K > 1.
"""
import numpy as np
import pytest
import torch

from tests.gpu_common import DEV, build_lib, ctrl_ws, f64

pytestmark = pytest.mark.gpu

SHAPES = [(2, 64, 128), (3, 136, 264), (2, 384, 1536), (1, 1024, 4096), (2, 520, 776), (1, 8, 8), (4, 256, 2048)]


@pytest.fixture(scope="module")
def L():
    return build_lib()


def _x(K, m, n, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((K, m, n), generator=g, dtype=torch.float64) / np.sqrt(n)
    return x.to(torch.bfloat16).to(DEV)


def _check(got, ref, tol):
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} elements out of tolerance; worst excess {np.max(np.abs(got - ref) - tol):.3e}"


@pytest.mark.parametrize("K,m,n", SHAPES)
def test_gram(L, K, m, n):
    x = _x(K, m, n, 1 + m + n)
    g = torch.full((K, m, m), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = ctrl_ws()
    alpha = 1.25
    L.ns_gram(x, g, alpha, ws)
    assert L.muon_check(ws) == L.MUON_OK
    X = f64(x)
    got = f64(g)
    ref = alpha * X @ X.transpose(0, 2, 1)
    S = alpha * np.abs(X) @ np.abs(X).transpose(0, 2, 1)
    _check(got, ref, 2.0 ** -8 * np.abs(ref) + 1e-5 * S)
    # symmetric by construction: each value is computed once and stored twice
    assert np.array_equal(got, got.transpose(0, 2, 1))


@pytest.mark.parametrize("K,m,n", SHAPES)
def test_poly(L, K, m, n):
    x = _x(K, m, n, 7 + m)
    X = f64(x)
    G = X @ X.transpose(0, 2, 1)
    G = (G + G.transpose(0, 2, 1)) / 2
    g = torch.from_numpy(G).to(torch.bfloat16).to(DEV)
    Gb = f64(g)
    h = torch.full((K, m, m), float("nan"), dtype=torch.bfloat16, device=DEV)
    a, b, c = 3.4445, -4.7750, 2.0315
    ws = ctrl_ws()
    L.ns_poly(g, h, a, b, c, ws)
    assert L.muon_check(ws) == L.MUON_OK
    got = f64(h)
    GG = Gb @ Gb
    eye = np.eye(m)[None]
    ref = a * eye + b * Gb + c * GG
    terms = a * eye + abs(b) * np.abs(Gb) + abs(c) * np.abs(GG)
    _check(got, ref, 2.0 ** -8 * terms + abs(c) * 1e-5 * (np.abs(Gb) @ np.abs(Gb)) + 2.0 ** -8 * np.abs(ref))
    assert np.array_equal(got, got.transpose(0, 2, 1))


@pytest.mark.parametrize("K,m,n", SHAPES)
def test_apply(L, K, m, n):
    x = _x(K, m, n, 11 + n)
    X = f64(x)
    gen = torch.Generator().manual_seed(5 + m)
    H = torch.randn((K, m, m), generator=gen, dtype=torch.float64) / np.sqrt(m)
    H = (H + H.transpose(1, 2)) / 2 + 3.4445 * torch.eye(m, dtype=torch.float64)   # a*I + symmetric, as ns_poly makes
    h = H.to(torch.bfloat16).to(DEV)
    Hb = f64(h)
    out = torch.full((K, m, n), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = ctrl_ws()
    L.ns_apply(h, x, out, ws)
    assert L.muon_check(ws) == L.MUON_OK
    got = f64(out)
    ref = Hb @ X
    _check(got, ref, 1e-5 * (np.abs(Hb) @ np.abs(X)) + 2.0 ** -8 * np.abs(ref))


def test_bounded_wait_reports_timeout_and_context_survives(L):
    ws = ctrl_ws()
    L.muon_debug_wait_timeout(ws, 50_000_000)   # 50 ms on a barrier nothing completes
    assert L.muon_check(ws) == L.MUON_ERR_TIMEOUT
    assert L.muon_check(ws) == L.MUON_OK        # the word was cleared
    x = _x(1, 64, 128, 3)
    g = torch.zeros((1, 64, 64), dtype=torch.bfloat16, device=DEV)
    L.ns_gram(x, g, 1.0, ws)
    assert L.muon_check(ws) == L.MUON_OK
    X = f64(x)
    assert np.allclose(f64(g), X @ X.transpose(0, 2, 1), rtol=1e-2, atol=1e-3)


def test_launch_count_and_trace(L):
    x = _x(2, 64, 128, 4)
    g = torch.zeros((2, 64, 64), dtype=torch.bfloat16, device=DEV)
    ws = ctrl_ws()
    before = L.muon_launch_count()
    L.muon_trace_enable(True)
    L.ns_gram(x, g, 1.0, ws)
    L.ns_gram(x, g, 1.0, ws)
    L.muon_trace_enable(False)
    rec = L.muon_trace_collect()
    assert L.muon_launch_count() - before == 2
    assert [k for k, _ in rec] == ["ns_gram", "ns_gram"] and all(ms > 0 for _, ms in rec)
