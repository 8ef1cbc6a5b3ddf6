"""GPU parity of the Gram-space Newton-Schulz path ("DMuon", section 2.2, "Efficient Gram Newton-Schulz
Iteration") against the fp64 oracle, through the C ABI.

The path takes wide iterates with m = min(A, B) <= 256 rows that the fused small-matrix kernel does not take,
by default when n = max(A, B) >= 4 m (muon_gram_space_route); muon_debug_gram_space(1) forces it onto every
such shape and (0) keeps the plain chain. Bars as for the plain chain: relative Frobenius error <= 2e-2 of
the orthogonalised output (against both the oracle's plain iteration and its Gram-space restatement, which
agree in fp64), and of the parameter change for the Muon step. Shapes cover one and two 128-row blocks per
side, ragged m, tall stacks (transposed to wide and back), stacks whose matrix count leaves part of a
cluster idle, and very small m; inputs cover Gaussian, Student-t(3) and a rank-16 spike on noise, with the
classic quintic and the 8-step Polar Express table. The fp32 Gram that starts the path is also run with its
contraction split into slices (muon_debug_gram_split), against the unsplit result and the oracle.
"""
import numpy as np
import pytest
import torch

from oracle import muon as omuon
from tests.gpu_common import DEV, build_lib, f64, hp_struct, rel_fro, workspace
import workloads

pytestmark = pytest.mark.gpu

CLASSIC5 = [omuon.CLASSIC] * 5
PE8 = list(workloads.polar_express_coeffs(8))


@pytest.fixture(scope="module")
def L():
    lib = build_lib()
    yield lib
    lib.muon_debug_gram_space(-1)
    lib.muon_debug_gram_split(-1)


def _spike(K, A, B, seed):
    """Gaussian noise plus a rank-16 component ten times its size (per singular value), bf16."""
    rng = np.random.default_rng(seed)
    out = []
    m, n = min(A, B), max(A, B)
    for _ in range(K):
        noise = rng.standard_normal((m, n))
        U = np.linalg.qr(rng.standard_normal((m, 16)))[0]
        V = np.linalg.qr(rng.standard_normal((n, 16)))[0]
        x = noise + (U * (10.0 * np.sqrt(m * n) / 16)) @ V.T
        out.append(x if A <= B else x.T)
    return torch.from_numpy(np.stack(out)).to(torch.bfloat16)


def _input(kind, K, A, B, seed):
    if kind == "spike":
        return _spike(K, A, B, seed)
    g = np.random.default_rng(seed)
    x = g.standard_t(3, size=(K, A, B)) if kind == "t3" else g.standard_normal((K, A, B))
    return torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("K,A,B,kind,odt", [
    (4, 256, 1024, "gauss", torch.float32),      # two blocks per side
    (3, 1024, 256, "t3", torch.bfloat16),        # tall
    (2, 200, 1000, "gauss", torch.float32),      # ragged m, two blocks
    (5, 64, 4096, "t3", torch.float32),          # one block: 4 matrices per cluster, the second cluster 1 of 4
    (2, 130, 600, "spike", torch.float32),
    (3, 8, 2048, "gauss", torch.float32),        # m below one 32-column slice
    (2, 256, 16384, "spike", torch.bfloat16),    # the aspect set's shape
])
@pytest.mark.parametrize("coeffs", [CLASSIC5, PE8], ids=["classic5", "pe8"])
def test_gram_space_ns_matches_oracle(L, K, A, B, kind, odt, coeffs):
    assert L.muon_gram_space_route(A, B)
    x = _input(kind, K, A, B, K + A + B).to(DEV)
    out = torch.full((K, A, B), float("nan"), dtype=odt, device=DEV)
    ws = workspace(L, K, A, B)
    L.ns_orthogonalize(x, out, coeffs, 1e-7, ws)
    assert L.muon_check(ws) == L.MUON_OK
    X, got = f64(x), f64(out)
    for k in range(K):
        ref = omuon.newton_schulz(X[k], coeffs, 1e-7)
        assert rel_fro(got[k], ref) <= 2e-2, (k, rel_fro(got[k], ref))
        ref_g = omuon.newton_schulz_gram(X[k], coeffs, 1e-7)
        assert rel_fro(got[k], ref_g) <= 2e-2


@pytest.mark.parametrize("K,A,B", [(2, 256, 256), (3, 160, 320)])
def test_gram_space_forced_on_shapes_the_rule_leaves_plain(L, K, A, B):
    """Forced onto eligible shapes with n < 4 m (square included): still the oracle's result; and the plain
    chain on the same input (forced off) agrees with the oracle too."""
    assert not L.muon_gram_space_route(A, B)
    x = _input("gauss", K, A, B, 11).to(DEV)
    outs = {}
    try:
        for mode in (1, 0):
            L.muon_debug_gram_space(mode)
            out = torch.empty((K, A, B), dtype=torch.float32, device=DEV)
            ws = workspace(L, K, A, B)
            L.ns_orthogonalize(x, out, PE8, 1e-7, ws)
            assert L.muon_check(ws) == L.MUON_OK
            outs[mode] = f64(out)
    finally:
        L.muon_debug_gram_space(-1)
    X = f64(x)
    for k in range(K):
        ref = omuon.newton_schulz(X[k], PE8, 1e-7)
        assert rel_fro(outs[1][k], ref) <= 2e-2
        assert rel_fro(outs[0][k], ref) <= 2e-2


@pytest.mark.parametrize("K,A,B", [
    (4, 256, 1024),    # 16 contraction steps of 64: slices of 8, 6 + 6 + 4, 4
    (2, 200, 1000),    # ragged m and a ragged last step
    (3, 1024, 256),    # tall
    (2, 64, 300),      # 5 steps: 4 slices of 2 + 2 + 1 ... evened out to 3 of 2, 2, 1
])
def test_gram_split_matches_unsplit_and_oracle(L, K, A, B):
    """The Gram-space path's fp32 Gram with its contraction split into 2, 3 and 4 slices (summed in slice order
    by the reduce kernel): each within the bar of the oracle, within 1e-3 of the unsplit result (only the order
    of the fp32 additions differs), and the same bits when run again."""
    assert L.muon_gram_space_route(A, B)
    x = _input("t3", K, A, B, 7 * K + A).to(DEV)
    X = f64(x)
    outs = {}
    try:
        for split in (1, 2, 3, 4, 3):
            L.muon_debug_gram_split(split)
            out = torch.full((K, A, B), float("nan"), dtype=torch.float32, device=DEV)
            ws = workspace(L, K, A, B)
            L.ns_orthogonalize(x, out, PE8, 1e-7, ws)
            assert L.muon_check(ws) == L.MUON_OK
            if split in outs:
                assert torch.equal(out, outs[split]), split
            outs[split] = out
    finally:
        L.muon_debug_gram_split(-1)
    for split in (2, 3, 4):
        for k in range(K):
            got, base = f64(outs[split][k]), f64(outs[1][k])
            assert rel_fro(got, base) <= 1e-3, (split, k, rel_fro(got, base))
            assert rel_fro(got, omuon.newton_schulz(X[k], PE8, 1e-7)) <= 2e-2


def test_gram_space_routing_rule(L):
    assert L.muon_gram_space_route(256, 16384) and L.muon_gram_space_route(16384, 256)
    assert L.muon_gram_space_route(129, 516) and not L.muon_gram_space_route(129, 515)
    assert not L.muon_gram_space_route(257, 4096)          # m above 256
    assert not L.muon_gram_space_route(64, 128)            # the fused small-matrix kernel's
    assert L.muon_gram_space_route(64, 257)
    assert not L.muon_gram_space_route(768, 3072) and not L.muon_gram_space_route(1024, 4096)


def test_aspect_set_step_gram_space_and_plain_both_match_oracle(L):
    """The aspect set's two buckets (16 x 256 x 16384 and 16 x 16384 x 256; Student-t(3) gradients, 8 Polar
    Express steps, cautious decay, Nesterov) through muon_step_grouped, one step, on the Gram-space path (the
    rule's choice) and on the plain chain: both within the bar of the oracle's update on a sampled matrix of
    each bucket."""
    w = workloads.workload("aspect")
    hp = w.muon_hp
    assert L.muon_gram_space_route(256, 16384)
    shapes = [(16, 256, 16384), (16, 16384, 256)]
    base = []
    for b, (K, A, B) in enumerate(shapes):
        p = workloads.device_stack((K, A, B), "normal", w.param_std, 8000 + b, "bf16", DEV)
        g = workloads.device_stack((K, A, B), "student_t3", 1.0, 8100 + b, "bf16", DEV)
        base.append((p, g))
    results = {}
    try:
        for mode in (-1, 0):
            L.muon_debug_gram_space(mode)
            specs, ps = [], []
            for (K, A, B), (p0, g) in zip(shapes, base):
                p = p0.clone()
                m = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
                ps.append(p)
                specs.append((L.pointer_array([p[k] for k in range(K)], DEV),
                              L.pointer_array([g[k] for k in range(K)], DEV), m, K, A, B, L.MUON_BF16, L.MUON_BF16))
            bk = L.make_buckets(specs)
            ws = torch.zeros(L.muon_workspace_bytes_grouped(bk), dtype=torch.uint8, device=DEV)
            L.muon_step_grouped(bk, hp_struct(L, hp), ws)
            assert L.muon_check(ws) == L.MUON_OK
            results[mode] = ps
    finally:
        L.muon_debug_gram_space(-1)
    for b, ((K, A, B), (p0, g)) in enumerate(zip(shapes, base)):
        k = workloads.bucket_sample(K, w.cfg_id, 40 + b)[1]
        P0, Gk = f64(p0[k]), f64(g[k])
        ref, _, u = omuon.muon_update(P0, Gk, np.zeros_like(P0), lr=hp.lr, momentum=hp.momentum,
                                      weight_decay=hp.weight_decay, nesterov=hp.nesterov, cautious_wd=False,
                                      coeffs=hp.coeffs, eps=hp.eps, param_dtype="bf16")
        scale = omuon.update_scale(A, B)
        for mode in (-1, 0):
            got = f64(results[mode][b][k])
            # the cautious mask changes only the decay (lr * wd * p, a 2e-4 share of p): compare the step
            # itself, p_old - p_new with the decay term removed, against lr * scale * u
            step_gpu = P0 - got
            step_orc = hp.lr * scale * u
            decay = hp.lr * hp.weight_decay * np.abs(P0)
            err = np.linalg.norm(np.maximum(np.abs(step_gpu - step_orc) - decay, 0.0))
            assert err <= 2e-2 * np.linalg.norm(step_orc) + 2 ** -8 * np.linalg.norm(got), (mode, b, err)
