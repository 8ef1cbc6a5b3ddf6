"""muon_step_grouped: one grouped launch per Newton-Schulz step kind over several buckets.

Grouping changes only which CTA computes which tile, never the arithmetic of a tile, so the result must
equal, bit for bit, one muon_step_batched call per bucket on the same inputs (which the per-bucket tests
compare with the oracle). Covered: the GPT-2-small set (4 buckets, one of them transposed), ten buckets
of distinct ragged shapes with fp32 and bf16 parameters (more than one launch per step kind), eighteen
buckets (more than one launch of the momentum/norm pass), a workspace that another call with another
layout used in between, and steps cut into pieces of different sizes.
"""
import numpy as np
import pytest
import torch

from oracle.buckets import plan_buckets
from tests.gpu_common import DEV, build_lib, f64, hp_struct, rel_fro
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return build_lib()


def _make(shapes, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    out = []
    for (K, A, B) in shapes:
        p = (torch.randn((K, A, B), generator=g) * 1e-3).to(dtype).to(DEV)
        grads = [(torch.randn((K, A, B), generator=g) * 1e-3).to(dtype).to(DEV) for _ in range(2)]
        out.append((p, grads))
    return out


def _run_both(L, shapes, dtype, hp, seed=0):
    data = _make(shapes, dtype, seed)
    code = L.MUON_F32 if dtype == torch.float32 else L.MUON_BF16
    hps = hp_struct(L, hp)
    # per-bucket reference: muon_step_batched
    ref_p, ref_m = [], []
    for (K, A, B), (p0, grads) in zip(shapes, data):
        p = p0.clone()
        mom = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
        ws = torch.zeros(L.muon_workspace_bytes(K, A, B), dtype=torch.uint8, device=DEV)
        pp = L.pointer_array([p[k] for k in range(K)], DEV)
        for g in grads:
            L.muon_step_batched(pp, code, L.pointer_array([g[k] for k in range(K)], DEV), code, mom, K, A, B, hps, ws)
        assert L.muon_check(ws) == L.MUON_OK
        ref_p.append(p)
        ref_m.append(mom)
    # grouped
    ps = [p0.clone() for p0, _ in data]
    moms = [torch.zeros(s, dtype=torch.float32, device=DEV) for s in shapes]
    pptr = [L.pointer_array([p[k] for k in range(s[0])], DEV) for p, s in zip(ps, shapes)]
    for step in range(2):
        gptr = [L.pointer_array([g[step][k] for k in range(s[0])], DEV) for (_, g), s in zip(data, shapes)]
        bk = L.make_buckets([(pp, gp, m, K, A, B, code, code) for pp, gp, m, (K, A, B) in zip(pptr, gptr, moms, shapes)])
        ws = torch.zeros(L.muon_workspace_bytes_grouped(bk), dtype=torch.uint8, device=DEV)
        L.muon_step_grouped(bk, hps, ws)
        assert L.muon_check(ws) == L.MUON_OK
    for i in range(len(shapes)):
        assert torch.equal(ps[i], ref_p[i]), i
        assert torch.equal(moms[i], ref_m[i]), i
    return ps


def test_grouped_equals_per_bucket_gpt2_small(L):
    w = workloads.workload("gpt2s")
    plan = plan_buckets(workloads.shape_list(w))
    shapes = [(K, A, B) for (A, B), K in zip(plan["bucket_shapes"], plan["bucket_K"])]
    _run_both(L, shapes, torch.bfloat16, w.muon_hp, seed=1)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("deps", [1, 0])
def test_grouped_equals_per_bucket_ten_ragged_buckets(L, dtype, deps):
    """deps: the grouped chain's launches wait per matrix on counters (1) or on their whole predecessor (0);
    the library's own rule would pick the launch order for these small shapes, so both are forced."""
    shapes = [(3, 64, 128), (2, 136, 72), (1, 8, 24), (4, 200, 264), (2, 256, 256), (1, 520, 776),
              (2, 40, 1), (3, 1, 96), (2, 384, 130), (1, 130, 384)]
    hp = workloads.workload("tiny").muon_hp
    L.muon_debug_counter_deps(deps)
    try:
        ps = _run_both(L, shapes, dtype, hp, seed=2)
    finally:
        L.muon_debug_counter_deps(-1)
    assert all(torch.isfinite(p.float()).all() for p in ps)


def test_grouped_step_matches_oracle_on_one_sample(L):
    """A direct oracle check on the grouped path too (first matrix of each GPT-2-small bucket, step 1)."""
    from oracle import muon as omuon
    w = workloads.workload("gpt2s")
    hp = w.muon_hp
    plan = plan_buckets(workloads.shape_list(w))
    specs, keep = [], []
    for b, ((A, B), K) in enumerate(zip(plan["bucket_shapes"], plan["bucket_K"])):
        members = [i for i, bid in enumerate(plan["bucket_id"]) if bid == b]
        p = torch.stack([workloads.muon_param_init(w, i) for i in members]).to(DEV)
        g = torch.stack([workloads.muon_grad(w, 1, i) for i in members]).to(DEV)
        m = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
        keep.append((p, g, m, members, f64(p[0])))
        specs.append((L.pointer_array([p[k] for k in range(K)], DEV), L.pointer_array([g[k] for k in range(K)], DEV),
                      m, K, A, B, L.MUON_BF16, L.MUON_BF16))
    bk = L.make_buckets(specs)
    ws = torch.zeros(L.muon_workspace_bytes_grouped(bk), dtype=torch.uint8, device=DEV)
    L.muon_step_grouped(bk, hp_struct(L, hp), ws)
    assert L.muon_check(ws) == L.MUON_OK
    for p, g, m, members, p0 in keep:
        ref, _, _ = omuon.muon_update(p0, f64(g[0]), np.zeros_like(p0), lr=hp.lr, momentum=hp.momentum,
                                      weight_decay=hp.weight_decay, nesterov=hp.nesterov, coeffs=hp.coeffs,
                                      eps=hp.eps, param_dtype="bf16")
        got = f64(p[0])
        assert np.linalg.norm(got - ref) <= 2e-2 * np.linalg.norm(ref - p0) + 2 ** -8 * np.linalg.norm(ref)


def test_grouped_equals_per_bucket_eighteen_buckets(L):
    shapes = [(1 + i % 3, 8 * (1 + i), 16 * (1 + (i * 7) % 5)) for i in range(18)]
    hp = workloads.workload("tiny").muon_hp
    _run_both(L, shapes, torch.bfloat16, hp, seed=3)


def test_workspace_reused_by_another_layout(L):
    """A call leaves the workspace full of its own data; a later call with another layout must not read
    any of it as state (its per-matrix counters are cleared by the call itself)."""
    hp = hp_struct(L, workloads.workload("tiny").muon_hp)
    shapes = [(3, 64, 128), (2, 136, 72)]
    data = _make(shapes, torch.bfloat16, 4)
    code = L.MUON_BF16

    def grouped(ws):
        ps = [p0.clone() for p0, _ in data]
        moms = [torch.zeros(s, dtype=torch.float32, device=DEV) for s in shapes]
        bk = L.make_buckets([(L.pointer_array([p[k] for k in range(K)], DEV),
                              L.pointer_array([g[0][k] for k in range(K)], DEV), m, K, A, B, code, code)
                             for p, m, (_, g), (K, A, B) in zip(ps, moms, data, shapes)])
        L.muon_step_grouped(bk, hp, ws)
        assert L.muon_check(ws) == L.MUON_OK
        return ps

    fresh = torch.zeros(L.muon_workspace_bytes(4, 256, 512), dtype=torch.uint8, device=DEV)
    ref = grouped(torch.zeros_like(fresh))
    # another layout writes the same bytes (counters of this call sit where the other call keeps data)
    big = torch.randn((4, 256, 512), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).to(DEV)
    out = torch.empty_like(big)
    L.ns_orthogonalize(big, out, [(3.4445, -4.775, 2.0315)] * 5, 1e-7, fresh)
    assert L.muon_check(fresh) == L.MUON_OK
    got = grouped(fresh)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("deps", [1, 0])
def test_grouped_equals_per_bucket_with_every_path(L, deps):
    """Buckets on all three paths in one grouped call: the fused small-matrix chain, the Gram-space chain (one
    and two 128-row blocks, wide and tall, a cluster left partly idle) and the plain GEMM chain, with the plain
    chain's launches overlapping through counters (1) or in launch order (0). The branches run first and the
    plain chain's first launch waits for them; every result equals the per-bucket calls bit for bit."""
    shapes = [(3, 64, 128), (2, 256, 2048), (3, 100, 1000), (2, 2048, 200), (2, 512, 768), (1, 40, 1)]
    assert L.muon_gram_space_route(256, 2048) and L.muon_gram_space_route(100, 1000)
    assert L.muon_gram_space_route(2048, 200) and not L.muon_gram_space_route(512, 768)
    hp = workloads.workload("aspect").muon_hp
    L.muon_debug_counter_deps(deps)
    try:
        ps = _run_both(L, shapes, torch.bfloat16, hp, seed=6)
    finally:
        L.muon_debug_counter_deps(-1)
    assert all(torch.isfinite(p.float()).all() for p in ps)


@pytest.mark.parametrize("elems", [1, 300_000])
def test_pieces_change_no_result(L, elems):
    """Every call runs its step in pieces (muon_debug_piece_elems): with one matrix per piece (1), or with stacks
    cut along K and small buckets packed together (300 000 elements), parameters equal the default's (one piece)
    bit for bit on every path, grouped and per bucket alike, and so does ns_orthogonalize. The fp32 Gram's slice
    count, which depends on a stack's K, is forced to 2 in both runs."""
    shapes = [(3, 64, 128), (4, 256, 2048), (2, 2048, 200), (3, 512, 768), (5, 100, 1000)]
    hp = workloads.workload("aspect").muon_hp
    results, ns = {}, {}
    gen = torch.Generator().manual_seed(12)
    x = torch.randn((4, 256, 2048), generator=gen).to(torch.bfloat16).to(DEV)
    L.muon_debug_gram_split(2)
    try:
        for e in (0, elems):
            L.muon_debug_piece_elems(e)
            results[e] = _run_both(L, shapes, torch.bfloat16, hp, seed=9)
            out = torch.empty_like(x)
            ws = torch.zeros(L.muon_workspace_bytes(4, 256, 2048), dtype=torch.uint8, device=DEV)
            L.ns_orthogonalize(x, out, hp.coeffs, 1e-7, ws)
            assert L.muon_check(ws) == L.MUON_OK
            ns[e] = out
    finally:
        L.muon_debug_piece_elems(0)
        L.muon_debug_gram_split(-1)
    for a, b in zip(results[0], results[elems]):
        assert torch.equal(a, b)
    assert torch.equal(ns[0], ns[elems])
