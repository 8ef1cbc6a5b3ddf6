"""The Newton-Schulz chain with G and H stored as their upper 256-blocks (the default) against the chain with
both halves stored.

A step that reads G or H takes a block below the diagonal as the transpose of the stored block above it. That
block holds the values the mirrored store would have written there, so the two modes must agree bit for bit:
in ns_orthogonalize on wide, tall, square and ragged stacks (m a multiple of 256 or not, one or several
256-blocks), in every POLY pipeline shape, and in grouped momentum steps with fp32 and bf16 parameters,
cautious decay and both launch-scheduling modes.
"""
import dataclasses

import pytest
import torch

from tests.gpu_common import DEV, build_lib, hp_struct, workspace
import workloads

pytestmark = pytest.mark.gpu

CLASSIC5 = [(3.4445, -4.7750, 2.0315)] * 5


@pytest.fixture(scope="module")
def L():
    lib = build_lib()
    yield lib
    lib.muon_debug_half_symmetric(1)


def _ns(L, x, odt, half):
    K, A, B = x.shape
    L.muon_debug_half_symmetric(half)
    out = torch.full((K, A, B), float("nan"), dtype=odt, device=DEV)
    ws = workspace(L, K, A, B)
    L.ns_orthogonalize(x, out, CLASSIC5, 1e-7, ws)
    assert L.muon_check(ws) == L.MUON_OK
    return out


@pytest.mark.parametrize("K,A,B,xdt,odt", [
    (3, 768, 2304, torch.bfloat16, torch.float32),   # three 256-blocks
    (2, 2304, 768, torch.float32, torch.bfloat16),   # tall: transposed to wide and back
    (2, 640, 640, torch.bfloat16, torch.float32),    # square, a partial third block
    (2, 700, 1000, torch.bfloat16, torch.bfloat16),  # ragged m and n
    (3, 300, 2000, torch.float32, torch.float32),    # two blocks, the second nearly empty
    (1, 1536, 1664, torch.bfloat16, torch.float32),  # six blocks
])
def test_half_stored_chain_is_bitwise_the_whole_chain(L, K, A, B, xdt, odt):
    g = torch.Generator().manual_seed(K * 7 + A + B)
    x = torch.randn((K, A, B), generator=g, dtype=torch.float64).to(xdt).to(DEV)
    half = _ns(L, x, odt, 1)
    whole = _ns(L, x, odt, 0)
    assert torch.isfinite(half.float()).all()
    assert torch.equal(half, whole)


@pytest.mark.parametrize("dtype,deps", [(torch.bfloat16, 1), (torch.float32, 0)])
def test_half_stored_grouped_steps_are_bitwise_the_whole_ones(L, dtype, deps):
    shapes = [(3, 768, 2304), (2, 3072, 768), (2, 520, 520), (3, 260, 1100)]
    hp = dataclasses.replace(workloads.workload("tiny").muon_hp, cautious_wd=True)
    code = L.MUON_F32 if dtype == torch.float32 else L.MUON_BF16
    g = torch.Generator().manual_seed(11)
    p0 = [(torch.randn(s, generator=g) * 1e-3).to(dtype).to(DEV) for s in shapes]
    grads = [[(torch.randn(s, generator=g) * 1e-3).to(dtype).to(DEV) for s in shapes] for _ in range(2)]
    results = []
    L.muon_debug_counter_deps(deps)
    try:
        for half in (1, 0):
            L.muon_debug_half_symmetric(half)
            ps = [p.clone() for p in p0]
            moms = [torch.zeros(s, dtype=torch.float32, device=DEV) for s in shapes]
            pptr = [L.pointer_array([p[k] for k in range(s[0])], DEV) for p, s in zip(ps, shapes)]
            for step in range(2):
                gptr = [L.pointer_array([gr[k] for k in range(s[0])], DEV) for gr, s in zip(grads[step], shapes)]
                bk = L.make_buckets([(pp, gp, m, K, A, B, code, code)
                                     for pp, gp, m, (K, A, B) in zip(pptr, gptr, moms, shapes)])
                ws = torch.zeros(L.muon_workspace_bytes_grouped(bk), dtype=torch.uint8, device=DEV)
                L.muon_step_grouped(bk, hp_struct(L, hp), ws)
                assert L.muon_check(ws) == L.MUON_OK
            results.append((ps, moms))
    finally:
        L.muon_debug_counter_deps(-1)
        L.muon_debug_half_symmetric(1)
    (ph, mh), (pw, mw) = results
    for a, b in zip(ph, pw):
        assert torch.equal(a, b)
    for a, b in zip(mh, mw):
        assert torch.equal(a, b)
    assert any(not torch.equal(a, b) for a, b in zip(ph, p0))   # the steps moved the parameters


@pytest.mark.parametrize("shape", [0, 1, 2])
def test_half_stored_chain_in_every_poly_pipeline_shape(L, shape):
    # each POLY shape has its own ring of G blocks for b·G, which in upper-block mode also carries the blocks
    # below the diagonal of the diagonal pair tiles
    g = torch.Generator().manual_seed(40 + shape)
    x = torch.randn((2, 640, 1536), generator=g, dtype=torch.float64).to(torch.bfloat16).to(DEV)
    L.muon_debug_poly_shape(shape)
    try:
        half = _ns(L, x, torch.float32, 1)
        whole = _ns(L, x, torch.float32, 0)
    finally:
        L.muon_debug_poly_shape(-1)
        L.muon_debug_half_symmetric(1)
    assert torch.isfinite(half).all()
    assert torch.equal(half, whole)
