"""The per-shape autotune of the poly step's pipeline shape, through the C ABI.

The three compiled shapes (4 + 5, 5 + 3, 6 + 2 mainloop stages + epilogue slots) compute every tile the
same way, so each must give the same bits as the others on the same input (the shape the rule picks is
compared with the oracle in test_gpu_ns_steps); covered at a short, a long and a ragged contraction.
muon_autotune must record a shape for the grouped launch's contraction, and a grouped step after it must
equal, bit for bit, the same step with the table empty.
"""
import pytest
import torch

from tests.gpu_common import DEV, build_lib, ctrl_ws, hp_struct
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    lib = build_lib()
    yield lib
    lib.muon_debug_poly_shape(-1)
    lib.muon_autotune_reset()


@pytest.mark.parametrize("K,m", [(6, 768), (2, 2560), (3, 200)])
def test_every_poly_shape_gives_the_same_bits(L, K, m):
    gen = torch.Generator().manual_seed(m)
    x = torch.randn((K, m, m), generator=gen) / m ** 0.5
    g = (x + x.transpose(1, 2)).to(torch.bfloat16).to(DEV)   # symmetric, as the Gram is
    outs = []
    ws = ctrl_ws()
    try:
        for shape in range(3):
            L.muon_debug_poly_shape(shape)
            h = torch.full((K, m, m), float("nan"), dtype=torch.bfloat16, device=DEV)
            L.ns_poly(g, h, 3.4445, -4.7750, 2.0315, ws)
            torch.cuda.synchronize()
            outs.append(h)
    finally:
        L.muon_debug_poly_shape(-1)
    assert L.muon_check(ws) == L.MUON_OK
    assert not torch.isnan(outs[0].float()).any()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def _gpt2s_set(L, seed):
    w = workloads.workload("gpt2s")
    plan = L.muon_plan_buckets(workloads.shape_list(w))
    gen = torch.Generator().manual_seed(seed)
    specs, keep = [], []
    for (A, B), K in zip(plan["bucket_shapes"], plan["bucket_K"]):
        p = (torch.randn((K, A, B), generator=gen) * 1e-3).to(torch.bfloat16).to(DEV)
        gr = (torch.randn((K, A, B), generator=gen) * 1e-3).to(torch.bfloat16).to(DEV)
        mom = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
        keep.append((p, gr, mom))
        specs.append((L.pointer_array([p[k] for k in range(K)], DEV), L.pointer_array([gr[k] for k in range(K)], DEV),
                      mom, K, A, B, L.MUON_BF16, L.MUON_BF16))
    return L.make_buckets(specs), keep, hp_struct(L, w.muon_hp)


def test_autotune_records_a_shape_and_keeps_results(L):
    L.muon_autotune_reset()
    ref_b, ref, hp = _gpt2s_set(L, 3)
    got_b, got, _ = _gpt2s_set(L, 3)
    ws_ref = torch.zeros(L.muon_workspace_bytes_grouped(ref_b), dtype=torch.uint8, device=DEV)
    ws_got = torch.zeros_like(ws_ref)
    L.muon_step_grouped(ref_b, hp, ws_ref)          # table empty: the rule's shape
    L.muon_autotune(got_b, ws_got)
    shape = L.muon_autotune_poly_shape(768)
    assert shape in (0, 1, 2)
    assert L.muon_autotune_poly_shape(1024) == -1
    # the autotune touched only the workspace: parameters and momentum are as they were
    for (p, _, mom), (p0, _, mom0) in zip(got, ref):
        assert torch.count_nonzero(mom) == 0
    L.muon_step_grouped(got_b, hp, ws_got)          # the measured shape
    torch.cuda.synchronize()
    assert L.muon_check(ws_got) == L.MUON_OK
    for (p, _, mom), (p0, _, mom0) in zip(got, ref):
        assert torch.equal(p, p0) and torch.equal(mom, mom0)
    L.muon_autotune_reset()
    assert L.muon_autotune_poly_shape(768) == -1


def test_optimizer_autotune_option(L):
    """autotune=True measures the shape before the group's first step; the updates equal autotune=False's."""
    from adamw_hybrid_optimizer_gb300.optim import HybridMuonAdamW
    L.muon_autotune_reset()
    gen = torch.Generator().manual_seed(8)
    shapes = [(768, 768), (768, 3072), (3072, 768)]
    base = [(torch.randn(s, generator=gen) * 1e-3).to(torch.bfloat16) for s in shapes]
    grads = [[(torch.randn(s, generator=gen) * 1e-3).to(torch.bfloat16) for s in shapes] for _ in range(2)]
    runs = []
    for tune in (False, True):
        ps = [b.clone().to(DEV) for b in base]
        opt = HybridMuonAdamW([{"params": ps, "kind": "muon", "autotune": tune}])
        for gs in grads:
            for p, g in zip(ps, gs):
                p.grad = g.to(DEV)
            opt.step()
        torch.cuda.synchronize()
        runs.append(ps)
    assert L.muon_autotune_poly_shape(768) in (0, 1, 2)
    for a, b in zip(*runs):
        assert torch.equal(a, b)
    L.muon_autotune_reset()
