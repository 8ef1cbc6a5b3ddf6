"""The per-shape autotune, through the C ABI: the poly step's pipeline shape, the plain chain's scheduling,
and the Newton-Schulz path of stacks that can take the Gram-space chain.

The three compiled poly shapes (4 + 5, 5 + 3, 6 + 2 mainloop stages + epilogue slots) compute every tile the
same way, so each must give the same bits as the others on the same input (the shape the rule picks is
compared with the oracle in test_gpu_ns_steps); covered at a short, a long and a ragged contraction.
muon_autotune must record a shape for the grouped launch's contraction and a scheduling for the set, leave
parameters and momentum untouched, and a grouped step after it must equal, bit for bit, the same step with the
tables empty (shapes and scheduling never change a result). On the aspect set it must record a path for both
buckets, and the step after it must match the oracle.
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
    L.muon_autotune(got_b, hp, ws_got)
    shape = L.muon_autotune_poly_shape(768)
    assert shape in (0, 1, 2)
    assert L.muon_autotune_poly_shape(1024) == -1
    assert L.muon_autotune_scheduling(got_b) in (0, 1)
    print(f"GPT-2-small set: poly shape {shape}, scheduling {L.muon_autotune_scheduling(got_b)} (1 = counters)")
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
    assert L.muon_autotune_scheduling(got_b) == -1


def test_autotune_chooses_a_path_on_the_aspect_set(L):
    """Both aspect-set buckets can take the Gram-space chain; the autotune times each way and records a path
    (the Gram space, measured about twice as fast on these shapes). The step after it matches the oracle."""
    import numpy as np
    from oracle import muon as omuon
    from tests.gpu_common import f64
    L.muon_autotune_reset()
    w = workloads.workload("aspect")
    hp = w.muon_hp
    shapes = [(16, 256, 16384), (16, 16384, 256)]
    specs, keep = [], []
    for b, (K, A, B) in enumerate(shapes):
        p = workloads.device_stack((K, A, B), "normal", w.param_std, 8300 + b, "bf16", DEV)
        g = workloads.device_stack((K, A, B), "student_t3", 1.0, 8400 + b, "bf16", DEV)
        m = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
        keep.append((p, g, m, p[0].clone()))
        specs.append((L.pointer_array([p[k] for k in range(K)], DEV), L.pointer_array([g[k] for k in range(K)], DEV),
                      m, K, A, B, L.MUON_BF16, L.MUON_BF16))
    bk = L.make_buckets(specs)
    ws = torch.zeros(L.muon_workspace_bytes_grouped(bk), dtype=torch.uint8, device=DEV)
    hps = hp_struct(L, hp)
    L.muon_autotune(bk, hps, ws)
    routes = [L.muon_autotune_route(K, A, B) for K, A, B in shapes]
    splits = [L.muon_autotune_gram_split(K, A, B) for K, A, B in shapes]
    print(f"aspect set: recorded paths {routes} (1 = Gram space), fp32 Gram slices {splits}")
    assert routes == [1, 1]
    assert splits[0] == splits[1] and splits[0] in (1, 2, 3, 4)
    assert all(torch.count_nonzero(m) == 0 for _, _, m, _ in keep)
    L.muon_step_grouped(bk, hps, ws)
    assert L.muon_check(ws) == L.MUON_OK
    for (K, A, B), (p, g, m, p0) in zip(shapes, keep):
        P0, G0 = f64(p0), f64(g[0])
        ref, _, u = omuon.muon_update(P0, G0, np.zeros_like(P0), lr=hp.lr, momentum=hp.momentum,
                                      weight_decay=hp.weight_decay, nesterov=hp.nesterov, cautious_wd=False,
                                      coeffs=hp.coeffs, eps=hp.eps, param_dtype="bf16")
        # cautious decay changes only the decay term (lr * wd * p): compare the step with it allowed for
        step_gpu, step_orc = P0 - f64(p[0]), hp.lr * omuon.update_scale(A, B) * u
        err = np.linalg.norm(np.maximum(np.abs(step_gpu - step_orc) - hp.lr * hp.weight_decay * np.abs(P0), 0.0))
        assert err <= 2e-2 * np.linalg.norm(step_orc) + 2 ** -8 * np.linalg.norm(f64(p[0]))
    L.muon_autotune_reset()
    assert L.muon_autotune_route(16, 256, 16384) == -1
    assert L.muon_autotune_gram_split(16, 256, 16384) == -1


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
