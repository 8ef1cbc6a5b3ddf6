"""HybridMuonAdamW, the param_groups optimizer on top of the C ABI.

Checks, on a GPT-2-small-shaped layout cut to 2 layers: Muon groups route 2-D hidden matrices and AdamW
groups everything else, both match the oracle; optimizer state takes 4 bytes per Muon parameter and 8
per AdamW parameter (the budget printed in "Optimizers: AdamW, Muon and the distributed optimizer",
section "The optimizer's memory budget"); a run saved after step 2 and resumed in a fresh optimizer
matches an uninterrupted run bit for bit.
"""
import os

import numpy as np
import pytest
import torch

from oracle import adamw as oadamw
from oracle import muon as omuon
from tests.conftest import read_golden
from tests.gpu_common import DEV, build_lib, f64
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return build_lib()


def _model(seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: (torch.randn(s, generator=g) * 1e-3).to(torch.bfloat16).to(DEV)
    hidden = [mk(768, 2304), mk(768, 768), mk(768, 3072), mk(3072, 768), mk(768, 2304), mk(768, 768)]
    other = [mk(1000, 768), mk(768), mk(768)]
    return hidden, other


def _grads(params, step, seed):
    g = torch.Generator().manual_seed(1000 * seed + step)
    for p in params:
        p.grad = (torch.randn(p.shape, generator=g) * 1e-3).to(torch.bfloat16).to(DEV)


def _opt(hidden, other):
    from adamw_hybrid_optimizer_gb300 import HybridMuonAdamW
    m = workloads.workload("gpt2s").muon_hp
    a = workloads.workload("gpt2s").adamw_hp
    return HybridMuonAdamW([
        {"params": hidden, "kind": "muon", "lr": m.lr, "momentum": m.momentum, "weight_decay": m.weight_decay},
        {"params": other, "kind": "adamw", "lr": a.lr, "betas": (a.beta1, a.beta2), "eps": a.eps,
         "weight_decay": a.weight_decay},
    ])


def test_optimizer_matches_oracle_and_state_budget(L, golden_dir):
    hidden, other = _model(0)
    before = [f64(p) for p in hidden + other]
    opt = _opt(hidden, other)
    _grads(hidden + other, 1, 0)
    grads = [f64(p.grad) for p in hidden + other]
    opt.step()
    torch.cuda.synchronize()
    m = workloads.workload("gpt2s").muon_hp
    a = workloads.workload("gpt2s").adamw_hp
    for i, p in enumerate(hidden):
        ref, _, _ = omuon.muon_update(before[i], grads[i], np.zeros_like(before[i]), lr=m.lr, momentum=m.momentum,
                                      weight_decay=m.weight_decay, coeffs=m.coeffs, eps=m.eps, param_dtype="bf16")
        assert np.linalg.norm(f64(p) - ref) <= 2e-2 * np.linalg.norm(ref - before[i]) + 2 ** -8 * np.linalg.norm(ref)
    for j, p in enumerate(other):
        i = len(hidden) + j
        ref, _, _ = oadamw.adamw_update(before[i], grads[i], 0, 0, 1, lr=a.lr, beta1=a.beta1, beta2=a.beta2,
                                        eps=a.eps, weight_decay=a.weight_decay, param_dtype="bf16")
        ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(ref), 1e-30))[1] - 8)
        assert np.all(np.abs(f64(p) - ref) <= ulp * 1.0001 + 1e-6 * (np.abs(before[i]) + a.lr))
    fx = read_golden(os.path.join(golden_dir, "optimizer_state_bytes.txt"))
    state_bytes = lambda ps: sum(t.numel() * t.element_size() for p in ps for t in opt.state[p].values())
    assert state_bytes(hidden) / sum(p.numel() for p in hidden) == fx["muon"][0]
    assert state_bytes(other) / sum(p.numel() for p in other) == fx["adamw"][0]


def test_resume_bit_matches_uninterrupted_run(L):
    hidden, other = _model(1)
    params = hidden + other
    ref_opt = _opt(hidden, other)
    snap = [p.clone() for p in params]
    for step in (1, 2, 3, 4):
        _grads(params, step, 1)
        ref_opt.step()
    ref_final = [p.clone() for p in params]
    # rerun: two steps, checkpoint, fresh optimizer, restore, two more steps
    for p, s0 in zip(params, snap):
        p.data.copy_(s0)
    opt = _opt(hidden, other)
    for step in (1, 2):
        _grads(params, step, 1)
        opt.step()
    sd = opt.state_dict()
    saved = [p.clone() for p in params]
    opt2 = _opt(hidden, other)
    opt2.load_state_dict(sd)
    for p, s in zip(params, saved):
        p.data.copy_(s)
    for step in (3, 4):
        _grads(params, step, 1)
        opt2.step()
    torch.cuda.synchronize()
    for a_, b_ in zip(params, ref_final):
        assert torch.equal(a_, b_)


def test_is_adamw_false_group_takes_adam_with_l2(L):
    """An AdamW group with is_adamw=False runs Adam with L2 regularisation ("dtensor-muon 0.1.0", "Key options")."""
    from adamw_hybrid_optimizer_gb300 import HybridMuonAdamW
    a = workloads.workload("gpt2s").adamw_hp
    _, other = _model(3)
    before = [f64(p) for p in other]
    opt = HybridMuonAdamW([{"params": other, "kind": "adamw", "lr": a.lr, "betas": (a.beta1, a.beta2), "eps": a.eps,
                            "weight_decay": 0.1, "is_adamw": False}])
    _grads(other, 1, 3)
    grads = [f64(p.grad) for p in other]
    opt.step()
    torch.cuda.synchronize()
    for i, p in enumerate(other):
        ref, _, _ = oadamw.adam_l2_update(before[i], grads[i], 0, 0, 1, lr=a.lr, beta1=a.beta1, beta2=a.beta2,
                                          eps=a.eps, weight_decay=0.1, param_dtype="bf16")
        ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(ref), 1e-30))[1] - 8)
        assert np.all(np.abs(f64(p) - ref) <= ulp * 1.0001 + 1e-6 * (np.abs(before[i]) + a.lr))
        # and it is not the decoupled rule on this input
        dec, _, _ = oadamw.adamw_update(before[i], grads[i], 0, 0, 1, lr=a.lr, beta1=a.beta1, beta2=a.beta2,
                                        eps=a.eps, weight_decay=0.1, param_dtype="bf16")
        assert not np.array_equal(dec, ref)


def test_master_weights_option(L):
    """master_weights=True: fp32 masters take the update (the oracle's fp32-parameter rules), and every bf16
    parameter equals its master rounded to bf16."""
    from adamw_hybrid_optimizer_gb300 import HybridMuonAdamW
    m = workloads.workload("gpt2s").muon_hp
    a = workloads.workload("gpt2s").adamw_hp
    hidden, other = _model(5)
    before = [f64(p) for p in hidden + other]
    opt = HybridMuonAdamW([
        {"params": hidden, "kind": "muon", "lr": m.lr, "momentum": m.momentum, "weight_decay": m.weight_decay,
         "master_weights": True},
        {"params": other, "kind": "adamw", "lr": a.lr, "betas": (a.beta1, a.beta2), "eps": a.eps,
         "weight_decay": a.weight_decay, "master_weights": True},
    ])
    _grads(hidden + other, 1, 5)
    grads = [f64(p.grad) for p in hidden + other]
    opt.step()
    torch.cuda.synchronize()
    for i, p in enumerate(hidden):
        master = opt.state[p]["master"]
        ref, _, _ = omuon.muon_update(before[i], grads[i], np.zeros_like(before[i]), lr=m.lr, momentum=m.momentum,
                                      weight_decay=m.weight_decay, coeffs=m.coeffs, eps=m.eps, param_dtype="f32")
        assert np.linalg.norm(f64(master) - ref) <= 2e-2 * np.linalg.norm(ref - before[i])
        assert torch.equal(p, master.to(torch.bfloat16))
    for j, p in enumerate(other):
        i = len(hidden) + j
        master = opt.state[p]["master"]
        ref, _, _ = oadamw.adamw_update(before[i], grads[i], 0, 0, 1, lr=a.lr, beta1=a.beta1, beta2=a.beta2,
                                        eps=a.eps, weight_decay=a.weight_decay, param_dtype="f32")
        assert np.all(np.abs(f64(master) - ref) <= 1e-6 * (np.abs(before[i]) + a.lr))
        assert torch.equal(p, master.to(torch.bfloat16))


def test_several_groups_equal_one_optimizer_per_group(L):
    """Two Muon groups (different lr and decay) and two AdamW groups (with and without decay) in one optimizer:
    the step issues muon_step_grouped for the first Muon group and one hybrid_step for the second with every
    AdamW tensor. Groups are independent, so each parameter must end bit for bit where one optimizer per
    group puts it."""
    from adamw_hybrid_optimizer_gb300.optim import HybridMuonAdamW
    gen = torch.Generator().manual_seed(77)
    shapes = {"m1": [(256, 512), (256, 512)], "m2": [(768, 768), (512, 256)], "a1": [(5000,)], "a2": [(768,), (33,)]}
    init = {k: [(torch.randn(s, generator=gen) * 1e-2).to(torch.bfloat16) for s in v] for k, v in shapes.items()}
    grads = [{k: [(torch.randn(s, generator=gen) * 1e-3).to(torch.bfloat16) for s in v] for k, v in shapes.items()}
             for _ in range(3)]
    spec = {"m1": {"kind": "muon", "lr": 0.02, "weight_decay": 0.01},
            "m2": {"kind": "muon", "lr": 0.01, "weight_decay": 0.0, "cautious_wd": True},
            "a1": {"kind": "adamw", "lr": 3e-4, "weight_decay": 0.1},
            "a2": {"kind": "adamw", "lr": 1e-3, "weight_decay": 0.0}}

    def run(keys):
        ps = {k: [t.clone().to(DEV) for t in init[k]] for k in keys}
        opt = HybridMuonAdamW([dict(spec[k], params=ps[k]) for k in keys])
        for g in grads:
            for k in keys:
                for p, gr in zip(ps[k], g[k]):
                    p.grad = gr.to(DEV)
            opt.step()
        torch.cuda.synchronize()
        return ps

    together = run(["m1", "m2", "a1", "a2"])
    for k in shapes:
        alone = run([k])[k]
        for a, b in zip(together[k], alone):
            assert torch.equal(a, b), k
