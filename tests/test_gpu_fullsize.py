"""Full-size GPU runs checked against the oracle on sampled matrices.

* Llama-3-8B-shaped Muon set: 32 layers x {q, o 4096x4096; k, v 1024x4096; gate, up 14336x4096;
  down 4096x14336} bf16, fp32 momentum, the workload's 3 grouped steps over all four buckets (the launch
  configuration of the bench's grouped call) with momentum carried. Inputs are drawn on the device from
  seeded generators; the oracle checks one seeded matrix of each large bucket and the first, last and one
  seeded matrix of the 1024x4096 one.
* Llama-3-8B AdamW set (1,050,939,392 elements) through one grouped call, 3 steps, sampled.
* Newton-Schulz sweep sizes n = 2048, 4096, 8192 (K = 64 square bf16 stacks): the oracle checks sampled
  matrices (three at 2048, one at the larger sizes).
Bars as elsewhere: relative Frobenius error <= 2e-2 of the update / of the orthogonalised output.
"""
import numpy as np
import pytest
import torch

from oracle import adamw as oadamw
from oracle import muon as omuon
from oracle.buckets import plan_buckets
from tests.gpu_common import DEV, bf16_ulp, build_lib, f64, hp_struct, rel_fro
import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def L():
    return build_lib()


def test_llama8b_grouped_three_steps_sampled(L):
    """The workload's 3 steps with momentum carried, so steps 2 and 3 orthogonalise G + mu*M with M != 0
    (Nesterov). Every step: the sampled matrices' momentum element by element, and their parameters against
    the oracle's own trajectory."""
    w = workloads.workload("llama8b")
    hp = w.muon_hp
    assert w.steps == 3 and hp.nesterov
    plan = plan_buckets(workloads.shape_list(w))
    buckets = []
    for b, ((A, B), K) in enumerate(zip(plan["bucket_shapes"], plan["bucket_K"])):
        p = workloads.device_stack((K, A, B), "normal", w.param_std, 3000 + b, "bf16", DEV)
        g = torch.empty((K, A, B), dtype=torch.bfloat16, device=DEV)
        m = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
        if K > 32 and A * B <= 1024 * 4096:
            sample = workloads.bucket_sample(K, w.cfg_id, b)
        else:
            sample = [workloads.bucket_sample(K, w.cfg_id, b)[1]]
        orc = {k: {"p": f64(p[k]), "m": np.zeros((A, B))} for k in sample}
        for k in sample:
            orc[k]["p0"] = orc[k]["p"].copy()
        buckets.append((p, g, m, K, A, B, sample, orc))
    specs = [(L.pointer_array([p[k] for k in range(K)], DEV), L.pointer_array([g[k] for k in range(K)], DEV), m, K, A,
              B, L.MUON_BF16, L.MUON_BF16) for p, g, m, K, A, B, _, _ in buckets]
    arr = L.make_buckets(specs)
    ws = torch.zeros(L.muon_workspace_bytes_grouped(arr), dtype=torch.uint8, device=DEV)
    hps = hp_struct(L, hp)
    for step in range(1, w.steps + 1):
        before = []
        for b, (p, g, m, K, A, B, sample, orc) in enumerate(buckets):
            g.copy_(workloads.device_stack((K, A, B), "normal", w.grad_std, 3100 + 16 * step + b, "bf16", DEV))
            before.append({k: f64(m[k]) for k in sample})
        L.muon_step_grouped(arr, hps, ws)
        assert L.muon_check(ws) == L.MUON_OK
        for (p, g, m, K, A, B, sample, orc), m_before in zip(buckets, before):
            assert torch.isfinite(p.float()).all()
            for k in sample:
                gk = f64(g[k])
                o = orc[k]
                m_prev = o["m"]
                ref, mref, _ = omuon.muon_update(o["p"], gk, m_prev, lr=hp.lr, momentum=hp.momentum,
                                                 weight_decay=hp.weight_decay, nesterov=hp.nesterov,
                                                 coeffs=hp.coeffs, eps=hp.eps, param_dtype="bf16")
                o["p"], o["m"] = ref, mref
                got_m = f64(m[k])
                if step == 1:
                    assert np.array_equal(got_m, mref)     # M = G exactly
                else:
                    assert np.count_nonzero(m_before[k]) > 0
                    carried = hp.momentum * np.abs(m_before[k] - m_prev) * (1 + 1e-6)
                    terms = np.abs(hp.momentum * m_before[k]) + np.abs(gk)
                    assert np.all(np.abs(got_m - mref) <= carried + 1e-6 * terms + 1e-30), (step, A, B, k)
                got = f64(p[k])
                moved = np.linalg.norm(ref - o["p0"])
                assert np.linalg.norm(got - ref) <= 2e-2 * moved + 2 ** -8 * np.linalg.norm(ref), (step, A, B, k)
    del ws, arr, specs, buckets
    torch.cuda.empty_cache()


def test_llama8b_adamw_set_grouped_sampled(L):
    """AdamW on the Llama-3-8B set at full size through one grouped call: embedding and head (128256 x 4096,
    wd 0.1) and the 65 RMSNorm 4096-vectors (wd 0), bf16 params and grads, fp32 moments, 3 steps. The oracle
    follows its own trajectory on a seeded sample of each large tensor plus its first and last 1000 elements,
    and on every element of the norm vectors."""
    w = workloads.workload("llama8b")
    a = w.adamw_hp
    n_total = sum(t.numel for t in w.adamw)
    assert n_total == 1_050_939_392
    p = workloads.device_stack((1, 1, n_total), "normal", w.param_std, 3200, "bf16", DEV).view(-1)
    g = torch.empty(n_total, dtype=torch.bfloat16, device=DEV)
    mo = torch.zeros(n_total, dtype=torch.float32, device=DEV)
    vo = torch.zeros(n_total, dtype=torch.float32, device=DEV)
    hps, specs, samples, off = {}, [], [], 0
    rng = np.random.default_rng(31)
    for t in w.adamw:
        h = hps.setdefault(t.weight_decay, L.make_adamw_hparams(a.lr, a.beta1, a.beta2, a.eps, t.weight_decay, 1))
        sl = slice(off, off + t.numel)
        specs.append((p[sl], g[sl], mo[sl], vo[sl], h))
        if t.numel > 100_000:
            idx = np.unique(np.concatenate([rng.integers(0, t.numel, 200_000), np.arange(1000),
                                            np.arange(t.numel - 1000, t.numel)]))
        else:
            idx = np.arange(t.numel)
        samples.append((off + idx, t.weight_decay))
        off += t.numel
    tensors = L.make_adamw_tensors(specs)
    aws = torch.zeros(L.adamw_workspace_bytes_grouped(len(specs)), dtype=torch.uint8, device=DEV)
    allidx = np.concatenate([s for s, _ in samples])
    wd = np.concatenate([np.full(len(s), d) for s, d in samples])
    idx_t = torch.from_numpy(allidx).to(DEV)
    po = f64(p[idx_t])
    mref, vref = np.zeros(len(allidx)), np.zeros(len(allidx))
    em, ev = np.zeros(len(allidx)), np.zeros(len(allidx))   # fp32 rounding carried from step to step
    dp = np.zeros(len(allidx))                                # |gpu p - oracle p| after the previous step
    for step in range(1, 4):
        g.copy_(workloads.device_stack((1, 1, n_total), "normal", w.grad_std, 3300 + step, "bf16", DEV).view(-1))
        for h in hps.values():
            h.step = step
        L.adamw_step_grouped(tensors, aws)
        torch.cuda.synchronize()
        gi = f64(g[idx_t])
        po_prev, m_prev = po, mref
        po, mref, vref = oadamw.adamw_update(po, gi, mref, vref, step, lr=a.lr, beta1=a.beta1, beta2=a.beta2,
                                             eps=a.eps, weight_decay=wd, param_dtype="bf16")
        got_p, got_m, got_v = f64(p[idx_t]), f64(mo[idx_t]), f64(vo[idx_t])
        # independent bf16 trajectories: a parameter difference carries into the next step scaled by the decay
        # factor (the update itself reads only m and v), and each step's two roundings add at most one ulp
        terms = np.abs(po_prev) + a.lr * (1 + 1e-3)
        carried = dp * (1.0 - a.lr * wd)
        off = np.abs(got_p - po)
        bound = carried + bf16_ulp(np.maximum(np.abs(got_p), np.abs(po))) * 1.0001 + 1e-6 * terms
        assert np.all(off <= bound), (step, int(np.sum(off > bound)))
        dp = off
        em = a.beta1 * em + 1e-6 * (a.beta1 * np.abs(m_prev) + np.abs(gi))
        ev = a.beta2 * ev + 1e-6 * (np.abs(vref) + gi * gi)
        assert np.all(np.abs(got_m - mref) <= em + 1e-30), step
        assert np.all(np.abs(got_v - vref) <= ev + 1e-30), step
    del p, g, mo, vo, tensors, specs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n", [2048, 4096, 8192])
def test_ns_sweep_large_sizes_sampled(L, n):
    K = workloads.NS_SWEEP_K
    x = workloads.ns_sweep_input(n, K, 0, device=DEV)
    out = torch.empty_like(x)
    ws = torch.zeros(L.muon_workspace_bytes(K, n, n), dtype=torch.uint8, device=DEV)
    L.ns_orthogonalize(x, out, [omuon.CLASSIC] * 5, 1e-7, ws)
    assert L.muon_check(ws) == L.MUON_OK
    picks = workloads.bucket_sample(K, 4, n) if n == 2048 else [workloads.bucket_sample(K, 4, n)[1]]
    for k in picks:
        ref = omuon.newton_schulz(f64(x[k]), [omuon.CLASSIC] * 5, 1e-7)
        assert rel_fro(f64(out[k]), ref) <= 2e-2, k
    del x, out, ws
    torch.cuda.empty_cache()
