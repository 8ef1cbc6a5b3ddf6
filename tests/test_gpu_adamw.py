"""GPU parity of adamw_step against the fp64 oracle, through the C ABI: AdamW (decoupled decay) and, with
l2=True, Adam with L2 regularisation (the is_adamw=False option)."""
import numpy as np
import pytest
import torch

from oracle import adamw as oadamw
from tests.gpu_common import DEV, bf16_ulp, build_lib, f64
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return build_lib()


def _run(L, p, g_list, hp, wd, sample=None, pdt="f32", l2=False, master=False):
    """Runs len(g_list) AdamW steps on the GPU and the oracle; compares p, m, v on `sample` indices.
    master=True: p is an fp32 master copy updated by adamw_step_master, whose bf16 parameter must equal the
    master rounded to bf16 after every step."""
    oracle_step = oadamw.adam_l2_update if l2 else oadamw.adamw_update
    bf16_param = p.to(torch.bfloat16) if master else None
    n = p.numel()
    idx = np.arange(n) if sample is None else sample
    m = torch.zeros(n, dtype=torch.float32, device=DEV)
    v = torch.zeros(n, dtype=torch.float32, device=DEV)
    po, mo, vo = f64(p)[idx], np.zeros(len(idx)), np.zeros(len(idx))
    # error allowance carried from step to step: the moments' earlier rounding is scaled by beta each step
    # and a new 1e-6 of this step's terms is added (independent trajectories keep each other's error)
    em, ev = np.zeros(len(idx)), np.zeros(len(idx))
    dp = np.zeros(len(idx))   # |gpu p - oracle p| entering this step (bf16 trajectories may differ)
    for t, g in enumerate(g_list, start=1):
        if master:
            L.adamw_step_master(p, bf16_param, g, m, v, hp.lr, hp.beta1, hp.beta2, hp.eps, wd, t, l2=l2)
        else:
            L.adamw_step(p, g, m, v, hp.lr, hp.beta1, hp.beta2, hp.eps, wd, t, l2=l2)
        po_prev, mo_prev = po, mo
        po, mo, vo = oracle_step(po, f64(g)[idx], mo, vo, t, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2,
                                 eps=hp.eps, weight_decay=wd, param_dtype=pdt)
        torch.cuda.synchronize()
        got_p, got_m, got_v = f64(p)[idx], f64(m)[idx], f64(v)[idx]
        if master:
            assert torch.equal(bf16_param, p.to(torch.bfloat16)), t
        if pdt == "f32":
            scale = np.abs(po_prev) + hp.lr * (1 + 1e-3)
            assert np.max(np.abs(got_p - po) / scale) <= 1e-6, t
        else:
            # independent trajectories: each bf16 store may round the other way once. With decoupled decay a
            # parameter difference carries into the next step scaled by the decay factor (the update reads only
            # m and v) and the step's two roundings add at most one ulp; with L2 the moments see the difference
            # too, and the allowance stays one ulp per step taken so far
            terms = np.abs(po_prev) + hp.lr * (1 + 1e-3)
            one = bf16_ulp(np.maximum(np.abs(got_p), np.abs(po))) * 1.0001
            carried = dp * (1.0 - hp.lr * wd) + one if not l2 else t * bf16_ulp(po) * 1.0001
            assert np.all(np.abs(got_p - po) <= np.maximum(carried, t * bf16_ulp(po) * 1.0001) + 1e-6 * terms), t
        gi = f64(g)[idx]
        if l2:
            # the moments see g + wd*p: its fp32 rounding adds to their budget, and so does the difference of
            # the two parameter trajectories it starts from (wd * dp, scaled by 1 - beta into m and v)
            gi = np.abs(gi) + abs(wd) * np.abs(po_prev)
            em = em + (1 - hp.beta1) * abs(wd) * dp
            ev = ev + (1 - hp.beta2) * (2 * gi * abs(wd) * dp + (wd * dp) ** 2)
        em = hp.beta1 * em + 1e-6 * (hp.beta1 * np.abs(mo_prev) + np.abs(gi))
        ev = hp.beta2 * ev + 1e-6 * (np.abs(vo) + gi * gi)
        dp = np.abs(got_p - po)
        bound_m = em + 1e-30
        bad = np.abs(got_m - mo) > bound_m
        if bad.any():
            j = int(np.argmax(np.abs(got_m - mo) - bound_m))
            raise AssertionError(f"exp_avg step {t}: {bad.sum()} elements off; worst at sample {j} (index {idx[j]}): "
                                 f"gpu {got_m[j]!r} oracle {mo[j]!r} previous {mo_prev[j]!r} grad {gi[j]!r}")
        assert np.all(np.abs(got_v - vo) <= ev + 1e-30)


def test_tiny_vector_three_steps(L):
    w = workloads.workload("tiny")
    p = workloads.adamw_param_init(w, 0).to(DEV)
    gs = [workloads.adamw_grad(w, t, 0).to(DEV) for t in range(1, w.steps + 1)]
    _run(L, p, gs, w.adamw_hp, w.adamw[0].weight_decay)


@pytest.mark.parametrize("n,offset", [(8195, 0), (8195, 1), (7, 0), (1, 0), (100_003, 3)])
def test_ragged_and_misaligned(L, n, offset):
    g0 = torch.Generator().manual_seed(n + offset)
    base_p = torch.randn(n + offset, generator=g0).to(DEV)
    base_g = torch.randn(n + offset, generator=g0).to(DEV)
    p, g = base_p[offset:], base_g[offset:]
    hp = workloads.workload("tiny").adamw_hp
    _run(L, p, [g, g * 0.5, -g], hp, 0.1)


def test_mixed_dtypes(L):
    hp = workloads.workload("tiny").adamw_hp
    g0 = torch.Generator().manual_seed(3)
    p = torch.randn(4099, generator=g0).to(DEV)
    g = torch.randn(4099, generator=g0).to(torch.bfloat16).to(DEV)
    _run(L, p, [g, g], hp, 0.1)


def test_gpt2_embedding_bf16_full_size_sampled(L):
    """The 50304 x 768 bf16 embedding at full size, 3 steps; the oracle checks a seeded sample and the tail."""
    w = workloads.workload("gpt2s")
    p = workloads.adamw_param_init(w, 0).to(DEV)
    gs = [workloads.adamw_grad(w, t, 0).to(DEV) for t in range(1, 4)]
    n = p.numel()
    rng = np.random.default_rng(0)
    sample = np.unique(np.concatenate([rng.integers(0, n, 200_000), np.arange(n - 1000, n), np.arange(1000)]))
    _run(L, p, gs, w.adamw_hp, 0.1, sample=sample, pdt="bf16")


def test_layernorm_vectors_no_decay_bf16(L):
    w = workloads.workload("gpt2s")
    p = workloads.adamw_param_init(w, 5).to(DEV)
    gs = [workloads.adamw_grad(w, t, 5).to(DEV) for t in range(1, 4)]
    _run(L, p, gs, w.adamw_hp, 0.0, pdt="bf16")


@pytest.mark.parametrize("n,offset", [(8195, 0), (8195, 1)])
def test_adam_l2_fp32(L, n, offset):
    g0 = torch.Generator().manual_seed(10 + n + offset)
    base_p = torch.randn(n + offset, generator=g0).to(DEV)
    base_g = torch.randn(n + offset, generator=g0).to(DEV)
    p, g = base_p[offset:], base_g[offset:]
    hp = workloads.workload("tiny").adamw_hp
    _run(L, p, [g, g * 0.5, -g], hp, 0.1, l2=True)


def test_adam_l2_bf16_params(L):
    hp = workloads.workload("gpt2s").adamw_hp
    g0 = torch.Generator().manual_seed(11)
    p = (torch.randn(40_003, generator=g0) * 1e-3).to(torch.bfloat16).to(DEV)
    gs = [(torch.randn(40_003, generator=g0) * 1e-3).to(torch.bfloat16).to(DEV) for _ in range(3)]
    _run(L, p, gs, hp, 0.1, pdt="bf16", l2=True)


@pytest.mark.parametrize("n,offset", [(40_003, 0), (8195, 1)])
def test_adamw_fp32_master_weights(L, n, offset):
    """adamw_step_master: the fp32 master follows the oracle's fp32-parameter AdamW; the bf16 parameter is the
    master rounded to bf16 ("Optimizers: AdamW, Muon and the distributed optimizer", "The optimizer's memory
    budget": fp32 master weights beside bf16 weights)."""
    g0 = torch.Generator().manual_seed(20 + n)
    base_p = (torch.randn(n + offset, generator=g0) * 1e-3).to(DEV)
    base_g = (torch.randn(n + offset, generator=g0) * 1e-3).to(torch.bfloat16).to(DEV)
    p, g = base_p[offset:], base_g[offset:]
    hp = workloads.workload("gpt2s").adamw_hp
    _run(L, p, [g, g * 0.5, -g], hp, 0.1, master=True)


@pytest.mark.parametrize("grouped", [False, True])
def test_bf16_each_step_within_one_ulp(L, grouped):
    """bf16 parameters, step by step: at every step count t = 1..10 both sides start from the same seeded
    state (p and g bf16, m and v fp32 of the size they reach by step t, zero at t = 1), so the one-step
    bound holds without a trajectory allowance: the GPU's parameter within one bf16 ulp of the oracle's
    (both round a value that agrees to fp32 precision; they can land on the two sides of a rounding point),
    plus the fp32 rounding of the terms where the update cancels the decayed parameter; the moments within
    1e-6 of their terms. Through adamw_step, or through adamw_step_grouped with the vector cut into two
    tensors with and without decay."""
    hp = workloads.workload("gpt2s").adamw_hp
    n = 300_007
    cut = 123_457
    for t in range(1, 11):
        rng = np.random.default_rng(1000 + t)
        p0 = workloads.round_to(rng.standard_normal(n) * 1e-3, "bf16")
        g0 = workloads.round_to(rng.standard_normal(n) * 1e-3, "bf16")
        m0 = workloads.round_to(rng.standard_normal(n) * 1e-3 * (1 - hp.beta1 ** (t - 1)), "f32")
        v0 = workloads.round_to((rng.standard_normal(n) * 1e-3) ** 2 * (1 - hp.beta2 ** (t - 1)), "f32")
        p, g, m, v = p0.to(DEV), g0.to(DEV), m0.to(DEV), v0.to(DEV)
        wd = np.full(n, 0.1)
        if grouped:
            wd[cut:] = 0.0
            h1 = L.make_adamw_hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, 0.1, t)
            h2 = L.make_adamw_hparams(hp.lr, hp.beta1, hp.beta2, hp.eps, 0.0, t)
            tensors = L.make_adamw_tensors([(p[:cut], g[:cut], m[:cut], v[:cut], h1),
                                            (p[cut:], g[cut:], m[cut:], v[cut:], h2)])
            aws = torch.zeros(L.adamw_workspace_bytes_grouped(2), dtype=torch.uint8, device=DEV)
            L.adamw_step_grouped(tensors, aws)
        else:
            L.adamw_step(p, g, m, v, hp.lr, hp.beta1, hp.beta2, hp.eps, 0.1, t)
        torch.cuda.synchronize()
        P0, G0, M0, V0 = f64(p0), f64(g0), f64(m0), f64(v0)
        po, mo, vo = oadamw.adamw_update(P0, G0, M0, V0, t, lr=hp.lr, beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                                         weight_decay=wd, param_dtype="bf16")
        got_p, got_m, got_v = f64(p), f64(m), f64(v)
        terms = np.abs(P0) + hp.lr * (1 + 1e-3)
        off = np.abs(got_p - po)
        assert np.all(off <= bf16_ulp(po) * 1.0001 + 1e-6 * terms), (t, float(np.max(off / bf16_ulp(po))))
        assert np.all(np.abs(got_m - mo) <= 1e-6 * (hp.beta1 * np.abs(M0) + np.abs(G0)) + 1e-30), t
        assert np.all(np.abs(got_v - vo) <= 1e-6 * (np.abs(vo) + G0 * G0) + 1e-30), t
