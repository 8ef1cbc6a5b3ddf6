"""GPU parity of ns_orthogonalize and muon_step_batched against the fp64 oracle, through the C ABI.

Inputs come from workloads (seeded); the oracle runs on the same rounded values and its own state
trajectory. Bar: relative Frobenius error <= 2e-2 for the orthogonalised output and for the
parameter change; momentum within 1e-6 of its terms' magnitude; bf16 parameters additionally allowed
their storage rounding (2^-8 of their norm).
"""
import numpy as np
import pytest
import torch

from oracle import muon as omuon
from oracle.bf16 import round_to
from tests.gpu_common import DEV, bf16_ulp, build_lib, f64, hp_struct, rel_fro, workspace
import workloads

pytestmark = pytest.mark.gpu

CLASSIC5 = [omuon.CLASSIC] * 5


@pytest.fixture(scope="module")
def L():
    return build_lib()


# ---------------------------------------------------------------------------------------- ns_orthogonalize

@pytest.mark.parametrize("K,A,B,xdt,odt", [
    (4, 64, 128, torch.float32, torch.float32),
    (4, 128, 64, torch.float32, torch.float32),       # tall: transpose-to-wide and back
    (3, 200, 72, torch.bfloat16, torch.float32),      # ragged tiles, tall
    (2, 72, 200, torch.bfloat16, torch.bfloat16),
    (2, 1, 40, torch.float32, torch.float32),         # one row
    (2, 40, 1, torch.float32, torch.float32),         # one column
    (2, 96, 96, torch.bfloat16, torch.float32),       # square: not transposed
    (3, 768, 3072, torch.bfloat16, torch.float32),
    # the one-CTA fused chain takes wide iterates up to 128 x 256; just past that, the grouped GEMMs
    (2, 128, 256, torch.bfloat16, torch.float32),
    (2, 256, 128, torch.float32, torch.bfloat16),
    (1, 16, 16, torch.float32, torch.float32),
    (2, 129, 256, torch.bfloat16, torch.float32),
    (2, 128, 257, torch.bfloat16, torch.float32),
])
def test_ns_orthogonalize_matches_oracle(L, K, A, B, xdt, odt):
    g = torch.Generator().manual_seed(K * 1000 + A + B)
    x = torch.randn((K, A, B), generator=g, dtype=torch.float64).to(xdt).to(DEV)
    out = torch.full((K, A, B), float("nan"), dtype=odt, device=DEV)
    ws = workspace(L, K, A, B)
    L.ns_orthogonalize(x, out, CLASSIC5, 1e-7, ws)
    assert L.muon_check(ws) == L.MUON_OK
    X = f64(x)
    got = f64(out)
    for k in range(K):
        ref = omuon.newton_schulz(X[k], CLASSIC5, 1e-7)
        assert rel_fro(got[k], ref) <= 2e-2, k


def test_ns_orthogonalize_transpose_symmetry(L):
    g = torch.Generator().manual_seed(9)
    x = torch.randn((3, 96, 160), generator=g).to(torch.bfloat16).to(DEV)
    xt = x.transpose(1, 2).contiguous()
    o = torch.empty((3, 96, 160), dtype=torch.float32, device=DEV)
    ot = torch.empty((3, 160, 96), dtype=torch.float32, device=DEV)
    ws = workspace(L, 3, 96, 160)
    L.ns_orthogonalize(x, o, CLASSIC5, 1e-7, ws)
    L.ns_orthogonalize(xt, ot, CLASSIC5, 1e-7, ws)
    assert L.muon_check(ws) == L.MUON_OK
    assert torch.equal(o, ot.transpose(1, 2))        # the same wide iterate, bit for bit


def test_ns_orthogonalize_zero_matrix(L):
    x = torch.zeros((2, 64, 128), dtype=torch.float32, device=DEV)
    out = torch.full((2, 64, 128), 7.0, dtype=torch.float32, device=DEV)
    ws = workspace(L, 2, 64, 128)
    L.ns_orthogonalize(x, out, CLASSIC5, 1e-7, ws)
    assert L.muon_check(ws) == L.MUON_OK
    assert torch.count_nonzero(out) == 0


@pytest.mark.parametrize("n", [512, 1024])
def test_ns_sweep_small_sizes_sampled(L, n):
    """Square bf16 stacks, K = 64, 5 classic steps; the oracle checks the first, last and one seeded matrix."""
    K = workloads.NS_SWEEP_K
    x = workloads.ns_sweep_input(n, K, 0).to(DEV)
    out = torch.empty((K, n, n), dtype=torch.bfloat16, device=DEV)
    ws = workspace(L, K, n, n)
    L.ns_orthogonalize(x, out, CLASSIC5, 1e-7, ws)
    assert L.muon_check(ws) == L.MUON_OK
    for k in workloads.bucket_sample(K, 4, n):
        ref = omuon.newton_schulz(f64(x[k]), CLASSIC5, 1e-7)
        assert rel_fro(f64(out[k]), ref) <= 2e-2


# ---------------------------------------------------------------------------------------- muon_step_batched

def _cautious_twin_update(L, params, mom, grads, K, A, B, hp, code):
    """The orthogonalised update u the GPU computes in a cautious step, read from a twin step without the
    cautious mask on copies of the same state: both steps compute u identically (same inputs, same kernels;
    the mask only changes the epilogue's decay), and without the mask p_new = p - lr*wd*p - lr*scale*u, so
    u = (p - lr*wd*p - p_new) / (lr*scale). Returns u per matrix (fp64) and the recovery error bound per
    element (half a storage ulp of p_new over lr*scale)."""
    import dataclasses
    twin_hp = dataclasses.replace(hp, cautious_wd=False)
    tp = [p.clone() for p in params]
    tm = mom.clone()
    tws = workspace(L, K, A, B)
    L.muon_step_batched(L.pointer_array(tp, DEV), code, L.pointer_array(grads, DEV), code, tm, K, A, B,
                        hp_struct(L, twin_hp), tws)
    assert L.muon_check(tws) == L.MUON_OK
    lr_scale = np.float64(np.float32(hp.lr * omuon.update_scale(A, B, hp.scale_mode)))
    lr_wd = np.float64(np.float32(np.float64(np.float32(hp.lr)) * np.float64(np.float32(hp.weight_decay))))
    us, du = [], []
    for k in range(K):
        p0, p1 = f64(params[k]), f64(tp[k])
        us.append((p0 - lr_wd * p0 - p1) / lr_scale)
        ulp = bf16_ulp(p1) if code == L.MUON_BF16 else np.abs(p1) * 2.0 ** -23 + 1e-45
        du.append((0.5 * ulp + 1e-7 * (np.abs(p0) + np.abs(p1))) / lr_scale)
    return us, du


def _run_bucket(L, w, shape, members, steps, sample=None, hp=None):
    """Runs muon_step_batched on one (K, A, B) bucket for `steps` steps and the oracle on `sample`."""
    hp = hp or w.muon_hp
    A, B = shape
    K = len(members)
    pdt = "f32" if w.muon_dtype == "f32" else "bf16"
    tdt = torch.float32 if pdt == "f32" else torch.bfloat16
    params = [workloads.muon_param_init(w, i).to(DEV) for i in members]
    p_orc = {k: f64(params[k]) for k in (sample or range(K))}
    m_orc = {k: np.zeros((A, B)) for k in p_orc}
    p_first = {k: v.copy() for k, v in p_orc.items()}
    mom = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
    ws = workspace(L, K, A, B)
    pptr = L.pointer_array(params, DEV)
    hps = hp_struct(L, hp)
    code = L.MUON_F32 if pdt == "f32" else L.MUON_BF16
    for step in range(1, steps + 1):
        grads = [workloads.muon_grad(w, step, i).to(DEV) for i in members]
        mom_before = {k: f64(mom[k]) for k in p_orc}
        m_prev_orc = {k: m_orc[k].copy() for k in p_orc}
        p_gpu_before = {k: f64(params[k]) for k in p_orc}
        if hp.cautious_wd:
            u_gpu, u_err = _cautious_twin_update(L, params, mom, grads, K, A, B, hp, code)
        L.muon_step_batched(pptr, code, L.pointer_array(grads, DEV), code, mom, K, A, B, hps, ws)
        assert L.muon_check(ws) == L.MUON_OK
        for k in p_orc:
            g = f64(grads[k])
            p_prev = p_orc[k]
            p_new, m_new, u = omuon.muon_update(p_prev, g, m_orc[k], lr=hp.lr, momentum=hp.momentum,
                                                weight_decay=hp.weight_decay, nesterov=hp.nesterov,
                                                cautious_wd=hp.cautious_wd, coeffs=hp.coeffs, eps=hp.eps,
                                                scale_mode=hp.scale_mode, param_dtype=pdt)
            p_orc[k], m_orc[k] = p_new, m_new
            expect = p_new
            if hp.cautious_wd:
                # the decay mask [u*p > 0] is a decision on floating-point values: where the oracle's u (or p)
                # is within the GPU's measured deviation from it of zero, the sign may differ and either
                # decision is correct; take the one the GPU took there. Everywhere else the mask is the oracle's.
                dev_u = np.abs(u_gpu[k] - u) + u_err[k]
                dev_p = np.abs(p_gpu_before[k] - p_prev)
                ambiguous = (np.abs(u) <= 3.0 * dev_u) | (np.abs(p_prev) <= dev_p)
                assert rel_fro(u_gpu[k], u) <= 2e-2, (step, k)
                scale = omuon.update_scale(A, B, hp.scale_mode)
                with_decay = round_to(p_prev - hp.lr * hp.weight_decay * p_prev - hp.lr * scale * u, pdt)
                without = round_to(p_prev - hp.lr * scale * u, pdt)
                got_now = f64(params[k])
                pick = np.where(np.abs(got_now - with_decay) <= np.abs(got_now - without), with_decay, without)
                expect = np.where(ambiguous, pick, p_new)
                share = float(np.mean(ambiguous))
                print(f"cautious mask: step {step} matrix {k}: {100 * share:.3f}% of elements within the measured "
                      f"deviation of a sign change")
                assert share < 0.05
            got_m = f64(mom[k])
            # one fp32 rounding per step (fma) on top of the deviation carried from the previous step, which
            # the recurrence scales by mu (the oracle's momentum is exact, the GPU's is rounded each step)
            terms = np.abs(hp.momentum * mom_before[k]) + np.abs(g)
            carried = hp.momentum * np.abs(mom_before[k] - m_prev_orc[k]) * (1 + 1e-6)
            assert np.all(np.abs(got_m - m_new) <= carried + 1e-6 * terms + 1e-30), (step, k)
            got_p = f64(params[k])
            moved = np.linalg.norm(p_new - p_first[k])
            bound = 2e-2 * moved + (2.0 ** -8 * np.linalg.norm(p_new) if pdt == "bf16" else 0.0)
            assert np.linalg.norm(got_p - expect) <= bound, (step, k, np.linalg.norm(got_p - expect), bound)
    return params


def test_tiny_set_three_steps(L):
    """4 x (64 x 128) fp32, Nesterov 0.95, lr 0.02, wd 0.01, classic quintic, 3 optimizer steps; every matrix."""
    w = workloads.workload("tiny")
    _run_bucket(L, w, (64, 128), list(range(4)), w.steps)


@pytest.mark.parametrize("variant", ["no_nesterov", "cautious_big_wd", "scale_mode_1", "tall", "tall_ragged",
                                     "tall_ragged_vec"])
def test_step_variants(L, variant):
    import dataclasses
    w = workloads.workload("tiny")
    hp = w.muon_hp
    shape = (64, 128)
    if variant == "no_nesterov":
        hp = dataclasses.replace(hp, nesterov=False)
    elif variant == "cautious_big_wd":
        # lr*wd = 0.1 makes the mask visible; one step, since a mask decided the other way on an ambiguous
        # element moves the independent trajectories apart by 10% of that element
        hp = dataclasses.replace(hp, cautious_wd=True, weight_decay=5.0)
        _run_bucket(L, w, shape, list(range(4)), 1, hp=hp)
        return
    elif variant == "scale_mode_1":
        hp = dataclasses.replace(hp, scale_mode=1)
    elif variant == "tall":
        w = dataclasses.replace(w, muon=tuple(workloads.MuonTensor(f"t{i}", (128, 64)) for i in range(4)))
        shape = (128, 64)
    elif variant.startswith("tall_ragged"):
        # momentum on a stack stored tall, its norm pass's 64 x 64 transposed tiles cut ragged on both sides:
        # 258 columns (not a multiple of 4: scalar loads) or 260 (vector loads, a 4-column last tile)
        shape = (333, 258) if variant == "tall_ragged" else (200, 260)
        w = dataclasses.replace(w, muon=tuple(workloads.MuonTensor(f"t{i}", shape) for i in range(3)))
        _run_bucket(L, w, shape, list(range(3)), 2, hp=hp)
        return
    _run_bucket(L, w, shape, list(range(4)), 3, hp=hp)


def test_zero_gradient_step_only_decays(L):
    K, A, B = 2, 64, 128
    p = torch.randn((K, A, B), device=DEV)
    p0 = p.clone()
    g = torch.zeros((K, A, B), device=DEV)
    mom = torch.zeros((K, A, B), device=DEV)
    ws = workspace(L, K, A, B)
    hp = L.make_muon_hparams(0.02, 0.95, 0.01)
    L.muon_step_batched(L.pointer_array([p[0], p[1]], DEV), L.MUON_F32, L.pointer_array([g[0], g[1]], DEV),
                        L.MUON_F32, mom, K, A, B, hp, ws)
    assert L.muon_check(ws) == L.MUON_OK
    lr_wd = np.float32(np.float64(np.float32(0.02)) * np.float64(np.float32(0.01)))
    expect = f64(p0) - np.float64(lr_wd) * f64(p0)
    assert np.max(np.abs(f64(p) - expect)) <= 1e-7 * np.max(np.abs(expect))


def test_gpt2_small_set_sampled(L):
    """GPT-2-small Muon set (4 buckets x 12, bf16 params/grads), full stacks on the GPU, the workload's 10
    steps with momentum carried, sampled oracle (first, last and one seeded matrix per bucket)."""
    w = workloads.workload("gpt2s")
    assert w.steps == 10
    from oracle.buckets import plan_buckets
    plan = plan_buckets(workloads.shape_list(w))
    for b, (shape, K) in enumerate(zip(plan["bucket_shapes"], plan["bucket_K"])):
        members = [i for i, bid in enumerate(plan["bucket_id"]) if bid == b]
        _run_bucket(L, w, shape, members, w.steps, sample=workloads.bucket_sample(K, w.cfg_id, b))


def test_aspect_polar_express_cautious_sampled(L):
    """K=16 of 256 x 16384 and K=16 of 16384 x 256, Student-t(3) gradients, 8 Polar Express steps, cautious WD."""
    w = workloads.workload("aspect")
    for b, (shape, members) in enumerate([((256, 16384), list(range(16))), ((16384, 256), list(range(16, 32)))]):
        _run_bucket(L, w, shape, members, 3, sample=workloads.bucket_sample(16, w.cfg_id, b))


@pytest.mark.parametrize("K,A,B", [(4, 256, 512), (3, 640, 256), (2, 1024, 1024)])
def test_ns_orthogonalize_scheduling_modes_agree(L, K, A, B):
    """The single-stack chain's launches wait per matrix on readiness counters (1) or on their whole
    predecessor (0): the tiles are computed the same way, so the outputs must agree bit for bit (the default
    rule is compared with the oracle above)."""
    gen = torch.Generator().manual_seed(A + B + K)
    x = torch.randn((K, A, B), generator=gen).to(torch.bfloat16).to(DEV)
    outs = []
    try:
        for mode in (1, 0):
            L.muon_debug_counter_deps(mode)
            ws = workspace(L, K, A, B)
            out = torch.empty((K, A, B), dtype=torch.float32, device=DEV)
            L.ns_orthogonalize(x, out, CLASSIC5, 1e-7, ws)
            torch.cuda.synchronize()
            assert L.muon_check(ws) == L.MUON_OK
            outs.append(out)
    finally:
        L.muon_debug_counter_deps(-1)
    assert torch.isfinite(outs[0]).all()
    assert torch.equal(outs[0], outs[1])
