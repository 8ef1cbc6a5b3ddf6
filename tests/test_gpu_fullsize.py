"""Full-size GPU runs checked against the oracle on sampled matrices.

* Llama-3-8B-shaped Muon set: 32 layers x {q, o 4096x4096; k, v 1024x4096; gate, up 14336x4096;
  down 4096x14336} bf16, fp32 momentum, one grouped step over all four buckets (the launch configuration
  of the bench's grouped call). Inputs are drawn on the device from seeded generators; the oracle checks
  one seeded matrix of each large bucket and the first, last and one seeded matrix of the 1024x4096 one.
* Newton-Schulz sweep sizes n = 2048, 4096, 8192 (K = 64 square bf16 stacks): the oracle checks sampled
  matrices (three at 2048, one at the larger sizes).
Bars as elsewhere: relative Frobenius error <= 2e-2 of the update / of the orthogonalised output.
"""
import numpy as np
import pytest
import torch

from oracle import muon as omuon
from oracle.buckets import plan_buckets
from tests.gpu_common import DEV, build_lib, f64, hp_struct, rel_fro
import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def L():
    return build_lib()


def test_llama8b_grouped_step_sampled(L):
    w = workloads.workload("llama8b")
    hp = w.muon_hp
    plan = plan_buckets(workloads.shape_list(w))
    buckets = []
    for b, ((A, B), K) in enumerate(zip(plan["bucket_shapes"], plan["bucket_K"])):
        p = workloads.device_stack((K, A, B), "normal", w.param_std, 3000 + b, "bf16", DEV)
        g = workloads.device_stack((K, A, B), "normal", w.grad_std, 3100 + b, "bf16", DEV)
        m = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
        if K > 32:
            sample = workloads.bucket_sample(K, w.cfg_id, b) if A * B <= 1024 * 4096 else \
                [workloads.bucket_sample(K, w.cfg_id, b)[1]]
        else:
            sample = [workloads.bucket_sample(K, w.cfg_id, b)[1]]
        before = {k: f64(p[k]) for k in sample}
        buckets.append((p, g, m, K, A, B, sample, before))
    specs = [(L.pointer_array([p[k] for k in range(K)], DEV), L.pointer_array([g[k] for k in range(K)], DEV), m, K, A,
              B, L.MUON_BF16, L.MUON_BF16) for p, g, m, K, A, B, _, _ in buckets]
    arr = L.make_buckets(specs)
    ws = torch.zeros(L.muon_workspace_bytes_grouped(arr), dtype=torch.uint8, device=DEV)
    L.muon_step_grouped(arr, hp_struct(L, hp), ws)
    assert L.muon_check(ws) == L.MUON_OK
    for p, g, m, K, A, B, sample, before in buckets:
        assert torch.isfinite(p.float()).all()
        for k in sample:
            gk = f64(g[k])
            ref, mref, _ = omuon.muon_update(before[k], gk, np.zeros_like(gk), lr=hp.lr, momentum=hp.momentum,
                                             weight_decay=hp.weight_decay, nesterov=hp.nesterov, coeffs=hp.coeffs,
                                             eps=hp.eps, param_dtype="bf16")
            got = f64(p[k])
            assert np.linalg.norm(got - ref) <= 2e-2 * np.linalg.norm(ref - before[k]) + 2 ** -8 * np.linalg.norm(ref), \
                (A, B, k)
            assert np.array_equal(f64(m[k]), mref)     # first step: M = G exactly
    del ws


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
