"""The seeded input module: deterministic draws, stated shapes and dtypes."""
import numpy as np
import torch

import workloads


def test_draws_are_deterministic_and_distinct():
    w = workloads.workload("tiny")
    a = workloads.muon_grad(w, 1, 0)
    b = workloads.muon_grad(w, 1, 0)
    c = workloads.muon_grad(w, 2, 0)
    d = workloads.muon_grad(w, 1, 1)
    assert torch.equal(a, b) and not torch.equal(a, c) and not torch.equal(a, d)
    assert a.dtype == torch.float32 and a.shape == (64, 128)


def test_model_sets():
    g = workloads.workload("gpt2s")
    assert g.muon_elems == 84_934_656 and g.adamw_elems == 77_285_376
    ll = workloads.workload("llama8b")
    assert ll.muon_elems == 6_979_321_856 and ll.adamw_elems == 1_050_939_392
    a = workloads.workload("aspect")
    assert a.muon_hp.ns_steps == 8 and len(a.muon_hp.coeffs) == 8 and a.muon_hp.cautious_wd


def test_bf16_inputs_are_rounded_and_hyperparameters_are_float32():
    w = workloads.workload("gpt2s")
    x = workloads.muon_grad(w, 1, 3)
    assert x.dtype == torch.bfloat16
    assert abs(float(x.float().std()) - 1e-3) < 1e-4
    for v in (w.muon_hp.lr, w.muon_hp.momentum, w.adamw_hp.beta2, w.adamw_hp.eps):
        assert float(np.float32(v)) == v


def test_student_t_tails():
    w = workloads.workload("aspect")
    x = workloads.as_f64(workloads.muon_grad(w, 1, 0))
    kurt = np.mean(x ** 4) / np.mean(x ** 2) ** 2
    assert kurt > 6.0      # t(3) has infinite kurtosis; a normal would sit at 3
