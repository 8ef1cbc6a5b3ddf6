"""Helpers shared by the GPU tests: device setup, tolerance checks, oracle runners.

Tolerances (derived from the arithmetic, stated once here):
  * a bf16 result rounded from an fp32 value is within 2^-8 of it, relative (8 significant bits, round to
    nearest: unit roundoff 2^-8);
  * an fp32 sum of n products has error at most ~ sqrt(n) * 2^-24 * sum|a_k b_k| in practice; we allow
    1e-5 * sum|a_k b_k|, above that for n <= 16384;
  * Newton-Schulz output and the Muon update: relative Frobenius error <= 2e-2 (the bf16 target);
  * fp32 elementwise results (momentum, AdamW with fp32 params): error <= 1e-6 of the magnitude of the
    terms they are computed from (a difference of rounded terms has no relative bound in its result);
  * AdamW with bf16 params: within one bf16 ulp of the oracle's value per step (independent trajectories
    may round a value the other way once per step), plus the fp32 rounding of the terms where they cancel.
"""
import numpy as np
import torch

import workloads

DEV = torch.device("cuda:0")


def build_lib():
    import __graft_entry__
    __graft_entry__.build()
    from adamw_hybrid_optimizer_gb300 import libmuon as L
    L.lib()
    torch.cuda.set_device(DEV)
    return L


def f64(t) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rel_fro(got, ref) -> float:
    d = np.linalg.norm(np.asarray(got) - np.asarray(ref))
    n = np.linalg.norm(np.asarray(ref))
    return float(d / n) if n > 0 else float(d)


def bf16_ulp(x) -> np.ndarray:
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(x == 0, 1.0, x))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def workspace(L, K, A, B):
    return torch.zeros(L.muon_workspace_bytes(K, A, B), dtype=torch.uint8, device=DEV)


def ctrl_ws():
    return torch.zeros(4096, dtype=torch.uint8, device=DEV)


def hp_struct(L, hp: workloads.MuonHP):
    return L.make_muon_hparams(hp.lr, hp.momentum, hp.weight_decay, hp.nesterov, hp.cautious_wd, hp.scale_mode,
                               hp.coeffs, hp.eps)
