"""Seeded synthetic inputs for the hybrid Muon + AdamW optimizer step.

This module only *describes* workloads and *draws* their random inputs. It holds
none of the optimizer's arithmetic, so both the fp64 oracle (``oracle/``) and the
CUDA path (``adamw_hybrid_optimizer_gb300``) may take their inputs from here.

Every array is drawn from NumPy ``Generator(PCG64(SeedSequence([cfg, step, role,
index])))`` in float64, then rounded to its storage dtype (float32 or bfloat16,
round-to-nearest-even through ``torch``'s dtype conversion). The rounded values
are what both sides receive. The largest stacks (Llama-3-8B-shaped, 8192-wide
sweeps) are drawn on the device with a seeded ``torch.Generator`` instead, and
the few matrices the oracle checks are copied back to the host.

Shapes follow the parameter sets named for the optimizer's workloads:
  tiny      4 Muon matrices 64x128 fp32 + one 8192-element AdamW vector
  gpt2s     GPT-2-small: 12 x {768x2304, 768x768, 768x3072, 3072x768} + embedding/head/LayerNorms
  llama8b   Llama-3-8B: 32 x {q, o 4096x4096; k, v 1024x4096; gate, up 14336x4096; down 4096x14336}
  nssweep   K=64 square n x n stacks, n in {512, ..., 8192}, Newton-Schulz only
  aspect    K=16 of 256x16384 and K=16 of 16384x256, Student-t(3) gradients, Polar Express, cautious WD
"""
from __future__ import annotations

import dataclasses
import json
import os
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

# Role codes mixed into the seed so that params, grads and AdamW tensors never share a stream.
ROLE_MUON_PARAM = 0
ROLE_MUON_GRAD = 1
ROLE_ADAMW_PARAM = 2
ROLE_ADAMW_GRAD = 3
ROLE_NS_INPUT = 4
ROLE_SAMPLE = 5

CLASSIC_QUINTIC = (3.4445, -4.7750, 2.0315)

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "tests", "golden")


@dataclasses.dataclass(frozen=True)
class MuonHP:
    lr: float = 0.02
    momentum: float = 0.95
    weight_decay: float = 0.01
    nesterov: bool = True
    cautious_wd: bool = False
    ns_steps: int = 5
    coeffs: Tuple[Tuple[float, float, float], ...] = (CLASSIC_QUINTIC,) * 5
    eps: float = 1e-7
    scale_mode: int = 0  # 0: 0.2*sqrt(max(A,B)); 1: sqrt(max(1, A/B))


@dataclasses.dataclass(frozen=True)
class AdamWHP:
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1


@dataclasses.dataclass(frozen=True)
class MuonTensor:
    name: str
    shape: Tuple[int, int]


@dataclasses.dataclass(frozen=True)
class AdamWTensor:
    name: str
    numel: int
    weight_decay: float


@dataclasses.dataclass(frozen=True)
class Workload:
    cfg_id: int
    name: str
    muon: Tuple[MuonTensor, ...]
    adamw: Tuple[AdamWTensor, ...]
    muon_dtype: str          # storage dtype of Muon params and grads: "f32" | "bf16"
    adamw_dtype: str         # storage dtype of AdamW params and grads
    muon_hp: MuonHP
    adamw_hp: AdamWHP
    steps: int
    grad_dist: str = "normal"      # "normal" | "student_t3"
    grad_std: float = 1.0
    param_std: float = 1.0

    @property
    def muon_elems(self) -> int:
        return sum(t.shape[0] * t.shape[1] for t in self.muon)

    @property
    def adamw_elems(self) -> int:
        return sum(t.numel for t in self.adamw)


def _f32(x: float) -> float:
    """Hyperparameters are passed to the kernels as float32; both sides use that value."""
    return float(np.float32(x))


def _muon_hp(**kw) -> MuonHP:
    hp = MuonHP(**kw)
    return dataclasses.replace(
        hp, lr=_f32(hp.lr), momentum=_f32(hp.momentum), weight_decay=_f32(hp.weight_decay), eps=_f32(hp.eps),
        coeffs=tuple(tuple(_f32(c) for c in abc) for abc in hp.coeffs))


def _adamw_hp(**kw) -> AdamWHP:
    hp = AdamWHP(**kw)
    return dataclasses.replace(hp, lr=_f32(hp.lr), beta1=_f32(hp.beta1), beta2=_f32(hp.beta2), eps=_f32(hp.eps),
                               weight_decay=_f32(hp.weight_decay))


def polar_express_coeffs(steps: int = 8) -> Tuple[Tuple[float, float, float], ...]:
    """The per-step Polar Express table stored under tests/golden (written by oracle/polar_express.py)."""
    path = os.path.join(GOLDEN_DIR, f"polar_express_{steps}step.json")
    with open(path) as f:
        table = json.load(f)["coeffs"]
    return tuple(tuple(_f32(c) for c in abc) for abc in table)


def _gpt2_small() -> Workload:
    muon = []
    for layer in range(12):
        muon += [MuonTensor(f"h{layer}.attn.qkv", (768, 2304)), MuonTensor(f"h{layer}.attn.proj", (768, 768)),
                 MuonTensor(f"h{layer}.mlp.fc", (768, 3072)), MuonTensor(f"h{layer}.mlp.proj", (3072, 768))]
    adamw = [AdamWTensor("wte", 50304 * 768, 0.1), AdamWTensor("lm_head", 50304 * 768, 0.1)]
    adamw += [AdamWTensor(f"ln{i}", 768, 0.0) for i in range(24)]
    return Workload(2, "gpt2s", tuple(muon), tuple(adamw), "bf16", "bf16", _muon_hp(), _adamw_hp(), 10,
                    grad_std=1e-3, param_std=1e-3)


def _llama8b() -> Workload:
    muon = []
    for layer in range(32):
        muon += [MuonTensor(f"l{layer}.q", (4096, 4096)), MuonTensor(f"l{layer}.o", (4096, 4096)),
                 MuonTensor(f"l{layer}.k", (1024, 4096)), MuonTensor(f"l{layer}.v", (1024, 4096)),
                 MuonTensor(f"l{layer}.gate", (14336, 4096)), MuonTensor(f"l{layer}.up", (14336, 4096)),
                 MuonTensor(f"l{layer}.down", (4096, 14336))]
    adamw = [AdamWTensor("embed", 128256 * 4096, 0.1), AdamWTensor("head", 128256 * 4096, 0.1)]
    adamw += [AdamWTensor(f"rms{i}", 4096, 0.0) for i in range(65)]
    return Workload(3, "llama8b", tuple(muon), tuple(adamw), "bf16", "bf16", _muon_hp(), _adamw_hp(), 3,
                    grad_std=1e-3, param_std=1e-3)


def _tiny() -> Workload:
    muon = tuple(MuonTensor(f"w{i}", (64, 128)) for i in range(4))
    adamw = (AdamWTensor("vec", 8192, 0.1),)
    return Workload(1, "tiny", muon, adamw, "f32", "f32", _muon_hp(), _adamw_hp(), 3)


def _aspect() -> Workload:
    muon = tuple(MuonTensor(f"wide{i}", (256, 16384)) for i in range(16))
    muon += tuple(MuonTensor(f"tall{i}", (16384, 256)) for i in range(16))
    pe = polar_express_coeffs(8)
    return Workload(5, "aspect", muon, (), "bf16", "bf16",
                    _muon_hp(cautious_wd=True, nesterov=True, ns_steps=8, coeffs=pe), _adamw_hp(), 3,
                    grad_dist="student_t3", grad_std=1.0, param_std=1e-3)


NS_SWEEP_SIZES = (512, 1024, 2048, 4096, 8192)
NS_SWEEP_K = 64


def workload(name: str) -> Workload:
    table = {"tiny": _tiny, "gpt2s": _gpt2_small, "llama8b": _llama8b, "aspect": _aspect}
    return table[name]()


# ----------------------------------------------------------------------------------------------------------------
# Drawing inputs
# ----------------------------------------------------------------------------------------------------------------

def rng(cfg_id: int, step: int, role: int, index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([cfg_id, step, role, index])))


def draw(shape: Sequence[int], dist: str, std: float, gen: np.random.Generator) -> np.ndarray:
    if dist == "normal":
        return gen.standard_normal(tuple(shape)) * std
    if dist == "student_t3":
        return gen.standard_t(3, size=tuple(shape)) * std
    raise ValueError(dist)


def round_to(x: np.ndarray, dtype: str):
    """Round float64 values to the storage dtype. Returns a torch CPU tensor of that dtype."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    return t.to(torch.float32 if dtype == "f32" else torch.bfloat16)


def as_f64(t) -> np.ndarray:
    import torch
    return t.detach().to("cpu", torch.float64).numpy()


def muon_param_init(w: Workload, idx: int):
    t = w.muon[idx]
    return round_to(draw(t.shape, "normal", w.param_std, rng(w.cfg_id, 0, ROLE_MUON_PARAM, idx)), w.muon_dtype)


def muon_grad(w: Workload, step: int, idx: int):
    t = w.muon[idx]
    return round_to(draw(t.shape, w.grad_dist, w.grad_std, rng(w.cfg_id, step, ROLE_MUON_GRAD, idx)), w.muon_dtype)


def adamw_param_init(w: Workload, idx: int):
    t = w.adamw[idx]
    return round_to(draw((t.numel,), "normal", w.param_std, rng(w.cfg_id, 0, ROLE_ADAMW_PARAM, idx)), w.adamw_dtype)


def adamw_grad(w: Workload, step: int, idx: int):
    t = w.adamw[idx]
    return round_to(draw((t.numel,), "normal", w.grad_std, rng(w.cfg_id, step, ROLE_ADAMW_GRAD, idx)), w.adamw_dtype)


def ns_sweep_input(n: int, K: int, index: int, device: Optional[str] = None):
    """K x n x n bf16 stack, N(0,1). Host NumPy draw for small n, seeded torch draw on ``device`` otherwise."""
    import torch
    if device is None:
        x = np.stack([draw((n, n), "normal", 1.0, rng(4, n, ROLE_NS_INPUT, index * 4096 + k)) for k in range(K)])
        return round_to(x, "bf16")
    g = torch.Generator(device=device)
    g.manual_seed(4_000_000 + 1000 * n + index)
    return torch.randn((K, n, n), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def device_stack(shape: Tuple[int, int, int], dist: str, std: float, seed: int, dtype: str, device: str):
    """Seeded device draw for stacks too large for a host NumPy draw (Llama-3-8B-shaped buckets)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if dist == "normal":
        x = torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std
    elif dist == "student_t3":
        # t(3) = Z / sqrt(chi2_3 / 3); chi2_3 drawn as a sum of three squared normals.
        z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        c = torch.zeros(shape, device=device, dtype=torch.float32)
        for _ in range(3):
            c += torch.randn(shape, generator=g, device=device, dtype=torch.float32) ** 2
        x = z / torch.sqrt(c / 3) * std
    else:
        raise ValueError(dist)
    return x.to(torch.float32 if dtype == "f32" else torch.bfloat16)


def bucket_sample(K: int, cfg_id: int, key: int) -> List[int]:
    """The matrices of a K-stack that a sampled parity check compares: first, last and one seeded pick."""
    pick = int(rng(cfg_id, 0, ROLE_SAMPLE, key).integers(0, K))
    return sorted({0, K - 1, pick})


def shape_list(w: Workload) -> List[Tuple[int, int]]:
    return [t.shape for t in w.muon]


__all__ = [n for n in dir() if not n.startswith("_")]
