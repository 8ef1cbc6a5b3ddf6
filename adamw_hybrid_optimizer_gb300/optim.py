"""HybridMuonAdamW: one optimizer for Muon (2-D hidden matrices) and AdamW (everything else).

The user-facing form of the pages' optimizer: ``Opt(param_groups).step()`` with groups tagged
``"kind": "muon"`` or ``"kind": "adamw"`` ("MuonAdamW vs DistMuonAdamW", sections "Usage
Examples" and "Do both optimizers support identical hyperparameters?"; "dtensor-muon 0.1.0",
sections "Usage" and "Key options"). Routing follows "Optimizers: AdamW, Muon and the distributed
optimizer" (Muon on hidden-layer matrices; embedding, output layer and vectors on AdamW): the
caller decides by the group's kind, and a Muon group must hold 2-D tensors only.

Muon matrices of one group are bucketed by shape (muon_plan_buckets); each bucket owns one fp32
(K, A, B) momentum stack, and all buckets of a group are updated by one muon_step_grouped call per
step. AdamW state is one fp32 exp_avg / exp_avg_sq pair per tensor and the group's step count. With
master_weights=True (bf16 parameters), each parameter also keeps an fp32 master copy ("master" in its
state) that takes the update; the parameter holds it rounded to bf16. All arithmetic runs in libmuon: the
AdamW tensors of all groups in one grouped pass, issued with the last Muon group by hybrid_step.
"""
from __future__ import annotations

from typing import Dict, List, Sequence

import torch

from . import libmuon as L

CLASSIC = (3.4445, -4.7750, 2.0315)

# master_weights=True (bf16 parameters only): an fp32 master copy per parameter takes the update and the
# parameter holds it rounded to bf16 ("Optimizers: AdamW, Muon and the distributed optimizer", section "The
# optimizer's memory budget")
# autotune=True: before the group's first step, the Newton-Schulz path of each bucket that can take the Gram-space
# chain, the poly step's pipeline shape and the chain's scheduling are measured on the group's own buckets and the
# fastest recorded (muon_autotune; "DMuon", section 2.4, shape-adaptive kernel autotuning)
MUON_DEFAULTS = dict(lr=0.02, momentum=0.95, weight_decay=0.01, nesterov=True, cautious_wd=False, scale_mode=0,
                     ns_steps=5, ns_coefficients=None, eps=1e-7, master_weights=False, autotune=False)
# is_adamw=False: Adam with L2 regularisation instead of decoupled decay ("dtensor-muon 0.1.0", "Key options")
ADAMW_DEFAULTS = dict(lr=3e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1, is_adamw=True, master_weights=False)


class _Bucket:
    def __init__(self, params: List[torch.Tensor], shape, device, master_weights: bool = False):
        self.params = params
        self.K = len(params)
        self.A, self.B = shape
        self.momentum = torch.zeros((self.K, self.A, self.B), dtype=torch.float32, device=device)
        self.param_ptrs = L.pointer_array(params, device)
        self.master = None
        self.master_ptrs = None
        if master_weights:
            if any(p.dtype != torch.bfloat16 for p in params):
                raise ValueError("master_weights needs bf16 parameters")
            self.master = torch.stack([p.detach().float() for p in params])
            self.master_ptrs = L.pointer_array([self.master[k] for k in range(self.K)], device)
        self.grad_ptrs = None
        self._grad_key = None

    def refresh_grads(self, device):
        grads = [p.grad for p in self.params]
        key = tuple(g.data_ptr() for g in grads)
        if key != self._grad_key:
            self.grad_ptrs = L.pointer_array(grads, device)
            self._grad_key = key
        return grads


class HybridMuonAdamW:
    def __init__(self, param_groups: Sequence[Dict]):
        self.param_groups = []
        self.state: Dict[torch.Tensor, Dict] = {}
        self._buckets: List[List[_Bucket]] = []
        ws_bytes = 0
        device = None
        for g in param_groups:
            kind = g.get("kind", "muon")
            defaults = MUON_DEFAULTS if kind == "muon" else ADAMW_DEFAULTS
            if kind not in ("muon", "adamw"):
                raise ValueError(f"unknown kind {kind!r}")
            group = dict(defaults)
            group.update(g)
            group["kind"] = kind
            group["params"] = list(g["params"])
            for p in group["params"]:
                if not p.is_cuda:
                    raise ValueError("HybridMuonAdamW runs on the GPU only: parameters must be CUDA tensors")
                device = p.device
            buckets = []
            if kind == "muon":
                if group["ns_coefficients"] is None:
                    group["ns_coefficients"] = [CLASSIC] * int(group["ns_steps"])
                group["ns_steps"] = len(group["ns_coefficients"])
                for p in group["params"]:
                    if p.dim() != 2:
                        raise ValueError("a Muon group holds 2-D matrices only; route vectors to an AdamW group")
                plan = L.muon_plan_buckets([tuple(p.shape) for p in group["params"]])
                members = [[] for _ in plan["bucket_K"]]
                for p, b in zip(group["params"], plan["bucket_id"]):
                    members[b].append(p)
                for shape, ps in zip(plan["bucket_shapes"], members):
                    bk = _Bucket(ps, shape, device, group["master_weights"])
                    buckets.append(bk)
                    for k, p in enumerate(ps):
                        self.state[p] = {"momentum_buffer": bk.momentum[k]}
                        if bk.master is not None:
                            self.state[p]["master"] = bk.master[k]
                shapes = (L.muon_bucket * len(buckets))(*[L.muon_bucket(None, None, None, bk.K, bk.A, bk.B, 0, 0)
                                                           for bk in buckets])
                ws_bytes = max(ws_bytes, L.muon_workspace_bytes_grouped(shapes) if buckets else 0)
            else:
                group["step"] = 0
                for p in group["params"]:
                    self.state[p] = {"exp_avg": torch.zeros(p.shape, dtype=torch.float32, device=p.device),
                                     "exp_avg_sq": torch.zeros(p.shape, dtype=torch.float32, device=p.device)}
                    if group["master_weights"]:
                        if p.dtype != torch.bfloat16:
                            raise ValueError("master_weights needs bf16 parameters")
                        self.state[p]["master"] = p.detach().float().clone()
            self.param_groups.append(group)
            self._buckets.append(buckets)
        # zero-filled: the control block's error word must start at zero
        self._ws = torch.zeros(max(ws_bytes, 256), dtype=torch.uint8, device=device) if device is not None else None
        self._adamw_ws = None   # the grouped AdamW pass's counters, sized on first use
        self._tuned = set()     # Muon groups whose autotune has run

    @torch.no_grad()
    def step(self):
        """One step of every group. The AdamW tensors of all groups go through one grouped pass, issued in one
        call (hybrid_step) with the last Muon group."""
        muon_calls = []
        adamw_specs = []
        for group, buckets in zip(self.param_groups, self._buckets):
            if group["kind"] == "muon":
                hp = L.make_muon_hparams(group["lr"], group["momentum"], group["weight_decay"], group["nesterov"],
                                         group["cautious_wd"], group["scale_mode"], group["ns_coefficients"],
                                         group["eps"])
                specs = []
                for bk in buckets:
                    if any(p.grad is None for p in bk.params):
                        continue
                    grads = bk.refresh_grads(self._ws.device)
                    pdt = L._dtype_code(bk.params[0])
                    gdt = L._dtype_code(grads[0])
                    for p, gr in zip(bk.params, grads):
                        if L._dtype_code(p) != pdt or L._dtype_code(gr) != gdt or not p.is_contiguous() \
                                or not gr.is_contiguous():
                            raise ValueError("a Muon bucket needs contiguous tensors of one dtype")
                    specs.append((bk.param_ptrs, bk.grad_ptrs, bk.momentum, bk.K, bk.A, bk.B, pdt, gdt, bk.master_ptrs))
                if specs:
                    arr = L.make_buckets(specs)
                    if group["autotune"] and id(group) not in self._tuned:
                        L.muon_autotune(arr, hp, self._ws)
                        self._tuned.add(id(group))
                    muon_calls.append((arr, hp))
            else:
                group["step"] += 1
                b1, b2 = group["betas"]
                hp = L.make_adamw_hparams(group["lr"], b1, b2, group["eps"], group["weight_decay"], group["step"],
                                          l2=not group["is_adamw"])
                for p in group["params"]:
                    if p.grad is None:
                        continue
                    if not p.is_contiguous() or not p.grad.is_contiguous():
                        raise ValueError("AdamW needs contiguous parameters and gradients")
                    st = self.state[p]
                    adamw_specs.append((p, p.grad, st["exp_avg"], st["exp_avg_sq"], hp)
                                       + ((st["master"],) if "master" in st else ()))
        if not adamw_specs:
            for bk, hp in muon_calls:
                L.muon_step_grouped(bk, hp, self._ws)
            return
        for bk, hp in muon_calls[:-1]:
            L.muon_step_grouped(bk, hp, self._ws)
        tensors = L.make_adamw_tensors(adamw_specs)
        need = L.adamw_workspace_bytes_grouped(len(adamw_specs))
        if self._adamw_ws is None or self._adamw_ws.numel() < need:
            self._adamw_ws = torch.zeros(need, dtype=torch.uint8, device=self._ws.device)
        if muon_calls:
            bk, hp = muon_calls[-1]
            L.hybrid_step(bk, hp, self._ws, tensors, self._adamw_ws)
        else:
            L.adamw_step_grouped(tensors, self._adamw_ws)

    def zero_grad(self, set_to_none: bool = True):
        for group in self.param_groups:
            for p in group["params"]:
                if p.grad is not None:
                    if set_to_none:
                        p.grad = None
                    else:
                        p.grad.zero_()

    def state_dict(self):
        flat = [p for g in self.param_groups for p in g["params"]]
        return {
            "state": {i: {k: v.clone() for k, v in self.state[p].items()} for i, p in enumerate(flat)},
            "steps": [g.get("step", 0) for g in self.param_groups],
        }

    def load_state_dict(self, sd):
        flat = [p for g in self.param_groups for p in g["params"]]
        for i, p in enumerate(flat):
            for k, v in sd["state"][i].items():
                self.state[p][k].copy_(v)
        for g, s in zip(self.param_groups, sd["steps"]):
            if g["kind"] == "adamw":
                g["step"] = s
