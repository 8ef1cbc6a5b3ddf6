"""Benchmark of the hybrid Muon + AdamW optimizer step on GB300.

A step is one full optimizer step over the Llama-3-8B-shaped parameter set: four Muon buckets of bf16
matrices (32 layers x {q, o 4096x4096; k, v 1024x4096; gate, up 14336x4096 (transposed path);
down 4096x14336}, 224 matrices, 6,979,321,856 elements; fp32 momentum; Nesterov 0.95; 5 classic
Newton-Schulz steps) and AdamW over 1,050,939,392 bf16 elements (embedding and head 128256x4096 with
decay, 65 RMSNorm 4096-vectors without; fp32 moments). Inputs are synthetic (seeded N(0, 1e-3^2) params
and grads drawn on the device) and resident in HBM; one gradient set is reused by every step. Each step
touches well over 100 GB, far more than the 129 MB L2, so no separate flush. The GPT-2-small-shaped set
is timed too and reported under its own key.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Under torchrun with N > 1 every rank runs an independent replica
(the step has no cross-GPU exchange); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Muon step ms & NS TFLOP/s (frac of bf16 peak); AdamW GB/s (frac of HBM)"
WORKLOADS = {
    "llama8b": ("llama-3-8b-shaped parameter set: Muon 4 buckets bf16 (K=64 4096x4096, K=64 1024x4096, "
                "K=64 14336x4096 transposed path, K=32 4096x14336; 6,979,321,856 elements), fp32 momentum, "
                "Nesterov 0.95, 5 classic quintic NS steps; AdamW on 2x128256x4096 bf16 (wd 0.1) + 65x4096 "
                "RMSNorm bf16 (wd 0), fp32 moments"),
    "gpt2s": ("gpt2-small-shaped parameter set: Muon 4 buckets x K=12 bf16 (768x2304, 768x768, 768x3072, "
              "3072x768 transposed path), fp32 momentum, Nesterov 0.95, 5 classic quintic NS steps; AdamW on "
              "2x50304x768 bf16 (wd 0.1) + 24x768 LayerNorm bf16 (wd 0), fp32 moments"),
}
HEADLINE = "llama8b"
WORKLOAD = WORKLOADS[HEADLINE]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ------------------------------------------------------------------------------------------------ workload

class Workload:
    """Device buffers of one bench step: Muon bucket stacks and the AdamW tensors (views of one flat buffer per
    dtype), drawn on the device from seeded generators."""

    def __init__(self, L, device, name=HEADLINE):
        import torch
        import workloads
        self.L = L
        self.device = device
        w = workloads.workload(name)
        self.w = w
        self.name = name
        plan = L.muon_plan_buckets(workloads.shape_list(w))
        self.buckets = []
        for b, (shape, K) in enumerate(zip(plan["bucket_shapes"], plan["bucket_K"])):
            A, B = shape
            p = workloads.device_stack((K, A, B), "normal", w.param_std, 7000 + b, "bf16", device)
            g = workloads.device_stack((K, A, B), w.grad_dist, w.grad_std, 7100 + b, "bf16", device)
            mom = torch.zeros((K, A, B), dtype=torch.float32, device=device)
            self.buckets.append(dict(K=K, A=A, B=B, p=p, g=g, mom=mom,
                                     pptr=L.pointer_array([p[k] for k in range(K)], device),
                                     gptr=L.pointer_array([g[k] for k in range(K)], device)))
        self.bucket_array = L.make_buckets([self._spec(bk) for bk in self.buckets])
        self.ws = torch.zeros(L.muon_workspace_bytes_grouped(self.bucket_array), dtype=torch.uint8, device=device)
        h = w.muon_hp
        self.hp = L.make_muon_hparams(h.lr, h.momentum, h.weight_decay, h.nesterov, h.cautious_wd, h.scale_mode,
                                      h.coeffs, h.eps)
        # AdamW: the workload's tensors as views of one flat bf16 buffer, each with its own weight decay
        n = w.adamw_elems
        self.adamw_flat = dict(p=workloads.device_stack((1, 1, n), "normal", w.param_std, 7200, "bf16",
                                                        device).view(-1),
                               g=workloads.device_stack((1, 1, n), "normal", w.grad_std, 7201, "bf16",
                                                        device).view(-1),
                               m=torch.zeros(n, dtype=torch.float32, device=device),
                               v=torch.zeros(n, dtype=torch.float32, device=device))
        a = w.adamw_hp
        self.adamw_hps = {}
        specs, off = [], 0
        for t in w.adamw:
            hp = self.adamw_hps.setdefault(t.weight_decay,
                                           L.make_adamw_hparams(a.lr, a.beta1, a.beta2, a.eps, t.weight_decay, 1))
            sl = slice(off, off + t.numel)
            specs.append(tuple(self.adamw_flat[k][sl] for k in "pgmv") + (hp,))
            off += t.numel
        self.adamw_tensors = L.make_adamw_tensors(specs)
        self.adamw_ws = torch.zeros(L.adamw_workspace_bytes_grouped(len(specs)), dtype=torch.uint8, device=device)
        self.t = 0

    def _spec(self, bk):
        L = self.L
        return (bk["pptr"], bk["gptr"], bk["mom"], bk["K"], bk["A"], bk["B"], L.MUON_BF16, L.MUON_BF16)

    def step(self, stream=None):
        """One whole optimizer step through hybrid_step: the grouped Muon step, then the grouped AdamW pass."""
        self.begin_step()
        self.L.hybrid_step(self.bucket_array, self.hp, self.ws, self.adamw_tensors, self.adamw_ws, stream)

    # the two halves of hybrid_step as separate calls, for a caller that overlaps its own copies with them
    def begin_step(self):
        self.t += 1
        for h in self.adamw_hps.values():
            h.step = self.t

    def muon_part(self, stream=None, which=None):
        """which: None for every bucket, else an index into the pieces of split_pieces()."""
        arr = self.bucket_array if which is None else self.piece_arrays[which]
        self.L.muon_step_grouped(arr, self.hp, self.ws, stream)

    def split_pieces(self, max_bytes=1.5e9):
        """Cuts the Muon buckets along K into pieces of at most max_bytes of gradients (at least one matrix), so
        that a caller can start each piece's chain as soon as its gradients are in and copy its parameters out
        while the next one runs. A Muon piece computes longer than its copies take, the AdamW pass far shorter,
        so the order keeps the three streams (copy in, compute, copy out) busy with little waiting at either
        end: the smallest piece first, in two halves (the first compute waits for half of it only), the AdamW
        pass after the next piece (Muon chains on both sides hide its copies), the rest by size, and the
        largest piece last, cut into parts that halve down to one matrix (each part's compute covers the
        previous part's copy out, so what is left after the last compute is one matrix's copy). Cutting and
        ordering change no result: each matrix's chain is computed the same way in any launch. Returns
        (pieces, adamw_at): the (bucket, k0, k1) pieces in order, and the index in that order before which
        the AdamW pass runs."""
        L = self.L
        pieces = []
        for b, bk in enumerate(self.buckets):
            per = bk["A"] * bk["B"] * bk["g"].element_size()
            n = min(bk["K"], max(1, -(-bk["K"] * per // int(max_bytes))))   # equal parts, none above max_bytes
            cuts = [round(i * bk["K"] / n) for i in range(n + 1)]
            pieces += [(b, cuts[i], cuts[i + 1]) for i in range(n)]
        size = lambda pc: (pc[2] - pc[1]) * self.buckets[pc[0]]["A"] * self.buckets[pc[0]]["B"]
        pieces.sort(key=size)   # stable: equal pieces keep bucket order
        b, k0, k1 = pieces.pop(0)
        head = [(b, k0, (k0 + k1 + 1) // 2), (b, (k0 + k1 + 1) // 2, k1)] if k1 - k0 > 1 else [(b, k0, k1)]
        tail = []
        if pieces:
            b, k0, k1 = pieces.pop()
            while k1 - k0 > 1:
                k = k0 + (k1 - k0 + 1) // 2
                tail.append((b, k0, k))
                k0 = k
            tail.append((b, k0, k1))
        order = head + pieces + tail
        adamw_at = min(len(order), len(head) + 1)
        self.piece_arrays = []
        for b, k0, k1 in order:
            bk = self.buckets[b]
            self.piece_arrays.append(L.make_buckets([(
                L.pointer_array([bk["p"][k] for k in range(k0, k1)], self.device),
                L.pointer_array([bk["g"][k] for k in range(k0, k1)], self.device),
                bk["mom"][k0:k1], k1 - k0, bk["A"], bk["B"], L.MUON_BF16, L.MUON_BF16)]))
        return order, adamw_at

    def adamw_part(self, stream=None):
        self.L.adamw_step_grouped(self.adamw_tensors, self.adamw_ws, stream)

    # algorithmic work of one step, per kernel kind
    def work(self):
        ns = self.w.muon_hp.ns_steps
        flops = {"ns_gram": 0.0, "ns_poly": 0.0, "ns_apply": 0.0, "ns_final": 0.0}
        nominal = 0.0
        bytes_ = {"nesterov_norm": 0.0, "adamw": 0.0}
        for bk in self.buckets:
            K, m, n = bk["K"], min(bk["A"], bk["B"]), max(bk["A"], bk["B"])
            flops["ns_gram"] += ns * K * m * m * n            # one triangle of X X^T
            flops["ns_poly"] += ns * K * m * m * m            # one triangle of G G
            flops["ns_apply"] += (ns - 1) * K * 2 * m * m * n
            flops["ns_final"] += K * 2 * m * m * n
            nominal += ns * K * (4 * m * m * n + 2 * m ** 3)
            bytes_["nesterov_norm"] += K * m * n * (2 + 4 + 4 + 2)
        bytes_["adamw"] = self.w.adamw_elems * 22
        return flops, nominal, bytes_

    # host <-> device views for the end-to-end leg: (gradient, parameter) device tensors, per bucket, then AdamW
    def host_views(self):
        dev_g = [bk["g"] for bk in self.buckets] + [self.adamw_flat["g"]]
        dev_p = [bk["p"] for bk in self.buckets] + [self.adamw_flat["p"]]
        return dev_g, dev_p


# ------------------------------------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.skip = 0
        fd, self.path = tempfile.mkstemp(prefix="muon_bench_clocks_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "25"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        # the timed region starts only once the sampler is producing lines
        t0 = time.time()
        while time.time() - t0 < 10 and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)
        with open(self.path) as f:
            self.skip = sum(1 for _ in f)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, sm_max_default):
        if self.proc is None or not os.path.exists(self.path):
            if os.path.exists(self.path):
                os.remove(self.path)
            return {"sm_mhz": None, "sm_max_mhz": sm_max_default, "reasons": ["nvidia-smi unavailable"]}
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        # samples taken before the timed region started are dropped (unless nothing else came)
        if len(lines) > self.skip:
            lines = lines[self.skip:]
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxes) if maxes else sm_max_default,
                "samples": len(sms), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------------------ oracle timing

def oracle_sample_time(shapes_to_time, adamw_sample: int = 1 << 21):
    """Times the oracle (fp64 NumPy, as it stands) on a bounded sample of the headline step: one Muon update
    (momentum, Nesterov input, Newton-Schulz, decay and step) of one matrix of each bucket in shapes_to_time,
    and AdamW on adamw_sample elements. The full step's time is extrapolated: each bucket's Muon work by its
    nominal Newton-Schulz flops at the fp64 rate measured on the timed matrices, AdamW by element count.
    Returns (extrapolated ms per full step, sample description, seconds spent, matrices timed)."""
    import workloads
    from oracle import adamw as oadamw
    from oracle import muon as omuon
    from oracle.buckets import plan_buckets
    w = workloads.workload(HEADLINE)
    hp = w.muon_hp
    plan = plan_buckets(workloads.shape_list(w))
    t_start = time.perf_counter()

    def ns_flops(A, B):
        m, n = min(A, B), max(A, B)
        return hp.ns_steps * (4.0 * m * m * n + 2.0 * m ** 3)

    timed_flops = timed_s = 0.0
    parts = []
    rng = np.random.default_rng(17)
    for (A, B), K in zip(plan["bucket_shapes"], plan["bucket_K"]):
        if (A, B) not in shapes_to_time:
            continue
        p = rng.standard_normal((A, B)) * w.param_std
        g = rng.standard_normal((A, B)) * w.grad_std
        t0 = time.perf_counter()
        omuon.muon_update(p, g, np.zeros_like(p), lr=hp.lr, momentum=hp.momentum, weight_decay=hp.weight_decay,
                          nesterov=hp.nesterov, coeffs=hp.coeffs, eps=hp.eps, param_dtype="bf16")
        timed_s += time.perf_counter() - t0
        timed_flops += ns_flops(A, B)
        parts.append(f"1 of {K} {A}x{B}")
    rate = timed_flops / timed_s
    muon_ms = sum(K * ns_flops(A, B) for (A, B), K in zip(plan["bucket_shapes"], plan["bucket_K"])) / rate * 1e3
    p, g = rng.standard_normal((2, adamw_sample)) * 1e-3
    a = w.adamw_hp
    t0 = time.perf_counter()
    oadamw.adamw_update(p, g, np.zeros(adamw_sample), np.zeros(adamw_sample), 1, lr=a.lr, beta1=a.beta1,
                        beta2=a.beta2, eps=a.eps, weight_decay=0.1, param_dtype="bf16")
    adamw_ms = (time.perf_counter() - t0) * 1e3 * w.adamw_elems / adamw_sample
    desc = ("oracle (NumPy fp64) Muon update of " + ", ".join(parts) + f" matrices ({rate / 1e9:.1f} GFLOP/s "
            f"fp64 measured), AdamW on {adamw_sample} elements; the full step (224 matrices, "
            f"{w.adamw_elems} AdamW elements) extrapolated by Newton-Schulz flop count and element count")
    return muon_ms + adamw_ms, desc, time.perf_counter() - t_start, len(parts)


# ------------------------------------------------------------------------------------------------ arms

def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest replica's value (the job's time is the max over ranks)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def run_reference(args):
    """The reference arm: the oracle, timed as it stands on the host cores, each step a bounded sample of the
    headline step (one 1024x4096 Muon matrix and 2^21 AdamW elements) extrapolated to the full step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    times = []
    desc, timed = "", 0
    for i in range(args.warmup + args.steps):
        ms, desc, _, n = oracle_sample_time({(1024, 4096)})
        if i >= args.warmup:
            times.append(ms)
            timed += n
    value = float(np.mean(times))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "ms",
            "higher_is_better": False, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(value, 3), "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD},
            "extrapolated": True,
            "oracle_samples_timed": {"muon_matrices": timed, "adamw_elements": (1 << 21) * args.steps,
                                     "note": "each timed step is a sample of the full step, extrapolated; "
                                             "no full step was run"},
            "cpu_baseline": {"value": round(value, 3), "unit": "ms", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 3), "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _kernel_table(L, wl, steps, peaks):
    """Per-kernel device times of `steps` traced steps (an event pair around every launch)."""
    import torch
    L.muon_trace_enable(True)
    for _ in range(steps):
        wl.step()
    torch.cuda.synchronize()
    L.muon_trace_enable(False)
    per_kind = {}
    for kind, t in L.muon_trace_collect():
        d = per_kind.setdefault(kind, [0.0, 0])
        d[0] += t
        d[1] += 1
    flops, nominal, bytes_ = wl.work()
    tot = {k: v[0] / steps for k, v in per_kind.items()}          # ms per step per kind
    launches_per_step = {k: v[1] / steps for k, v in per_kind.items()}
    kernels = {}
    for k, t in tot.items():
        entry = {"ms_per_step": round(t, 4), "launches_per_step": launches_per_step[k],
                 "avg_launch_us": round(1e3 * t / launches_per_step[k], 2)}
        if k in flops:
            tf = flops[k] / (t * 1e-3) / 1e12
            entry.update({"tflops": round(tf, 1), "frac_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                          "frac_bf16_sustained": round(tf / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]),
                                                      4)})
        if k in bytes_:
            gbs = bytes_[k] / (t * 1e-3) / 1e9
            entry.update({"gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)})
        kernels[k] = entry
    return tot, kernels, flops, nominal, bytes_


def _timed_steps(wl, steps, stream):
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        wl.step()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def _run_e2e(wl, args, stream, world, device, barrier):
    """The step through the C ABI with host buffers: every step, the gradients go in from pinned host memory
    and the updated parameters come back out, inside the timed region. The copies overlap the compute: the
    step runs as several calls on the compute stream, each started as soon as its inputs are in (the Muon
    chains of the pieces of split_pieces() with the AdamW pass among them, in the order it gives); inputs go in
    on one copy stream in that order, and each call's parameters come out on a second copy stream once it is
    done. The host issues the calls and copies interleaved, each copy after the call it should overlap."""
    import torch
    dev_g, dev_p = wl.host_views()
    h2d = sum(t.numel() * t.element_size() for t in dev_g)
    d2h = sum(t.numel() * t.element_size() for t in dev_p)
    # every local replica pins its own host buffers: stay within half of the host's memory
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    try:
        host_bytes = os.sysconf("SC_PAGE_SIZE") * os.sysconf("SC_PHYS_PAGES")
    except (ValueError, OSError, AttributeError):
        host_bytes = 0
    if host_bytes and (h2d + d2h) * local_world > host_bytes // 2:
        return {"value": None, "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "skipped": f"{local_world} replicas would pin {(h2d + d2h) * local_world / 1e9:.0f} GB of "
                           f"{host_bytes / 1e9:.0f} GB host memory"}
    host_g = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_g]
    host_p = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_p]
    for hg, dg in zip(host_g, dev_g):
        hg.copy_(dg)
    torch.cuda.synchronize()
    # the pinned-copy bandwidth of this machine, each way, on the largest buffer (the floor of the end-to-end step)
    big = max(range(len(dev_g)), key=lambda i: dev_g[i].numel())
    nbytes = dev_g[big].numel() * dev_g[big].element_size()
    c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    c0.record()
    dev_g[big].copy_(host_g[big], non_blocking=True)
    c1.record()
    host_p[big].copy_(dev_p[big], non_blocking=True)
    c2.record()
    torch.cuda.synchronize()
    h2d_gbs = nbytes / (c0.elapsed_time(c1) * 1e-3) / 1e9
    d2h_gbs = nbytes / (c1.elapsed_time(c2) * 1e-3) / 1e9
    e2e_steps = max(3, args.steps // 4)
    nb = len(wl.buckets)
    # (tensor index, k0, k1) slices to copy, and the call, per piece; AdamW's flat tensors are index nb
    order, adamw_at = wl.split_pieces()
    pieces = [([(b, k0, k1)], lambda j=j: wl.muon_part(stream, j)) for j, (b, k0, k1) in enumerate(order)]
    pieces.insert(adamw_at, ([(nb, 0, None)], lambda: wl.adamw_part(stream)))
    copy_in, copy_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in pieces]
    ev_done = [torch.cuda.Event() for _ in pieces]

    def put(j):   # call j's gradients in, on the input copy stream
        with torch.cuda.stream(copy_in):
            for i, k0, k1 in pieces[j][0]:
                dev_g[i][k0:k1].copy_(host_g[i][k0:k1], non_blocking=True)
            ev_in[j].record(copy_in)

    def get(j):   # call j's parameters out, on the output copy stream, once the call is done
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(ev_done[j])
            for i, k0, k1 in pieces[j][0]:
                host_p[i][k0:k1].copy_(dev_p[i][k0:k1], non_blocking=True)

    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        wl.begin_step()
        # issued in pipeline order: a host whose copy calls return only once the data has moved (as on some
        # boxes) still has call j queued on the GPU while it copies call j + 1's inputs and call j - 1's
        # outputs; where copies are asynchronous the order changes nothing
        put(0)
        for j, (_, run) in enumerate(pieces):
            stream.wait_event(ev_in[j])
            run()
            ev_done[j].record(stream)
            if j + 1 < len(pieces):
                put(j + 1)
            if j > 0:
                get(j - 1)
        get(len(pieces) - 1)
        copy_out.synchronize()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(1e3 * (time.perf_counter() - t0) / e2e_steps, world, device)
    barrier()
    return {"value": round(e2e_ms, 3), "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": e2e_steps, "pinned_copy_gbs": {"h2d": round(h2d_gbs, 1), "d2h": round(d2h_gbs, 1)}}


def _run_gpt2s(L, device, args, stream, peaks):
    """The GPT-2-small-shaped set's step, device time only, with its per-kernel table."""
    import torch
    small = Workload(L, device, "gpt2s")
    L.muon_autotune(small.bucket_array, small.hp, small.ws)
    for _ in range(max(3, args.warmup)):
        small.step()
    torch.cuda.synchronize()
    small_ms = _timed_steps(small, max(50, args.steps), stream)
    s_tot, s_kernels, _, s_nominal, s_bytes = _kernel_table(L, small, 3, peaks)
    s_ns = sum(s_tot.get(k, 0.0) for k in ("ns_gram", "ns_poly", "ns_apply", "ns_final"))
    s_adamw = s_tot.get("adamw", 0.0)
    if L.muon_check(small.ws) != L.MUON_OK:
        raise RuntimeError("a device-side wait ran out during the GPT-2-small steps")
    out = {"workload": WORKLOADS["gpt2s"], "ms_per_step": round(small_ms, 4), "ns_ms": round(s_ns, 4),
           "ns_frac_bf16_peak_nominal": round(s_nominal / (s_ns * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)
           if s_ns else None,
           "adamw_gbs": round(s_bytes["adamw"] / (s_adamw * 1e-3) / 1e9, 1) if s_adamw else None,
           "kernels": s_kernels}
    del small
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device(f"cuda:{local}")
    torch.cuda.set_device(device)
    import __graft_entry__
    __graft_entry__.build()
    from adamw_hybrid_optimizer_gb300 import libmuon as L

    peaks, peak_src = load_peaks()
    peak_tf = peaks["bf16_tflops"]
    peak_bw = peaks["hbm_gbs"]
    wl = Workload(L, device, HEADLINE)
    stream = torch.cuda.current_stream(device)
    # initialisation, outside every timed region: the poly step's pipeline shape measured on these buckets
    if not args.no_autotune:
        L.muon_autotune(wl.bucket_array, wl.hp, wl.ws)
    ms_ = sorted({min(bk["A"], bk["B"]) for bk in wl.buckets})
    poly_shape = {m: {0: "4+5", 1: "5+3", 2: "6+2"}.get(L.muon_autotune_poly_shape(m), "rule") for m in ms_}
    sched = {0: "launch order", 1: "per-matrix counters", 2: "per piece"}.get(
        L.muon_autotune_scheduling(wl.bucket_array), "rule")

    def barrier():
        if world > 1:
            dist.barrier()

    # warm-up
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    if L.muon_check(wl.ws) != L.MUON_OK:
        raise RuntimeError("a device-side wait ran out during warm-up")

    # timed region: device time of K steps
    barrier()
    torch.cuda.synchronize()
    launches0 = L.muon_launch_count()
    with ClockSampler(local) as clocks:
        ms = _timed_steps(wl, args.steps, stream)
    barrier()
    launches = L.muon_launch_count() - launches0
    ms = max_over_ranks(ms, world, device)
    clk = clocks.summary(peaks.get("sm_max_mhz"))

    # traced pass: per-kernel durations from events around each launch (same stream)
    trace_steps = max(1, min(args.steps, 3))
    tot, kernels, flops, nominal, bytes_ = _kernel_table(L, wl, trace_steps, peaks)
    # the dominant kernel among those with an algorithmic work model (the GEMMs, the two bandwidth passes)
    modelled = [k for k in tot if k in flops or k in bytes_]
    dominant = max(modelled, key=tot.get)
    ns_ms = sum(tot.get(k, 0.0) for k in ("ns_gram", "ns_poly", "ns_apply", "ns_final"))
    if dominant in flops:
        # the traced pass runs whole steps back to back (a second or more of tensor-core work under the power
        # cap), so the kernel's denominator is the sustained bf16 figure; the burst fraction is given beside it
        peak_sus = peaks.get("bf16_tflops_sustained", peak_tf)
        ach = flops[dominant] / (tot[dominant] * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dominant, "achieved": round(ach, 2), "peak": peak_sus,
                "unit": "TFLOP/s", "frac": round(ach / peak_sus, 4), "traffic": None,
                "peak_source": f"{peak_src} bf16 sustained (timed inside steps run back to back)",
                "frac_of_burst_peak": round(ach / peak_tf, 4)}
    else:
        ach = bytes_[dominant] / (tot[dominant] * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1), "peak": peak_bw, "unit": "GB/s",
                "frac": round(ach / peak_bw, 4), "traffic": None, "peak_source": f"{peak_src} copy"}
    traffic = _traffic_from_profiles(HEADLINE, dominant)
    if traffic is not None:
        roof["traffic"] = traffic

    # end to end through the C ABI with host buffers: gradients in from pinned host memory, updated
    # parameters back out, every step, inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = _run_e2e(wl, args, stream, world, device, barrier)
    if L.muon_check(wl.ws) != L.MUON_OK:
        raise RuntimeError("a device-side wait ran out during the timed steps")
    adamw_ms = tot.get("adamw", 0.0)
    head_cfg = {"muon_matrices": sum(bk["K"] for bk in wl.buckets), "adamw_elems": wl.w.adamw_elems}
    del wl
    torch.cuda.empty_cache()

    # the GPT-2-small-shaped set, device time only (reported under its own key)
    gpt2s = None
    if not args.no_gpt2s:
        gpt2s = _run_gpt2s(L, device, args, stream, peaks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cms, desc, _, n = oracle_sample_time({(1024, 4096), (4096, 4096)})
        cpu = {"value": round(cms, 1), "unit": "ms", "cores": os.cpu_count(), "kind": "oracle", "sample": desc,
               "extrapolated": True}

    if rank == 0:
        sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
        line = {
            "metric": METRIC, "value": round(ms, 4), "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": dict({"workload": WORKLOAD, "parallelism": "replicas" if world > 1 else "single",
                            "l2": "inputs larger than L2: >100 GB touched per step, no separate flush",
                            "poly_pipeline": {str(m): f"{v} stages+slots" for m, v in poly_shape.items()},
                            "chain_scheduling": f"{sched} (measured at init)"},
                           **head_cfg),
            "ms_at_sm_max_clock": round(ms * sm / smax, 4) if sm and smax else None,
            "muon_ms": round(sum(tot.get(k, 0.0) for k in tot if k != "adamw"), 4),
            "ns_ms": round(ns_ms, 4),
            "ns_tflops_nominal": round(nominal / (ns_ms * 1e-3) / 1e12, 1) if ns_ms > 0 else None,
            "ns_frac_bf16_peak_nominal": round(nominal / (ns_ms * 1e-3) / 1e12 / peak_tf, 4) if ns_ms > 0 else None,
            # the flops the kernels do for their results: one triangle of each symmetric product, all of the others
            "ns_tflops_useful": round(sum(flops.values()) / (ns_ms * 1e-3) / 1e12, 1) if ns_ms > 0 else None,
            "adamw_ms": round(adamw_ms, 4),
            "adamw_gbs": round(bytes_["adamw"] / (adamw_ms * 1e-3) / 1e9, 1) if adamw_ms > 0 else None,
            "adamw_frac_hbm": round(bytes_["adamw"] / (adamw_ms * 1e-3) / 1e9 / peak_bw, 4) if adamw_ms > 0 else None,
            "kernels": kernels,
            "roofline": roof,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
            "cpu_baseline": cpu,
            "gpt2s": gpt2s,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_profile_small(args):
    """One grouped Muon step, with no warm-up and no autotune, on a small case of a parameter set, so that an ncu
    capture can pick its launches by position: counter reset, norm pass, then per Newton-Schulz step the Gram,
    polynomial and apply (final at the last step) launches (Gram-space buckets: fp32 Gram, m x m chain, final);
    for the GPT-2-small set, the whole set and then its AdamW pass. The stacks are larger than L2, so DRAM figures
    mean something; prints the launches."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from adamw_hybrid_optimizer_gb300 import libmuon as L
    import workloads
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    name = args.profile_small
    if name == "gpt2s":
        # the whole set, small enough: its grouped Muon step, then its AdamW pass
        wl = Workload(L, dev, name)
        torch.cuda.synchronize()
        n0 = L.muon_launch_count()
        wl.begin_step()
        wl.muon_part()
        wl.adamw_part()
        torch.cuda.synchronize()
        if L.muon_check(wl.ws) != L.MUON_OK:
            raise RuntimeError("a device-side wait ran out")
        print(json.dumps({"profile_small": name, "matrices_per_bucket": "all",
                          "buckets": [f"{bk['A']}x{bk['B']}" for bk in wl.buckets], "adamw_elems": wl.w.adamw_elems,
                          "launches": L.muon_launch_count() - n0}), flush=True)
        return 0
    w = workloads.workload(name)
    per_bucket_K = {"llama8b": 2, "aspect": 8}[name]
    plan = L.muon_plan_buckets(workloads.shape_list(w))
    specs, keep = [], []
    for b, (A, B) in enumerate(plan["bucket_shapes"]):
        K = per_bucket_K
        p = workloads.device_stack((K, A, B), "normal", w.param_std, 9000 + b, "bf16", dev)
        g = workloads.device_stack((K, A, B), w.grad_dist, w.grad_std, 9100 + b, "bf16", dev)
        m = torch.zeros((K, A, B), dtype=torch.float32, device=dev)
        keep += [p, g, m]
        specs.append((L.pointer_array([p[k] for k in range(K)], dev), L.pointer_array([g[k] for k in range(K)], dev),
                      m, K, A, B, L.MUON_BF16, L.MUON_BF16))
    arr = L.make_buckets(specs)
    ws = torch.zeros(L.muon_workspace_bytes_grouped(arr), dtype=torch.uint8, device=dev)
    h = w.muon_hp
    hp = L.make_muon_hparams(h.lr, h.momentum, h.weight_decay, h.nesterov, h.cautious_wd, h.scale_mode, h.coeffs,
                             h.eps)
    torch.cuda.synchronize()
    n0 = L.muon_launch_count()
    L.muon_step_grouped(arr, hp, ws)
    torch.cuda.synchronize()
    if L.muon_check(ws) != L.MUON_OK:
        raise RuntimeError("a device-side wait ran out")
    print(json.dumps({"profile_small": name, "matrices_per_bucket": per_bucket_K,
                      "buckets": [f"{A}x{B}" for A, B in plan["bucket_shapes"]],
                      "launches": L.muon_launch_count() - n0}), flush=True)
    return 0


def _traffic_from_profiles(workload, kernel):
    """DRAM bytes per launch of `kernel` on `workload`, from the committed summary of an ncu capture of the
    current kernels ({workload: {kernel: bytes}}), if there is one."""
    path = os.path.join(ROOT, "profiles", "dram_traffic_per_launch.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    v = d.get(workload, {}).get(kernel) if isinstance(d.get(workload), dict) else None
    return v if isinstance(v, (int, float)) else None


def run_config_sweep(args):
    """The optimizer step on the other configurations (tiny, aspect-ratio Polar Express, Llama-3-8B-shaped):
    seeded device-side inputs, 2 warm-up steps, then the device time of a few steps per configuration. One
    JSON line each (not the bench line)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from adamw_hybrid_optimizer_gb300 import libmuon as L
    import workloads
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    sweep = [("tiny", 50, -1), ("aspect", 5, -1), ("aspect", 5, 0), ("llama8b", 3, -1)]
    for name, steps, gram_mode in sweep:
        L.muon_debug_gram_space(gram_mode)
        w = workloads.workload(name)
        plan = L.muon_plan_buckets(workloads.shape_list(w))
        dt = "f32" if w.muon_dtype == "f32" else "bf16"
        code = L.MUON_F32 if dt == "f32" else L.MUON_BF16
        specs, keep, nominal = [], [], 0.0
        for b, ((A, B), K) in enumerate(zip(plan["bucket_shapes"], plan["bucket_K"])):
            p = workloads.device_stack((K, A, B), "normal", w.param_std, 5000 + b, dt, dev)
            g = workloads.device_stack((K, A, B), w.grad_dist, w.grad_std, 5100 + b, dt, dev)
            mom = torch.zeros((K, A, B), dtype=torch.float32, device=dev)
            keep += [p, g, mom]
            specs.append((L.pointer_array([p[k] for k in range(K)], dev), L.pointer_array([g[k] for k in range(K)], dev),
                          mom, K, A, B, code, code))
            m, n = min(A, B), max(A, B)
            nominal += w.muon_hp.ns_steps * K * (4.0 * m * m * n + 2.0 * m ** 3)
        arr = L.make_buckets(specs)
        ws = torch.zeros(L.muon_workspace_bytes_grouped(arr), dtype=torch.uint8, device=dev)
        hp = L.make_muon_hparams(w.muon_hp.lr, w.muon_hp.momentum, w.muon_hp.weight_decay, w.muon_hp.nesterov,
                                 w.muon_hp.cautious_wd, w.muon_hp.scale_mode, w.muon_hp.coeffs, w.muon_hp.eps)
        n_adamw = sum(t.numel for t in w.adamw)
        adt = torch.float32 if w.adamw_dtype == "f32" else torch.bfloat16
        ap = torch.zeros(max(n_adamw, 1), dtype=adt, device=dev)
        ag = workloads.device_stack((1, 1, max(n_adamw, 1)), "normal", w.grad_std, 5200, w.adamw_dtype, dev).view(-1)
        am = torch.zeros(max(n_adamw, 1), dtype=torch.float32, device=dev)
        av = torch.zeros(max(n_adamw, 1), dtype=torch.float32, device=dev)
        a = w.adamw_hp
        # one grouped AdamW pass over the configuration's tensors (views of the flat buffers), each with its
        # own weight decay
        hps, aspecs, off = {}, [], 0
        for t in w.adamw:
            h = hps.setdefault(t.weight_decay, L.make_adamw_hparams(a.lr, a.beta1, a.beta2, a.eps, t.weight_decay, 1))
            sl = slice(off, off + t.numel)
            aspecs.append((ap[sl], ag[sl], am[sl], av[sl], h))
            off += t.numel
        atensors = L.make_adamw_tensors(aspecs) if aspecs else None
        aws = torch.zeros(max(L.adamw_workspace_bytes_grouped(len(aspecs)), 256), dtype=torch.uint8, device=dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        abytes = n_adamw * (28 if w.adamw_dtype == "f32" else 22)
        it = 0
        # the chain with its launches overlapping through per-matrix counters (the default), then with each
        # launch waiting for its whole predecessor; and a traced step for the per-kernel times
        for deps in (1, 0):
            L.muon_debug_counter_deps(deps)
            t_muon = t_adamw = 0.0
            sampler = ClockSampler(0)
            sampler.__enter__()
            for rep in range(2 + steps):
                it += 1
                for h in hps.values():
                    h.step = it
                ev[0].record()
                L.muon_step_grouped(arr, hp, ws)
                ev[1].record()
                if atensors is not None:
                    L.adamw_step_grouped(atensors, aws)
                ev[2].record()
                torch.cuda.synchronize()
                if rep >= 2:
                    t_muon += ev[0].elapsed_time(ev[1]) / steps
                    t_adamw += ev[1].elapsed_time(ev[2]) / steps
            sampler.__exit__(None, None, None)
            clk = sampler.summary(peaks.get("sm_max_mhz"))
            L.muon_trace_enable(True)
            L.muon_step_grouped(arr, hp, ws)
            torch.cuda.synchronize()
            L.muon_trace_enable(False)
            per_kind = {}
            for kind, t in L.muon_trace_collect():
                per_kind[kind] = round(per_kind.get(kind, 0.0) + t, 4)
            if L.muon_check(ws) != L.MUON_OK:
                raise RuntimeError(f"device wait ran out in the {name} configuration")
            t_adamw = max(t_adamw, 1e-9)
            print(json.dumps({"config": name, "counter_deps": deps, "muon_matrices": sum(plan["bucket_K"]),
                              "gram_space": {f"{A}x{B}": L.muon_gram_space_route(A, B, K)
                                             for (A, B), K in zip(plan["bucket_shapes"], plan["bucket_K"])},
                              "buckets": len(plan["bucket_K"]), "muon_ms": round(t_muon, 4),
                              "ns_tflops_nominal": round(nominal / (t_muon * 1e-3) / 1e12, 1),
                              "ns_frac_nominal": round(nominal / (t_muon * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                              "adamw_ms": round(t_adamw, 4), "adamw_elems": n_adamw,
                              "adamw_gbs": round(abytes / (t_adamw * 1e-3) / 1e9, 1),
                              "adamw_frac_hbm": round(abytes / (t_adamw * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                              "traced_ms_per_kind": per_kind, "peaks": f"{peak_src}",
                              "clocks": clk}), flush=True)
        L.muon_debug_counter_deps(-1)
        L.muon_debug_gram_space(-1)
        del specs, keep, arr, ws, ap, ag, am, av, aspecs, atensors
        torch.cuda.empty_cache()
    return 0


def run_small_sweep(args):
    """Small stacks (wide iterates up to 128 x 256), 5 classic steps: the fused one-CTA-per-matrix chain
    (ns_orthogonalize) against the same chain as separate tensor-core launches per step (the no-allocation
    entry point runs those). One JSON line per shape (not the bench line)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from adamw_hybrid_optimizer_gb300 import libmuon as L
    import workloads
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    coeffs = [workloads.CLASSIC_QUINTIC] * 5
    for (K, A, B) in [(4, 64, 128), (48, 128, 256), (256, 128, 256), (64, 96, 96)]:
        g = torch.Generator(device=dev)
        g.manual_seed(K * 100003 + A * 101 + B)
        x = torch.randn((K, A, B), generator=g, device=dev).to(torch.bfloat16)
        out = torch.empty_like(x)
        ws = torch.zeros(L.muon_workspace_bytes(K, A, B), dtype=torch.uint8, device=dev)
        times = {}
        for name, call in (("fused", lambda: L.ns_orthogonalize(x, out, coeffs, 1e-7, ws)),
                           ("separate", lambda: L.ns_orthogonalize_noalloc(x, out, coeffs, 1e-7))):
            for _ in range(5):
                call()
            torch.cuda.synchronize()
            reps = 200
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            for _ in range(reps):
                call()
            s1.record()
            torch.cuda.synchronize()
            times[name] = s0.elapsed_time(s1) / reps * 1e3
        if L.muon_check(ws) != L.MUON_OK:
            raise RuntimeError("device wait ran out in the small sweep")
        m, n = min(A, B), max(A, B)
        flops = 5 * K * (4.0 * m * m * n + 2.0 * m ** 3)
        print(json.dumps({"sweep": "ns_small", "K": K, "A": A, "B": B, "us_fused": round(times["fused"], 2),
                          "us_separate_launches": round(times["separate"], 2),
                          "speedup": round(times["separate"] / times["fused"], 2),
                          "tflops_nominal_fused": round(flops / (times["fused"] * 1e-6) / 1e12, 2),
                          "peak": f"{peaks['bf16_tflops']} TFLOP/s {peak_src} burst"}), flush=True)
    return 0


def run_ns_sweep(args):
    """Newton-Schulz sweep: K=64 square bf16 stacks, 5 classic steps, one JSON line per size (not the bench line)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from adamw_hybrid_optimizer_gb300 import libmuon as L
    import workloads
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    coeffs = [workloads.CLASSIC_QUINTIC] * 5
    K = workloads.NS_SWEEP_K
    sizes = [int(v) for v in args.sizes.split(",")] if args.sizes else list(workloads.NS_SWEEP_SIZES)
    L.muon_debug_counter_deps(args.counter_deps)
    for n in sizes:
        x = workloads.ns_sweep_input(n, K, 0, device="cuda:0")
        out = torch.empty_like(x)
        ws = torch.zeros(L.muon_workspace_bytes(K, n, n), dtype=torch.uint8, device=dev)
        reps = 3 if n >= 4096 else 10
        for _ in range(2):
            L.ns_orthogonalize(x, out, coeffs, 1e-7, ws)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record()
        for _ in range(reps):
            L.ns_orthogonalize(x, out, coeffs, 1e-7, ws)
        s1.record()
        torch.cuda.synchronize()
        ms = s0.elapsed_time(s1) / reps
        L.muon_trace_enable(True)
        L.ns_orthogonalize(x, out, coeffs, 1e-7, ws)
        torch.cuda.synchronize()
        L.muon_trace_enable(False)
        per = {}
        for kind, t in L.muon_trace_collect():
            per[kind] = per.get(kind, 0.0) + t
        if L.muon_check(ws) != L.MUON_OK:
            raise RuntimeError("device wait ran out in the sweep")
        nominal = 5 * K * 6.0 * n ** 3
        work = {"ns_gram": 5 * K * n ** 3, "ns_poly": 5 * K * n ** 3, "ns_apply": 4 * K * 2.0 * n ** 3,
                "ns_final": K * 2.0 * n ** 3}
        kern = {k: {"ms": round(per[k], 3), "tflops": round(work[k] / (per[k] * 1e-3) / 1e12, 1),
                    "frac": round(work[k] / (per[k] * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)}
                for k in work if k in per}
        mma_ms = sum(per.get(k, 0.0) for k in work)
        issued = sum(work.values())
        print(json.dumps({"sweep": "ns_orthogonalize", "n": n, "K": K, "ms": round(ms, 3),
                          "tflops_nominal": round(nominal / (ms * 1e-3) / 1e12, 1),
                          "frac_nominal": round(nominal / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                          "tflops_gemm_kernels": round(issued / (mma_ms * 1e-3) / 1e12, 1),
                          "frac_gemm_kernels": round(issued / (mma_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                          "kernels": kern, "peak": f"{peaks['bf16_tflops']} TFLOP/s {peak_src} burst"}), flush=True)
        del x, out, ws
        torch.cuda.empty_cache()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (host buffers)")
    ap.add_argument("--no-gpt2s", action="store_true", help="skip the GPT-2-small figures")
    ap.add_argument("--no-autotune", action="store_true",
                    help="skip the measured choices at initialisation (the rules decide; for launch-list captures)")
    ap.add_argument("--profile-small", default="",
                    help="one grouped Muon step (no warm-up, no autotune) of a small case of the named set, "
                         "for ncu captures: 'llama8b' (K=2 per bucket), 'aspect' (K=8 per bucket) or 'gpt2s' "
                         "(the whole set, then its AdamW pass)")
    ap.add_argument("--ns-sweep", action="store_true", help="Newton-Schulz size sweep instead of the bench line")
    ap.add_argument("--sizes", default="", help="comma-separated n for --ns-sweep")
    ap.add_argument("--small-sweep", action="store_true", help="fused small-matrix chain vs separate launches")
    ap.add_argument("--config-sweep", action="store_true", help="the step on the tiny, aspect and Llama-3-8B sets")
    ap.add_argument("--counter-deps", type=int, choices=[-1, 0, 1], default=-1,
                    help="--ns-sweep: chain launches wait per matrix (1), per grid (0), or as the library decides (-1)")
    args = ap.parse_args()
    if args.profile_small:
        return run_profile_small(args)
    if args.ns_sweep:
        return run_ns_sweep(args)
    if args.small_sweep:
        return run_small_sweep(args)
    if args.config_sweep:
        return run_config_sweep(args)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
