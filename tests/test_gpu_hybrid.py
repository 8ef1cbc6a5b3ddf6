"""adamw_step_grouped and hybrid_step, through the C ABI.

adamw_step_grouped gives every tensor the per-element arithmetic of adamw_step / adamw_step_master, whatever
warp or launch takes which chunk, so its results must equal one adamw_step call per tensor bit for bit
(those are compared with the oracle in test_gpu_adamw); one case is also compared with the oracle directly.
hybrid_step is muon_step_grouped followed by adamw_step_grouped in one call, so its results must equal those
two calls bit for bit. Covered: every
parameter/gradient dtype pair, master weights, Adam with L2, per-tensor hyperparameters, ragged lengths,
misaligned tensors (scalar path), more than 96 tensors (two passes), the Muon-only and AdamW-only forms,
and the GPT-2-small-shaped step at full size.
"""
import numpy as np
import pytest
import torch

from oracle import adamw as oadamw
from tests.gpu_common import DEV, build_lib, f64, hp_struct
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return build_lib()


def _tensor_set(seed, specs):
    """specs: (n, pdt, gdt, master, offset); returns device tensors (p, g, m, v, master) per spec. offset > 0
    starts the tensors that many elements into a larger buffer, so that they lose 16-byte alignment."""
    gen = torch.Generator().manual_seed(seed)
    out = []
    for n, pdt, gdt, master, off in specs:
        p = (torch.randn(n + off, generator=gen) * 1e-2).to(pdt).to(DEV)[off:]
        g = (torch.randn(n + off, generator=gen) * 1e-3).to(gdt).to(DEV)[off:]
        m = (torch.randn(n + off, generator=gen) * 1e-4).to(DEV)[off:]
        v = (torch.rand(n + off, generator=gen) * 1e-6).to(DEV)[off:]
        ms = p.float().clone() if master else None
        out.append([p, g, m, v, ms])
    return out


def _clone(ts):
    return [[None if x is None else x.clone() for x in t] for t in ts]


def _hps(L, step, n, l2_every=0):
    hps = []
    for i in range(n):
        wd = 0.0 if i % 3 == 2 else 0.1 * (1 + i % 2)
        hps.append(L.make_adamw_hparams(1e-3 * (1 + i % 4), 0.9, 0.95 + 0.01 * (i % 2), 1e-8, wd, step,
                                        l2=bool(l2_every) and i % l2_every == 0))
    return hps


def _assert_same(a, b, what):
    for i, (x, y) in enumerate(zip(a, b)):
        for j, (u, w) in enumerate(zip(x, y)):
            if u is None:
                continue
            assert torch.equal(u, w), f"{what}: tensor {i} field {j}"


MIXED = [
    (100_003, torch.float32, torch.float32, False, 0),
    (3 * 8192 + 5, torch.bfloat16, torch.bfloat16, False, 0),
    (7, torch.float32, torch.bfloat16, False, 0),
    (65_536, torch.bfloat16, torch.float32, False, 0),
    (50_000, torch.bfloat16, torch.bfloat16, True, 0),
    (12_345, torch.bfloat16, torch.float32, True, 0),
    (9_999, torch.float32, torch.float32, False, 1),     # misaligned: scalar path
    (20_001, torch.bfloat16, torch.bfloat16, False, 3),  # misaligned bf16
    (1, torch.bfloat16, torch.bfloat16, True, 0),
    (8192, torch.float32, torch.float32, False, 0),      # exactly one chunk
]


@pytest.mark.parametrize("l2_every", [0, 2])
def test_grouped_equals_per_tensor(L, l2_every):
    ref = _tensor_set(1, MIXED)
    got = _clone(ref)
    ws = torch.zeros(L.adamw_workspace_bytes_grouped(len(MIXED)), dtype=torch.uint8, device=DEV)
    for step in (1, 2, 3):
        hps = _hps(L, step, len(MIXED), l2_every)
        for (p, g, m, v, ms), hp in zip(ref, hps):
            if ms is None:
                L.adamw_step(p, g, m, v, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, step, l2=bool(hp.l2))
            else:
                L.adamw_step_master(ms, p, g, m, v, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, step,
                                    l2=bool(hp.l2))
        arr = L.make_adamw_tensors([(p, g, m, v, hp) + ((ms,) if ms is not None else ())
                                    for (p, g, m, v, ms), hp in zip(got, hps)])
        L.adamw_step_grouped(arr, ws)
        torch.cuda.synchronize()
        _assert_same(got, ref, f"step {step}")


def test_grouped_two_passes(L):
    rng = np.random.default_rng(5)
    specs = [(int(rng.integers(1, 20_000)), torch.bfloat16 if i % 2 else torch.float32, torch.bfloat16, False,
              int(i % 5 == 0)) for i in range(150)]
    ref = _tensor_set(2, specs)
    got = _clone(ref)
    hps = _hps(L, 4, len(specs))
    for (p, g, m, v, _), hp in zip(ref, hps):
        L.adamw_step(p, g, m, v, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, 4)
    ws = torch.zeros(L.adamw_workspace_bytes_grouped(len(specs)), dtype=torch.uint8, device=DEV)
    assert ws.numel() == 2 * 256
    L.adamw_step_grouped(L.make_adamw_tensors([(p, g, m, v, hp) for (p, g, m, v, _), hp in zip(got, hps)]), ws)
    torch.cuda.synchronize()
    _assert_same(got, ref, "two passes")


def test_grouped_against_oracle(L):
    # fp32 parameters: the oracle's fp64 update within 1e-6 of the magnitude of its terms, three steps
    n = 3 * 8192 + 77
    (p, g, m, v, _), = _tensor_set(3, [(n, torch.float32, torch.float32, False, 0)])
    m.zero_()
    v.zero_()
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    po, mo, vo = f64(p), np.zeros(n), np.zeros(n)
    gen = torch.Generator().manual_seed(9)
    for t in (1, 2, 3):
        g.copy_(torch.randn(n, generator=gen) * 1e-3)
        hp = L.make_adamw_hparams(3e-4, 0.9, 0.95, 1e-8, 0.1, t)
        L.adamw_step_grouped(L.make_adamw_tensors([(p, g, m, v, hp)]), ws)
        prev = po
        po, mo, vo = oadamw.adamw_update(po, f64(g), mo, vo, t, lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8,
                                         weight_decay=0.1, param_dtype="f32")
        torch.cuda.synchronize()
        scale = np.abs(prev) + 3e-4 * (1 + 1e-3)
        assert np.max(np.abs(f64(p) - po) / scale) <= 1e-6 * t, t


def _muon_set(L, shapes, seed):
    gen = torch.Generator().manual_seed(seed)
    out = []
    for K, A, B, dt in shapes:
        p = (torch.randn((K, A, B), generator=gen) * 1e-3).to(dt).to(DEV)
        g = (torch.randn((K, A, B), generator=gen) * 1e-3).to(dt).to(DEV)
        out.append([p, g, torch.zeros((K, A, B), dtype=torch.float32, device=DEV)])
    return out


def _buckets(L, mset, shapes):
    code = lambda t: L.MUON_F32 if t.dtype == torch.float32 else L.MUON_BF16
    specs = []
    for (p, g, mom), (K, A, B, _) in zip(mset, shapes):
        specs.append((L.pointer_array([p[k] for k in range(K)], DEV), L.pointer_array([g[k] for k in range(K)], DEV),
                      mom, K, A, B, code(p), code(g)))
    return L.make_buckets(specs)


SHAPES = [(4, 256, 512, torch.bfloat16), (4, 512, 256, torch.bfloat16), (2, 384, 384, torch.float32),
          (3, 64, 128, torch.float32)]   # the last one takes the fused small-matrix path


@pytest.mark.parametrize("form", ["both", "muon_only", "adamw_only"])
def test_hybrid_equals_sequential(L, form):
    hp = hp_struct(L, workloads.workload("gpt2s").muon_hp)
    m_ref, m_got = _muon_set(L, SHAPES, 11), None
    m_got = [[x.clone() for x in t] for t in m_ref]
    a_specs = [(1_000_003, torch.bfloat16, torch.bfloat16, False, 0), (768, torch.bfloat16, torch.bfloat16, False, 0),
               (5000, torch.float32, torch.float32, False, 0), (40_000, torch.bfloat16, torch.bfloat16, True, 0),
               (300_001, torch.bfloat16, torch.float32, False, 0), (77, torch.float32, torch.float32, False, 1)]
    a_ref = _tensor_set(12, a_specs)
    a_got = _clone(a_ref)
    b_ref, b_got = _buckets(L, m_ref, SHAPES), _buckets(L, m_got, SHAPES)
    ws_ref = torch.zeros(L.muon_workspace_bytes_grouped(b_ref), dtype=torch.uint8, device=DEV)
    ws_got = torch.zeros_like(ws_ref)
    aws_ref = torch.zeros(256, dtype=torch.uint8, device=DEV)
    aws_got = torch.zeros(256, dtype=torch.uint8, device=DEV)
    for step in (1, 2):
        hps = _hps(L, step, len(a_specs))
        arr = lambda ts: L.make_adamw_tensors([(p, g, m, v, h) + ((ms,) if ms is not None else ())
                                               for (p, g, m, v, ms), h in zip(ts, hps)])
        if form != "adamw_only":
            L.muon_step_grouped(b_ref, hp, ws_ref)
        if form != "muon_only":
            L.adamw_step_grouped(arr(a_ref), aws_ref)
        L.hybrid_step(b_got if form != "adamw_only" else None, hp, ws_got,
                      arr(a_got) if form != "muon_only" else None, aws_got)
        # ordered on the caller's stream: compared there before any device-wide sync
        if form != "adamw_only":
            assert all(torch.equal(x, y) for t, u in zip(m_got, m_ref) for x, y in zip(t, u)), step
        torch.cuda.synchronize()
        if form != "muon_only":
            _assert_same(a_got, a_ref, f"adamw step {step}")
        assert L.muon_check(ws_got) == L.MUON_OK


def test_hybrid_gpt2_small_full_size(L):
    """The GPT-2-small-shaped step as the benchmark runs it (48 Muon matrices, 77 M AdamW elements)."""
    w = workloads.workload("gpt2s")
    plan = L.muon_plan_buckets(workloads.shape_list(w))
    shapes = [(K, A, B, torch.bfloat16) for (A, B), K in zip(plan["bucket_shapes"], plan["bucket_K"])]
    m_ref = _muon_set(L, shapes, 21)
    m_got = [[x.clone() for x in t] for t in m_ref]
    n_big = sum(t.numel for t in w.adamw if t.weight_decay != 0)
    n_small = sum(t.numel for t in w.adamw if t.weight_decay == 0)
    a_ref = _tensor_set(22, [(n_big, torch.bfloat16, torch.bfloat16, False, 0),
                             (n_small, torch.bfloat16, torch.bfloat16, False, 0)])
    a_got = _clone(a_ref)
    hp = hp_struct(L, w.muon_hp)
    b_ref, b_got = _buckets(L, m_ref, shapes), _buckets(L, m_got, shapes)
    ws_ref = torch.zeros(L.muon_workspace_bytes_grouped(b_ref), dtype=torch.uint8, device=DEV)
    ws_got = torch.zeros_like(ws_ref)
    aws_ref = torch.zeros(256, dtype=torch.uint8, device=DEV)
    aws_got = torch.zeros(256, dtype=torch.uint8, device=DEV)
    a = w.adamw_hp
    for step in (1, 2, 3):
        hps = [L.make_adamw_hparams(a.lr, a.beta1, a.beta2, a.eps, wd, step) for wd in (0.1, 0.0)]
        arr = lambda ts: L.make_adamw_tensors([(p, g, m, v, h) for (p, g, m, v, _), h in zip(ts, hps)])
        L.muon_step_grouped(b_ref, hp, ws_ref)
        L.adamw_step_grouped(arr(a_ref), aws_ref)
        L.hybrid_step(b_got, hp, ws_got, arr(a_got), aws_got)
    torch.cuda.synchronize()
    assert L.muon_check(ws_got) == L.MUON_OK
    for t, u in zip(m_got, m_ref):
        assert torch.equal(t[0], u[0]) and torch.equal(t[2], u[2])
    _assert_same(a_got, a_ref, "gpt2s adamw")


def test_hybrid_in_pieces(L):
    """hybrid_step with its Muon step cut into pieces of one matrix each (muon_debug_piece_elems): the AdamW pass's
    counters are cleared with the first piece's, and every result equals the uncut step's bit for bit."""
    hp = hp_struct(L, workloads.workload("gpt2s").muon_hp)
    a_specs = [(1_000_003, torch.bfloat16, torch.bfloat16, False, 0), (5000, torch.float32, torch.float32, False, 0)]
    runs = []
    try:
        for elems in (0, 1):
            L.muon_debug_piece_elems(elems)
            mset = _muon_set(L, SHAPES, 21)
            aset = _tensor_set(22, a_specs)
            bk = _buckets(L, mset, SHAPES)
            ws = torch.zeros(L.muon_workspace_bytes_grouped(bk), dtype=torch.uint8, device=DEV)
            aws = torch.zeros(256, dtype=torch.uint8, device=DEV)
            for step in (1, 2):
                hps = _hps(L, step, len(a_specs))
                arr = L.make_adamw_tensors([(p, g, m, v, h) + ((ms,) if ms is not None else ())
                                            for (p, g, m, v, ms), h in zip(aset, hps)])
                L.hybrid_step(bk, hp, ws, arr, aws)
            torch.cuda.synchronize()
            assert L.muon_check(ws) == L.MUON_OK
            runs.append((mset, aset))
    finally:
        L.muon_debug_piece_elems(0)
    (m0, a0), (m1, a1) = runs
    assert all(torch.equal(x, y) for t, u in zip(m0, m1) for x, y in zip(t, u))
    _assert_same(a1, a0, "adamw in pieces")
