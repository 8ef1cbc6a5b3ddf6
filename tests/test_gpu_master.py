"""fp32 master weights for bf16 Muon parameters (muon_bucket.master), through the C ABI.

The update (decay, step) is applied to the fp32 master and the bf16 parameter becomes the new master
rounded to bf16 ("Optimizers: AdamW, Muon and the distributed optimizer", section "The optimizer's memory
budget": fp32 master weights beside bf16 weights). The oracle is the fp32-parameter Muon update on the
master; the bf16 parameter must equal the GPU's master rounded to bf16, bit for bit, after every step.
Wide and tall (transposed path) ragged stacks, two steps, on the plain chain and (200 x 1000 and its
transpose) on the Gram-space path, whose final step is the same master-weight kernel with the [R_hi | R_lo]
operand; and a step cut into pieces of one matrix each, against the uncut step.
"""
import numpy as np
import pytest
import torch

from oracle import muon as omuon
from tests.gpu_common import DEV, build_lib, f64, hp_struct
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    return build_lib()


@pytest.mark.parametrize("shape", [(136, 264), (264, 136), (200, 1000), (1000, 200)])
def test_muon_fp32_master_two_steps(L, shape):
    A, B = shape
    K = 3
    assert L.muon_gram_space_route(A, B) == (min(A, B) == 200)
    hp = workloads.workload("tiny").muon_hp
    gen = torch.Generator().manual_seed(A * 7 + B)
    master = [(torch.randn((A, B), generator=gen) * 0.05).to(DEV) for _ in range(K)]
    params = [m.to(torch.bfloat16) for m in master]
    mom = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
    m_orc = [f64(m) for m in master]
    mom_orc = [np.zeros((A, B)) for _ in range(K)]
    first = [x.copy() for x in m_orc]
    pptr, mptr = L.pointer_array(params, DEV), L.pointer_array(master, DEV)
    hps = hp_struct(L, hp)
    for step in range(1, 3):
        grads = [(torch.randn((A, B), generator=gen) * 1e-3).to(torch.bfloat16).to(DEV) for _ in range(K)]
        bk = L.make_buckets([(pptr, L.pointer_array(grads, DEV), mom, K, A, B, L.MUON_BF16, L.MUON_BF16, mptr)])
        ws = torch.zeros(L.muon_workspace_bytes_grouped(bk), dtype=torch.uint8, device=DEV)
        L.muon_step_grouped(bk, hps, ws)
        assert L.muon_check(ws) == L.MUON_OK
        for k in range(K):
            g = f64(grads[k])
            ref, mref, _ = omuon.muon_update(m_orc[k], g, mom_orc[k], lr=hp.lr, momentum=hp.momentum,
                                             weight_decay=hp.weight_decay, nesterov=hp.nesterov, coeffs=hp.coeffs,
                                             eps=hp.eps, param_dtype="f32")
            m_orc[k], mom_orc[k] = ref, mref
            got = f64(master[k])
            assert np.linalg.norm(got - ref) <= 2e-2 * np.linalg.norm(ref - first[k]), (step, k)
            assert torch.equal(params[k], master[k].to(torch.bfloat16)), (step, k)
            assert np.all(np.abs(f64(mom[k]) - mref) <= 1e-6 * (np.abs(mref) + np.abs(g)) + 1e-30)



def test_master_weights_in_pieces(L):
    """A grouped step cut into pieces of one matrix each (muon_debug_piece_elems) gives the masters and the bf16
    parameters of the uncut step bit for bit, on the plain and the Gram-space paths (the fp32 Gram's slice count
    forced, since it depends on a stack's K)."""
    hp = hp_struct(L, workloads.workload("tiny").muon_hp)
    shapes = [(3, 136, 264), (3, 200, 1000)]
    gen = torch.Generator().manual_seed(31)
    base = []
    for K, A, B in shapes:
        master = (torch.randn((K, A, B), generator=gen) * 0.05).to(DEV)
        grad = (torch.randn((K, A, B), generator=gen) * 1e-3).to(torch.bfloat16).to(DEV)
        base.append((master, grad))
    results = {}
    L.muon_debug_gram_split(2)
    try:
        for elems in (0, 1):
            L.muon_debug_piece_elems(elems)
            specs, keep = [], []
            for (K, A, B), (m0, g) in zip(shapes, base):
                master = m0.clone()
                params = master.to(torch.bfloat16)
                mom = torch.zeros((K, A, B), dtype=torch.float32, device=DEV)
                keep.append((master, params, mom))
                specs.append((L.pointer_array([params[k] for k in range(K)], DEV),
                              L.pointer_array([g[k] for k in range(K)], DEV), mom, K, A, B, L.MUON_BF16, L.MUON_BF16,
                              L.pointer_array([master[k] for k in range(K)], DEV)))
            bk = L.make_buckets(specs)
            ws = torch.zeros(L.muon_workspace_bytes_grouped(bk), dtype=torch.uint8, device=DEV)
            for _ in range(2):
                L.muon_step_grouped(bk, hp, ws)
            assert L.muon_check(ws) == L.MUON_OK
            results[elems] = keep
    finally:
        L.muon_debug_piece_elems(0)
        L.muon_debug_gram_split(-1)
    for a, b in zip(results[0], results[1]):
        for x, y in zip(a, b):
            assert torch.equal(x, y)
