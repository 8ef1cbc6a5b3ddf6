"""ns_orthogonalize_noalloc, the entry point for callers that cannot allocate device memory.

Such callers (code inside an allocator's own hooks, plugins without an allocation API, runtimes with
a device-memory budget fixed at start-up) cannot hand the library a workspace; this call uses the
library's built-in scratch instead. The tests call it through the C ABI several times in a row, on
different inputs, and check each result against the fp64 oracle's Newton-Schulz output and against
ns_orthogonalize (which uses a caller-provided workspace), both within the tests' bound for
orthogonalised outputs (relative Frobenius error 2e-2). The shapes cover the fused small-matrix range
(where ns_orthogonalize runs another kernel), one stack above it (the same GEMM kernels on both sides),
a tall fp32 stack stored as bf16, and a wide stack that takes the Gram-space path. They also check that a stack too large for the built-in scratch is
refused before anything runs, and that a bounded wait that runs out is reported by
ns_orthogonalize_noalloc_check (and only once), with the context still usable afterwards.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from oracle import muon as omuon
from tests.gpu_common import DEV, build_lib, f64, rel_fro, workspace

pytestmark = pytest.mark.gpu

CLASSIC5 = [(3.4445, -4.7750, 2.0315)] * 5

CASES = [
    ((4, 64, 128), torch.float32, torch.float32, 1),
    ((3, 200, 72), torch.bfloat16, torch.bfloat16, 2),
    ((2, 512, 1024), torch.bfloat16, torch.float32, 3),     # above the fused small-matrix limit
    ((2, 640, 256), torch.float32, torch.bfloat16, 4),      # tall: transposed to wide and back
    ((3, 128, 2048), torch.bfloat16, torch.bfloat16, 5),    # the Gram-space path, its fp32 Gram split
]


@pytest.fixture(scope="module")
def L():
    return build_lib()


def test_noalloc_matches_oracle_and_workspace_entry_point_on_calls_in_a_row(L):
    for (K, A, B), xdt, odt, seed in CASES:
        g = torch.Generator().manual_seed(seed)
        x = torch.randn((K, A, B), generator=g, dtype=torch.float64).to(xdt).to(DEV)
        ref = torch.empty((K, A, B), dtype=odt, device=DEV)
        ws = workspace(L, K, A, B)
        L.ns_orthogonalize(x, ref, CLASSIC5, 1e-7, ws)
        got = torch.full((K, A, B), float("nan"), dtype=odt, device=DEV)
        L.ns_orthogonalize_noalloc(x, got, CLASSIC5, 1e-7)
        assert L.ns_orthogonalize_noalloc_check() == L.MUON_OK
        assert L.muon_check(ws) == L.MUON_OK
        X, r, o = f64(x), f64(ref), f64(got)
        assert np.all(np.isfinite(o))
        for k in range(K):
            orc = omuon.newton_schulz(X[k], CLASSIC5, 1e-7)
            assert rel_fro(o[k], orc) <= 2e-2, ((K, A, B), k, rel_fro(o[k], orc))
            assert rel_fro(o[k], r[k]) <= 2e-2, ((K, A, B), k)


def test_noalloc_refuses_stacks_beyond_its_scratch(L):
    x = torch.empty((64, 1024, 1024), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(x)
    with pytest.raises(L.MuonError) as e:
        L.ns_orthogonalize_noalloc(x, out, CLASSIC5, 1e-7)
    assert e.value.status == L.MUON_ERR_WORKSPACE


def test_noalloc_check_reports_a_wait_that_ran_out_once(L):
    # a wait on a barrier that nothing completes, bounded at 1 ms, reporting into the scratch's error word
    L.muon_debug_wait_timeout_noalloc(1_000_000)
    assert L.ns_orthogonalize_noalloc_check() == L.MUON_ERR_TIMEOUT
    assert L.ns_orthogonalize_noalloc_check() == L.MUON_OK          # read and cleared
    # the context keeps working: a call after the report is correct and reports nothing
    g = torch.Generator().manual_seed(7)
    x = torch.randn((2, 96, 160), generator=g, dtype=torch.float64).to(torch.float32).to(DEV)
    out = torch.empty_like(x)
    L.ns_orthogonalize_noalloc(x, out, CLASSIC5, 1e-7)
    assert L.ns_orthogonalize_noalloc_check() == L.MUON_OK
    X, o = f64(x), f64(out)
    for k in range(2):
        assert rel_fro(o[k], omuon.newton_schulz(X[k], CLASSIC5, 1e-7)) <= 2e-2
