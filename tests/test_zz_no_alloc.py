"""ns_orthogonalize_noalloc, the entry point for callers that cannot allocate device memory.

Such callers (code inside an allocator's own hooks, plugins without an allocation API, runtimes with
a device-memory budget fixed at start-up) cannot hand the library a workspace; this call uses the
library's built-in scratch instead. The test calls it through the C ABI twice in a row, on different
inputs, and checks each result against ns_orthogonalize (which uses a caller-provided workspace)
within the tests' bound for orthogonalised outputs (relative Frobenius error 2e-2); it also checks
that a stack too large for the built-in scratch is refused before anything runs.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from tests.gpu_common import DEV, build_lib, f64, rel_fro, workspace

pytestmark = pytest.mark.gpu

CLASSIC5 = [(3.4445, -4.7750, 2.0315)] * 5


@pytest.fixture(scope="module")
def L():
    return build_lib()


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row(L):
    cases = [((4, 64, 128), torch.float32, torch.float32, 1), ((3, 200, 72), torch.bfloat16, torch.bfloat16, 2)]
    for (K, A, B), xdt, odt, seed in cases:
        g = torch.Generator().manual_seed(seed)
        x = torch.randn((K, A, B), generator=g, dtype=torch.float64).to(xdt).to(DEV)
        ref = torch.empty((K, A, B), dtype=odt, device=DEV)
        ws = workspace(L, K, A, B)
        L.ns_orthogonalize(x, ref, CLASSIC5, 1e-7, ws)
        got = torch.full((K, A, B), float("nan"), dtype=odt, device=DEV)
        L.ns_orthogonalize_noalloc(x, got, CLASSIC5, 1e-7)
        torch.cuda.synchronize()
        assert L.muon_check(ws) == L.MUON_OK
        r, o = f64(ref), f64(got)
        assert np.all(np.isfinite(o))
        for k in range(K):
            assert rel_fro(o[k], r[k]) <= 2e-2


def test_noalloc_refuses_stacks_beyond_its_scratch(L):
    x = torch.empty((64, 1024, 1024), dtype=torch.bfloat16, device=DEV)
    out = torch.empty_like(x)
    with pytest.raises(L.MuonError) as e:
        L.ns_orthogonalize_noalloc(x, out, CLASSIC5, 1e-7)
    assert e.value.status == L.MUON_ERR_WORKSPACE
