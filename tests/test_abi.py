"""The C ABI without a GPU: the library loads, exports every symbol the header declares, its host-only
bucket planner matches the oracle bit for bit, and argument checks return their codes before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

from adamw_hybrid_optimizer_gb300 import libmuon as L
from oracle import buckets as obuckets
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "libmuon.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("muon_step_batched", "adamw_step", "ns_orthogonalize", "muon_workspace_bytes", "muon_plan_buckets",
                 "muon_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    lib = L.lib()
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(L.SIGNATURES)


def test_hparam_struct_layouts():
    # the C layout: five floats, the int32 mode, then the int64 step at offset 24
    assert ctypes.sizeof(L.adamw_hparams) == 32 and L.adamw_hparams.step.offset == 24
    assert L.adamw_hparams.l2.offset == 20


def test_status_strings():
    for code in range(0, 9):
        assert L.muon_status_string(code).startswith("MUON_")
    assert "unknown" in L.muon_status_string(99)


def _plan_both(shapes):
    ours = L.muon_plan_buckets(shapes)
    ref = obuckets.plan_buckets(shapes)
    assert ours["bucket_id"] == ref["bucket_id"]
    assert ours["index_in_bucket"] == ref["index_in_bucket"]
    assert ours["bucket_shapes"] == [tuple(s) for s in ref["bucket_shapes"]]
    assert ours["bucket_K"] == ref["bucket_K"]
    assert ours["momentum_offset"] == ref["momentum_offset"]


@pytest.mark.parametrize("name", ["tiny", "gpt2s", "llama8b", "aspect"])
def test_bucket_plan_matches_oracle_on_model_sets(name):
    _plan_both(workloads.shape_list(workloads.workload(name)))


def test_bucket_plan_matches_oracle_random_and_edge():
    rng = np.random.default_rng(0)
    _plan_both([])
    _plan_both([(1, 1)])
    _plan_both([(65536, 1), (1, 65536), (65536, 1)])
    _plan_both([(3, 5), (5, 3), (3, 5), (2**33, 7), (7, 2**33), (2**33, 7)])   # keys beyond 32 bits stay exact
    for _ in range(300):
        n = int(rng.integers(1, 40))
        _plan_both([tuple(int(v) for v in rng.integers(1, 5, 2)) for _ in range(n)])


def test_bucket_plan_rejects_bad_dims():
    with pytest.raises(L.MuonError) as e:
        L.muon_plan_buckets([(4, 0)])
    assert e.value.status == L.MUON_ERR_INVALID_ARG


def test_workspace_bytes():
    assert L.muon_workspace_bytes(0, 4, 4) == 0
    small = L.muon_workspace_bytes(4, 64, 128)
    assert small > 0 and small % 1024 == 0
    # two (K, m, n) bf16 iterates + two (K, m, m) Gram buffers dominate
    K, m, n = 12, 768, 3072
    big = L.muon_workspace_bytes(K, n, m)
    assert big >= 2 * 2 * K * m * n + 2 * 2 * K * m * m
    assert big == L.muon_workspace_bytes(K, m, n)


# ---------------------------------------------------------------------------------------- argument checks
# These return before anything touches CUDA, so they run without a GPU. Fake device pointers are never
# dereferenced on the host.

FAKE = 1 << 20


def _step(params=FAKE, grads=FAKE, mom=FAKE, K=4, A=64, B=128, pdt=L.MUON_F32, gdt=L.MUON_F32, hp=None, ws=FAKE,
          ws_bytes=None):
    if hp is None:
        hp = L.make_muon_hparams(0.02, 0.95, 0.01)
    if ws_bytes is None:
        ws_bytes = L.muon_workspace_bytes(max(K, 1), max(A, 1), max(B, 1))
    return L.lib().muon_step_batched(params, pdt, grads, gdt, mom, K, A, B, ctypes.byref(hp) if hp is not False else None,
                                     ws, ws_bytes, None)


def test_step_argument_checks():
    assert _step(params=None) == L.MUON_ERR_INVALID_ARG
    assert _step(grads=None) == L.MUON_ERR_INVALID_ARG
    assert _step(mom=None) == L.MUON_ERR_INVALID_ARG
    assert _step(ws=None) == L.MUON_ERR_INVALID_ARG
    assert _step(hp=False) == L.MUON_ERR_INVALID_ARG
    assert _step(K=0) == L.MUON_ERR_INVALID_ARG
    assert _step(A=-1) == L.MUON_ERR_INVALID_ARG
    assert _step(A=70000) == L.MUON_ERR_SHAPE
    assert _step(pdt=7) == L.MUON_ERR_DTYPE
    assert _step(hp=L.make_muon_hparams(0.02, 0.95, 0.01, coeffs=[])) == L.MUON_ERR_INVALID_ARG
    assert _step(hp=L.make_muon_hparams(0.02, 0.95, 0.01, coeffs=[(1, 2, 3)] * 33)) == L.MUON_ERR_INVALID_ARG
    assert _step(hp=L.make_muon_hparams(0.02, 0.95, 0.01, coeffs=[(float("nan"), 1, 1)])) == L.MUON_ERR_INVALID_ARG
    assert _step(hp=L.make_muon_hparams(0.02, 0.95, 0.01, scale_mode=3)) == L.MUON_ERR_INVALID_ARG
    assert _step(hp=L.make_muon_hparams(float("inf"), 0.95, 0.01)) == L.MUON_ERR_INVALID_ARG
    assert _step(ws=FAKE + 16) == L.MUON_ERR_ALIGNMENT
    assert _step(ws_bytes=1024) == L.MUON_ERR_WORKSPACE


def test_other_entry_point_checks():
    lib = L.lib()
    c, n = L._coeff_array([(3.4445, -4.775, 2.0315)] * 5)
    ws_b = L.muon_workspace_bytes(2, 16, 16)
    assert lib.ns_orthogonalize(None, 0, FAKE, 0, 2, 16, 16, n, c, 1e-7, FAKE, ws_b, None) == L.MUON_ERR_INVALID_ARG
    assert lib.ns_orthogonalize(FAKE, 5, FAKE, 0, 2, 16, 16, n, c, 1e-7, FAKE, ws_b, None) == L.MUON_ERR_DTYPE
    assert lib.ns_orthogonalize(FAKE, 0, FAKE, 0, 2, 16, 16, 0, c, 1e-7, FAKE, ws_b, None) == L.MUON_ERR_INVALID_ARG
    assert lib.ns_orthogonalize(FAKE, 0, FAKE, 0, 2, 16, 16, n, c, -1.0, FAKE, ws_b, None) == L.MUON_ERR_INVALID_ARG
    assert lib.ns_orthogonalize(FAKE, 0, FAKE, 0, 2, 16, 16, n, c, 1e-7, FAKE, 64, None) == L.MUON_ERR_WORKSPACE
    hp = L.adamw_hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1)
    assert lib.adamw_step(None, 0, FAKE, 0, FAKE, FAKE, 8, ctypes.byref(hp), None) == L.MUON_ERR_INVALID_ARG
    assert lib.adamw_step(FAKE, 0, FAKE, 0, FAKE, FAKE, 0, ctypes.byref(hp), None) == L.MUON_ERR_INVALID_ARG
    assert lib.adamw_step(FAKE, 2, FAKE, 0, FAKE, FAKE, 8, ctypes.byref(hp), None) == L.MUON_ERR_DTYPE
    bad = L.adamw_hparams(lr=1e-3, beta1=1.0, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1)
    assert lib.adamw_step(FAKE, 0, FAKE, 0, FAKE, FAKE, 8, ctypes.byref(bad), None) == L.MUON_ERR_INVALID_ARG
    t0 = L.adamw_hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=0)
    assert lib.adamw_step(FAKE, 0, FAKE, 0, FAKE, FAKE, 8, ctypes.byref(t0), None) == L.MUON_ERR_INVALID_ARG
    t0 = L.adamw_hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, l2=2, step=1)
    assert lib.adamw_step(FAKE, 0, FAKE, 0, FAKE, FAKE, 8, ctypes.byref(t0), None) == L.MUON_ERR_INVALID_ARG
    assert lib.ns_gram(FAKE, FAKE, 1, 12, 16, 1.0, FAKE, 256, None) == L.MUON_ERR_SHAPE       # m not a multiple of 8
    assert lib.ns_gram(FAKE + 8, FAKE, 1, 16, 16, 1.0, FAKE, 256, None) == L.MUON_ERR_ALIGNMENT
    assert lib.ns_gram(FAKE, FAKE, 1, 16, 16, 1.0, FAKE, 128, None) == L.MUON_ERR_WORKSPACE
    assert lib.ns_apply(FAKE, FAKE, FAKE, 1, 16, 16, FAKE, 256, None) == L.MUON_ERR_INVALID_ARG  # out aliases x
    assert lib.ns_poly(FAKE, FAKE, 1, 16, float("nan"), 1.0, 1.0, FAKE, 256, None) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_debug_wait_timeout(FAKE, 256, 0, None) == L.MUON_ERR_INVALID_ARG


def test_launch_counter_starts_at_zero_without_launches():
    assert L.muon_launch_count() >= 0
    assert L.muon_trace_collect() == []


def test_grouped_entry_point_checks():
    lib = L.lib()
    hp = L.make_muon_hparams(0.02, 0.95, 0.01)
    good = (L.muon_bucket * 2)(L.muon_bucket(FAKE, FAKE, FAKE, 4, 64, 128, 0, 0),
                               L.muon_bucket(FAKE, FAKE, FAKE, 2, 128, 64, 1, 1))
    need = L.muon_workspace_bytes_grouped(good)
    # one shared 1 KiB header (control block + one counter per matrix) instead of one per stack
    assert need == L.muon_workspace_bytes(4, 64, 128) + L.muon_workspace_bytes(2, 128, 64) - 1024
    st = lambda b, n=2, ws=FAKE, nb=need: lib.muon_step_grouped(b, n, ctypes.byref(hp), ws, nb, None)
    assert st(good, n=0) == L.MUON_ERR_INVALID_ARG
    assert st(good, ws=None) == L.MUON_ERR_INVALID_ARG
    assert st(good, ws=FAKE + 8) == L.MUON_ERR_ALIGNMENT
    assert st(good, nb=need - 1) == L.MUON_ERR_WORKSPACE
    bad = (L.muon_bucket * 2)(good[0], L.muon_bucket(None, FAKE, FAKE, 2, 128, 64, 1, 1))
    assert st(bad) == L.MUON_ERR_INVALID_ARG
    bad = (L.muon_bucket * 2)(good[0], L.muon_bucket(FAKE, FAKE, FAKE, 2, 128, 0, 1, 1))
    assert st(bad) == L.MUON_ERR_INVALID_ARG
    bad = (L.muon_bucket * 2)(good[0], L.muon_bucket(FAKE, FAKE, FAKE, 2, 128, 64, 1, 9))
    assert st(bad) == L.MUON_ERR_DTYPE
    assert L.muon_workspace_bytes_grouped((L.muon_bucket * 1)(L.muon_bucket(FAKE, FAKE, FAKE, 0, 1, 1, 0, 0))) == 0
    # fp32 master weights go with bf16 parameters only
    bad = (L.muon_bucket * 2)(good[0], L.muon_bucket(FAKE, FAKE, FAKE, 2, 128, 64, L.MUON_F32, 1, FAKE))
    assert st(bad) == L.MUON_ERR_DTYPE
    hp2 = L.adamw_hparams(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1)
    assert lib.adamw_step_master(None, FAKE, FAKE, 0, FAKE, FAKE, 8, ctypes.byref(hp2), None) == L.MUON_ERR_INVALID_ARG
    assert lib.adamw_step_master(FAKE, FAKE, FAKE, 5, FAKE, FAKE, 8, ctypes.byref(hp2), None) == L.MUON_ERR_DTYPE


def test_adamw_tensor_struct_layout():
    # five pointers, the int64 count at 40, the two dtype enums, then the hparams pointer at 56
    assert ctypes.sizeof(L.adamw_tensor) == 64
    assert L.adamw_tensor.n.offset == 40 and L.adamw_tensor.pdt.offset == 48 and L.adamw_tensor.hp.offset == 56


def _adamw_t(param=FAKE, grad=FAKE, m=FAKE, v=FAKE, master=None, n=8192, pdt=L.MUON_BF16, gdt=L.MUON_BF16, hp=None):
    if hp is None:
        hp = L.make_adamw_hparams(1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    t = L.adamw_tensor(param, grad, m, v, master, n, pdt, gdt, ctypes.pointer(hp) if hp is not False else None)
    t._hp = hp
    return t


def test_grouped_adamw_entry_point_checks():
    lib = L.lib()
    assert L.adamw_workspace_bytes_grouped(0) == 0
    assert L.adamw_workspace_bytes_grouped(1) == 256
    assert L.adamw_workspace_bytes_grouped(96) == 256 and L.adamw_workspace_bytes_grouped(97) == 512

    def st(*ts, ws=FAKE, nb=256, n=None):
        arr = (L.adamw_tensor * max(len(ts), 1))(*ts)
        return lib.adamw_step_grouped(arr, len(ts) if n is None else n, ws, nb, None)

    good = _adamw_t()
    assert st(good, n=0) == L.MUON_ERR_INVALID_ARG
    assert st(good, ws=None) == L.MUON_ERR_INVALID_ARG
    assert st(good, ws=FAKE + 16) == L.MUON_ERR_ALIGNMENT
    assert st(good, nb=255) == L.MUON_ERR_WORKSPACE
    assert st(*([good] * 97), nb=256) == L.MUON_ERR_WORKSPACE
    assert st(good, _adamw_t(param=None)) == L.MUON_ERR_INVALID_ARG
    assert st(good, _adamw_t(v=None)) == L.MUON_ERR_INVALID_ARG
    assert st(good, _adamw_t(n=0)) == L.MUON_ERR_INVALID_ARG
    assert st(good, _adamw_t(hp=False)) == L.MUON_ERR_INVALID_ARG
    assert st(good, _adamw_t(gdt=4)) == L.MUON_ERR_DTYPE
    # a master copy goes with bf16 parameters only
    assert st(good, _adamw_t(master=FAKE, pdt=L.MUON_F32)) == L.MUON_ERR_DTYPE
    assert st(good, _adamw_t(hp=L.make_adamw_hparams(1e-3, 0.9, 0.95, 1e-8, 0.1, 0))) == L.MUON_ERR_INVALID_ARG
    assert st(good, _adamw_t(hp=L.make_adamw_hparams(1e-3, 0.9, 1.0, 1e-8, 0.1, 1))) == L.MUON_ERR_INVALID_ARG


def test_hybrid_step_entry_point_checks():
    lib = L.lib()
    hp = L.make_muon_hparams(0.02, 0.95, 0.01)
    b = (L.muon_bucket * 1)(L.muon_bucket(FAKE, FAKE, FAKE, 4, 64, 128, 0, 0))
    need = L.muon_workspace_bytes_grouped(b)
    ts = (L.adamw_tensor * 1)(_adamw_t())
    aws = 1 << 30   # far from the Muon workspace at FAKE

    def st(nb=1, nt=1, ws=FAKE, wsb=need, a=aws, ab=256, bk=b, t=ts):
        return lib.hybrid_step(bk, nb, ctypes.byref(hp), ws, wsb, t, nt, a, ab, None)

    assert st(nb=0, nt=0) == L.MUON_ERR_INVALID_ARG
    assert st(nb=-1) == L.MUON_ERR_INVALID_ARG
    assert st(wsb=need - 1) == L.MUON_ERR_WORKSPACE
    assert st(ab=100) == L.MUON_ERR_WORKSPACE
    assert st(nb=0, ab=100) == L.MUON_ERR_WORKSPACE
    assert st(nt=0, wsb=need - 1) == L.MUON_ERR_WORKSPACE
    assert st(a=aws + 8) == L.MUON_ERR_ALIGNMENT
    # the AdamW counters may not lie inside the Muon workspace
    assert st(a=FAKE + 1024) == L.MUON_ERR_INVALID_ARG
    bad = (L.adamw_tensor * 1)(_adamw_t(grad=None))
    assert st(t=bad) == L.MUON_ERR_INVALID_ARG
    bad_b = (L.muon_bucket * 1)(L.muon_bucket(FAKE, FAKE, FAKE, 4, 64, 0, 0, 0))
    assert st(bk=bad_b) == L.MUON_ERR_INVALID_ARG
    # with every argument valid, the only thing left is the device (none in a CPU-only run)
    import torch
    if not torch.cuda.is_available():
        assert st() in (L.MUON_ERR_CUDA, L.MUON_ERR_UNSUPPORTED_DEVICE)


def test_autotune_entry_point_checks_and_table():
    lib = L.lib()
    good = (L.muon_bucket * 1)(L.muon_bucket(FAKE, FAKE, FAKE, 4, 768, 2304, 1, 1))
    need = L.muon_workspace_bytes_grouped(good)
    hp = ctypes.byref(L.make_muon_hparams(0.02, 0.95, 0.01))
    assert lib.muon_autotune(None, 1, hp, FAKE, need, None) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_autotune(good, 0, hp, FAKE, need, None) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_autotune(good, 1, None, FAKE, need, None) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_autotune(good, 1, hp, None, need, None) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_autotune(good, 1, hp, FAKE + 8, need, None) == L.MUON_ERR_ALIGNMENT
    assert lib.muon_autotune(good, 1, hp, FAKE, need - 1, None) == L.MUON_ERR_WORKSPACE
    bad = (L.muon_bucket * 1)(L.muon_bucket(FAKE, FAKE, FAKE, 4, 768, 0, 1, 1))
    assert lib.muon_autotune(bad, 1, hp, FAKE, need, None) == L.MUON_ERR_INVALID_ARG
    L.muon_autotune_reset()
    assert L.muon_autotune_poly_shape(768) == -1
    assert L.muon_autotune_poly_shape(0) == -1
    assert L.muon_autotune_route(16, 256, 16384) == -1 and L.muon_autotune_route(0, 256, 16384) == -1
    assert L.muon_autotune_scheduling(good) == -1
    assert lib.muon_autotune_scheduling(None, 1) == -1
    assert lib.muon_debug_poly_shape(3) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_debug_poly_shape(-2) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_debug_poly_shape(1) == L.MUON_OK
    assert lib.muon_debug_poly_shape(-1) == L.MUON_OK
    assert L.muon_autotune_gram_split(16, 256, 16384) == -1
    assert L.muon_autotune_gram_split(0, 256, 16384) == -1 and L.muon_autotune_gram_split(16, 0, 16384) == -1
    assert lib.muon_debug_piece_elems(-1) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_debug_piece_elems(1 << 20) == L.MUON_OK and lib.muon_debug_piece_elems(0) == L.MUON_OK
    for bad_split in (0, 5, -2):
        assert lib.muon_debug_gram_split(bad_split) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_debug_gram_split(4) == L.MUON_OK
    assert lib.muon_debug_gram_split(-1) == L.MUON_OK


def test_counter_deps_switch():
    lib = L.lib()
    assert lib.muon_debug_counter_deps(2) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_debug_counter_deps(-2) == L.MUON_ERR_INVALID_ARG
    for mode in (1, 0, -1):
        assert lib.muon_debug_counter_deps(mode) == L.MUON_OK
