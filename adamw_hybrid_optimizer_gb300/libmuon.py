"""ctypes binding of libmuon (include/libmuon.h): argument marshalling only.

Every function here has the name of the C entry point it calls. Tensors are passed as raw
device pointers with their sizes and dtypes; the default stream is torch's current stream.
No computation happens in Python. A missing or unloadable library raises ImportError:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libmuon.so")

MUON_OK = 0
MUON_ERR_INVALID_ARG = 1
MUON_ERR_SHAPE = 2
MUON_ERR_DTYPE = 3
MUON_ERR_ALIGNMENT = 4
MUON_ERR_WORKSPACE = 5
MUON_ERR_UNSUPPORTED_DEVICE = 6
MUON_ERR_CUDA = 7
MUON_ERR_TIMEOUT = 8

MUON_F32 = 0
MUON_BF16 = 1
MUON_MAX_NS_STEPS = 32

# the C signatures, checked against include/libmuon.h by tests/test_abi.py
_c_int64 = ctypes.c_int64
_vp = ctypes.c_void_p


class muon_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("momentum", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("nesterov", ctypes.c_int), ("cautious_wd", ctypes.c_int), ("scale_mode", ctypes.c_int),
                ("ns_steps", ctypes.c_int), ("coeffs", ctypes.POINTER(ctypes.c_float)), ("eps", ctypes.c_float)]


class adamw_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("l2", ctypes.c_int32),
                ("step", ctypes.c_int64)]


class muon_bucket(ctypes.Structure):
    _fields_ = [("params", ctypes.c_void_p), ("grads", ctypes.c_void_p), ("momentum", ctypes.c_void_p),
                ("K", ctypes.c_int64), ("A", ctypes.c_int64), ("B", ctypes.c_int64), ("pdt", ctypes.c_int),
                ("gdt", ctypes.c_int), ("master", ctypes.c_void_p)]


class adamw_tensor(ctypes.Structure):
    _fields_ = [("param", ctypes.c_void_p), ("grad", ctypes.c_void_p), ("exp_avg", ctypes.c_void_p),
                ("exp_avg_sq", ctypes.c_void_p), ("master", ctypes.c_void_p), ("n", ctypes.c_int64),
                ("pdt", ctypes.c_int), ("gdt", ctypes.c_int), ("hp", ctypes.POINTER(adamw_hparams))]


SIGNATURES = {
    "muon_workspace_bytes": (ctypes.c_size_t, [_c_int64, _c_int64, _c_int64]),
    "muon_step_batched": (ctypes.c_int, [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _c_int64, _c_int64, _c_int64,
                                         ctypes.POINTER(muon_hparams), _vp, ctypes.c_size_t, _vp]),
    "muon_workspace_bytes_grouped": (ctypes.c_size_t, [ctypes.POINTER(muon_bucket), ctypes.c_int]),
    "muon_step_grouped": (ctypes.c_int, [ctypes.POINTER(muon_bucket), ctypes.c_int, ctypes.POINTER(muon_hparams), _vp,
                                         ctypes.c_size_t, _vp]),
    "ns_orthogonalize": (ctypes.c_int, [_vp, ctypes.c_int, _vp, ctypes.c_int, _c_int64, _c_int64, _c_int64,
                                        ctypes.c_int, ctypes.POINTER(ctypes.c_float), ctypes.c_float, _vp,
                                        ctypes.c_size_t, _vp]),
    "ns_orthogonalize_noalloc": (ctypes.c_int, [_vp, ctypes.c_int, _vp, ctypes.c_int, _c_int64, _c_int64, _c_int64,
                                                ctypes.c_int, ctypes.POINTER(ctypes.c_float), ctypes.c_float, _vp]),
    "ns_orthogonalize_noalloc_check": (ctypes.c_int, [_vp]),
    "muon_debug_wait_timeout_noalloc": (ctypes.c_int, [ctypes.c_uint64, _vp]),
    "adamw_step": (ctypes.c_int, [_vp, ctypes.c_int, _vp, ctypes.c_int, _vp, _vp, _c_int64,
                                  ctypes.POINTER(adamw_hparams), _vp]),
    "adamw_step_master": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _c_int64,
                                         ctypes.POINTER(adamw_hparams), _vp]),
    "adamw_workspace_bytes_grouped": (ctypes.c_size_t, [_c_int64]),
    "adamw_step_grouped": (ctypes.c_int, [ctypes.POINTER(adamw_tensor), _c_int64, _vp, ctypes.c_size_t, _vp]),
    "hybrid_step": (ctypes.c_int, [ctypes.POINTER(muon_bucket), ctypes.c_int, ctypes.POINTER(muon_hparams), _vp,
                                   ctypes.c_size_t, ctypes.POINTER(adamw_tensor), _c_int64, _vp, ctypes.c_size_t,
                                   _vp]),
    "ns_gram": (ctypes.c_int, [_vp, _vp, _c_int64, _c_int64, _c_int64, ctypes.c_float, _vp, ctypes.c_size_t, _vp]),
    "ns_poly": (ctypes.c_int, [_vp, _vp, _c_int64, _c_int64, ctypes.c_float, ctypes.c_float, ctypes.c_float, _vp,
                               ctypes.c_size_t, _vp]),
    "ns_apply": (ctypes.c_int, [_vp, _vp, _vp, _c_int64, _c_int64, _c_int64, _vp, ctypes.c_size_t, _vp]),
    "muon_plan_buckets": (ctypes.c_int, [_c_int64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "muon_autotune": (ctypes.c_int, [ctypes.POINTER(muon_bucket), ctypes.c_int, ctypes.POINTER(muon_hparams), _vp,
                                     ctypes.c_size_t, _vp]),
    "muon_autotune_route": (ctypes.c_int32, [_c_int64, _c_int64, _c_int64]),
    "muon_autotune_scheduling": (ctypes.c_int32, [ctypes.POINTER(muon_bucket), ctypes.c_int]),
    "muon_autotune_poly_shape": (ctypes.c_int32, [_c_int64]),
    "muon_autotune_gram_split": (ctypes.c_int32, [_c_int64, _c_int64, _c_int64]),
    "muon_debug_piece_elems": (ctypes.c_int, [_c_int64]),
    "muon_autotune_reset": (None, []),
    "muon_debug_gram_split": (ctypes.c_int, [ctypes.c_int32]),
    "muon_debug_poly_shape": (ctypes.c_int, [ctypes.c_int32]),
    "muon_debug_counter_deps": (ctypes.c_int, [ctypes.c_int32]),
    "muon_debug_half_symmetric": (ctypes.c_int, [ctypes.c_int32]),
    "muon_debug_gram_space": (ctypes.c_int, [ctypes.c_int32]),
    "muon_gram_space_route": (ctypes.c_int32, [_c_int64, _c_int64, _c_int64]),
    "muon_check": (ctypes.c_int, [_vp, _vp]),
    "muon_set_timeout_ns": (None, [ctypes.c_uint64]),
    "muon_debug_wait_timeout": (ctypes.c_int, [_vp, ctypes.c_size_t, ctypes.c_uint64, _vp]),
    "muon_launch_count": (ctypes.c_int64, []),
    "muon_debug_timeline": (ctypes.c_int, [_vp, ctypes.c_int64, ctypes.c_int32]),
    "muon_trace_enable": (None, [ctypes.c_int]),
    "muon_trace_collect": (ctypes.c_int64, [_vp, _vp, _c_int64]),
    "muon_kernel_name": (ctypes.c_char_p, [ctypes.c_int32]),
    "muon_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Loads libmuon.so (built by __graft_entry__.build() or adamw_hybrid_optimizer_gb300/_build.py)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmuon.so is not built ({LIB_PATH}); run `python -c \"import __graft_entry__ as g; "
                              f"g.build()\"` first. There is no fallback implementation.")
        try:
            handle = ctypes.CDLL(LIB_PATH)
        except OSError as e:
            raise ImportError(f"libmuon.so failed to load: {e}") from e
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class MuonError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {muon_status_string(status)}")


def muon_status_string(status: int) -> str:
    return lib().muon_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != MUON_OK:
        raise MuonError(status, where)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return MUON_F32
    if t.dtype == torch.bfloat16:
        return MUON_BF16
    raise MuonError(MUON_ERR_DTYPE, f"dtype {t.dtype}")


def _stream(stream) -> int:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _coeff_array(coeffs: Sequence[Sequence[float]]):
    flat = [float(v) for abc in coeffs for v in abc]
    return (ctypes.c_float * len(flat))(*flat), len(flat) // 3


def muon_workspace_bytes(K: int, A: int, B: int) -> int:
    return int(lib().muon_workspace_bytes(K, A, B))


def make_muon_hparams(lr, momentum, weight_decay, nesterov=True, cautious_wd=False, scale_mode=0,
                      coeffs=((3.4445, -4.7750, 2.0315),) * 5, eps=1e-7):
    arr, steps = _coeff_array(coeffs)
    hp = muon_hparams(lr, momentum, weight_decay, int(bool(nesterov)), int(bool(cautious_wd)), int(scale_mode), steps,
                      ctypes.cast(arr, ctypes.POINTER(ctypes.c_float)), eps)
    hp._keep = arr  # the coefficient array lives as long as the struct
    return hp


def muon_step_batched(param_ptrs, pdt: int, grad_ptrs, gdt: int, momentum, K: int, A: int, B: int,
                      hp: muon_hparams, ws, stream=None):
    """param_ptrs / grad_ptrs: device int64 tensors of K data pointers (see pointer_array)."""
    st = lib().muon_step_batched(param_ptrs.data_ptr(), pdt, grad_ptrs.data_ptr(), gdt, momentum.data_ptr(), K, A, B,
                                 ctypes.byref(hp), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "muon_step_batched")


def make_buckets(specs):
    """specs: sequence of (param_ptrs, grad_ptrs, momentum, K, A, B, pdt, gdt[, master_ptrs]); returns a ctypes
    muon_bucket array. master_ptrs (optional): device array of K pointers to fp32 master copies.

    The array keeps the tensors it points at alive (its `tensors` attribute): a pointer array built inline
    in the call would otherwise be freed on return, and its memory could be reused before the GPU reads it."""
    arr = (muon_bucket * len(specs))()
    keep = []
    for i, spec in enumerate(specs):
        pp, gp, mom, K, A, B, pdt, gdt = spec[:8]
        mp = spec[8] if len(spec) > 8 else None
        keep += [pp, gp, mom] + ([mp] if mp is not None else [])
        arr[i] = muon_bucket(pp.data_ptr(), gp.data_ptr(), mom.data_ptr(), K, A, B, pdt, gdt,
                             mp.data_ptr() if mp is not None else None)
    arr.tensors = keep
    return arr


def muon_workspace_bytes_grouped(buckets) -> int:
    return int(lib().muon_workspace_bytes_grouped(buckets, len(buckets)))


def muon_step_grouped(buckets, hp: muon_hparams, ws, stream=None):
    """buckets: a ctypes muon_bucket array (see make_buckets)."""
    st = lib().muon_step_grouped(buckets, len(buckets), ctypes.byref(hp), ws.data_ptr(),
                                 ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "muon_step_grouped")


def pointer_array(tensors, device):
    """Device int64 tensor holding each tensor's data pointer (the K-pointer arrays muon_step_batched reads)."""
    import torch
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=device)


def ns_orthogonalize(x, out, coeffs, eps: float, ws, stream=None):
    """x, out: contiguous (K, A, B) float32 or bfloat16 device tensors."""
    K, A, B = x.shape
    arr, steps = _coeff_array(coeffs)
    st = lib().ns_orthogonalize(x.data_ptr(), _dtype_code(x), out.data_ptr(), _dtype_code(out), K, A, B, steps,
                                arr, eps, ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream))
    _check(st, "ns_orthogonalize")


def ns_orthogonalize_noalloc(x, out, coeffs, eps: float, stream=None):
    """ns_orthogonalize for callers that cannot allocate device memory: no workspace argument; the library's
    built-in 64 MiB scratch is used instead (see include/libmuon.h for the limits and the sharing rules)."""
    K, A, B = x.shape
    arr, steps = _coeff_array(coeffs)
    st = lib().ns_orthogonalize_noalloc(x.data_ptr(), _dtype_code(x), out.data_ptr(), _dtype_code(out), K, A, B,
                                        steps, arr, eps, _stream(stream))
    _check(st, "ns_orthogonalize_noalloc")


def ns_orthogonalize_noalloc_check(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the built-in scratch's sticky error status:
    MUON_ERR_TIMEOUT if a bounded wait of an ns_orthogonalize_noalloc call ran out since the last check."""
    return int(lib().ns_orthogonalize_noalloc_check(_stream(stream)))


def muon_debug_wait_timeout_noalloc(timeout_ns: int, stream=None):
    _check(lib().muon_debug_wait_timeout_noalloc(int(timeout_ns), _stream(stream)), "muon_debug_wait_timeout_noalloc")


def adamw_step(param, grad, exp_avg, exp_avg_sq, lr, beta1, beta2, eps, weight_decay, step: int, stream=None,
               l2: bool = False):
    """l2=False: AdamW (decoupled decay). l2=True: Adam with L2 regularisation (wd*p added to the gradient)."""
    hp = adamw_hparams(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay, l2=int(bool(l2)),
                       step=int(step))
    st = lib().adamw_step(param.data_ptr(), _dtype_code(param), grad.data_ptr(), _dtype_code(grad),
                          exp_avg.data_ptr(), exp_avg_sq.data_ptr(), param.numel(), ctypes.byref(hp), _stream(stream))
    _check(st, "adamw_step")


def adamw_step_master(master, param, grad, exp_avg, exp_avg_sq, lr, beta1, beta2, eps, weight_decay, step: int,
                      stream=None, l2: bool = False):
    """adamw_step on fp32 master weights; the bf16 param receives the new master rounded to bf16."""
    if _dtype_code(param) != MUON_BF16 or _dtype_code(master) != MUON_F32 or master.numel() != param.numel():
        raise ValueError("adamw_step_master: fp32 master and bf16 param of the same size")
    hp = adamw_hparams(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay, l2=int(bool(l2)),
                       step=int(step))
    st = lib().adamw_step_master(master.data_ptr(), param.data_ptr(), grad.data_ptr(), _dtype_code(grad),
                                 exp_avg.data_ptr(), exp_avg_sq.data_ptr(), param.numel(), ctypes.byref(hp),
                                 _stream(stream))
    _check(st, "adamw_step_master")


def make_adamw_hparams(lr, beta1, beta2, eps, weight_decay, step: int, l2: bool = False) -> adamw_hparams:
    return adamw_hparams(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=weight_decay, l2=int(bool(l2)),
                         step=int(step))


def make_adamw_tensors(specs):
    """specs: sequence of (param, grad, exp_avg, exp_avg_sq, hp[, master]) with hp an adamw_hparams; returns a
    ctypes adamw_tensor array that keeps the tensors and the hparams structs it points at alive."""
    arr = (adamw_tensor * len(specs))()
    keep = []
    for i, spec in enumerate(specs):
        p, g, m, v, hp = spec[:5]
        ms = spec[5] if len(spec) > 5 else None
        if ms is not None and (_dtype_code(p) != MUON_BF16 or _dtype_code(ms) != MUON_F32 or ms.numel() != p.numel()):
            raise ValueError("make_adamw_tensors: a master copy needs bf16 params and an fp32 master of their size")
        keep += [p, g, m, v, hp] + ([ms] if ms is not None else [])
        arr[i] = adamw_tensor(p.data_ptr(), g.data_ptr(), m.data_ptr(), v.data_ptr(),
                              ms.data_ptr() if ms is not None else None, p.numel(), _dtype_code(p), _dtype_code(g),
                              ctypes.pointer(hp))
    arr.tensors = keep
    return arr


def adamw_workspace_bytes_grouped(n: int) -> int:
    return int(lib().adamw_workspace_bytes_grouped(int(n)))


def adamw_step_grouped(tensors, ws, stream=None):
    """tensors: a ctypes adamw_tensor array (see make_adamw_tensors)."""
    _check(lib().adamw_step_grouped(tensors, len(tensors), ws.data_ptr(), ws.numel() * ws.element_size(),
                                    _stream(stream)), "adamw_step_grouped")


def hybrid_step(buckets, hp, ws, tensors, adamw_ws, stream=None):
    """buckets (make_buckets) with hp / ws as for muon_step_grouped, tensors (make_adamw_tensors) with adamw_ws as
    for adamw_step_grouped; either list may be empty."""
    nb = len(buckets) if buckets is not None else 0
    nt = len(tensors) if tensors is not None else 0
    _check(lib().hybrid_step(buckets if nb else None, nb, ctypes.byref(hp) if hp is not None else None,
                             ws.data_ptr() if ws is not None else None,
                             ws.numel() * ws.element_size() if ws is not None else 0, tensors if nt else None, nt,
                             adamw_ws.data_ptr() if adamw_ws is not None else None,
                             adamw_ws.numel() * adamw_ws.element_size() if adamw_ws is not None else 0,
                             _stream(stream)), "hybrid_step")


def ns_gram(x, g, alpha: float, ws, stream=None):
    K, m, n = x.shape
    _check(lib().ns_gram(x.data_ptr(), g.data_ptr(), K, m, n, alpha, ws.data_ptr(), ws.numel() * ws.element_size(),
                         _stream(stream)), "ns_gram")


def ns_poly(g, h, a: float, b: float, c: float, ws, stream=None):
    """h = a*I + b*g + c*g g."""
    K, m, _ = g.shape
    _check(lib().ns_poly(g.data_ptr(), h.data_ptr(), K, m, a, b, c, ws.data_ptr(), ws.numel() * ws.element_size(),
                         _stream(stream)), "ns_poly")


def ns_apply(h, x, out, ws, stream=None):
    """out = h x."""
    K, m, n = x.shape
    _check(lib().ns_apply(h.data_ptr(), x.data_ptr(), out.data_ptr(), K, m, n, ws.data_ptr(),
                          ws.numel() * ws.element_size(), _stream(stream)), "ns_apply")


def muon_plan_buckets(shapes: Sequence[Tuple[int, int]]):
    n = len(shapes)
    L = ctypes.c_int64 * max(n, 1)
    rows = L(*[int(s[0]) for s in shapes])
    cols = L(*[int(s[1]) for s in shapes])
    bid, idx, K, off = L(), L(), L(), L()
    shp = (ctypes.c_int64 * max(2 * n, 2))()
    nb = ctypes.c_int64(0)
    _check(lib().muon_plan_buckets(n, rows, cols, bid, idx, ctypes.byref(nb), shp, K, off), "muon_plan_buckets")
    b = nb.value
    return {
        "bucket_id": list(bid)[:n],
        "index_in_bucket": list(idx)[:n],
        "bucket_shapes": [(shp[2 * i], shp[2 * i + 1]) for i in range(b)],
        "bucket_K": list(K)[:b],
        "momentum_offset": list(off)[:b],
    }


def muon_autotune(buckets, hp, ws, stream=None):
    """Measures, on the workspace alone, each eligible bucket's Newton-Schulz path, the poly step's pipeline shape
    and the plain chain's scheduling for these buckets and hyperparameters, and records the fastest (synchronous)."""
    _check(lib().muon_autotune(buckets, len(buckets), ctypes.byref(hp), ws.data_ptr(), ws.numel() * ws.element_size(),
                               _stream(stream)), "muon_autotune")


def muon_autotune_route(K: int, A: int, B: int) -> int:
    """The recorded path: 1 Gram space, 0 plain chain, -1 none."""
    return int(lib().muon_autotune_route(int(K), int(A), int(B)))


def muon_autotune_scheduling(buckets) -> int:
    """The recorded scheduling of these buckets' plain chain: 1 counters, 0 launch order, -1 none."""
    return int(lib().muon_autotune_scheduling(buckets, len(buckets)))


def muon_autotune_poly_shape(contraction: int) -> int:
    return int(lib().muon_autotune_poly_shape(int(contraction)))


def muon_autotune_gram_split(K: int, A: int, B: int) -> int:
    """The recorded contraction slices of the Gram-space fp32 Gram of a K x A x B stack, or -1."""
    return int(lib().muon_autotune_gram_split(int(K), int(A), int(B)))


def muon_debug_piece_elems(elems: int):
    """Matrix elements per piece of every Muon call (0: the default)."""
    _check(lib().muon_debug_piece_elems(int(elems)), "muon_debug_piece_elems")


def muon_autotune_reset():
    lib().muon_autotune_reset()


def muon_debug_poly_shape(shape: int):
    _check(lib().muon_debug_poly_shape(int(shape)), "muon_debug_poly_shape")


def muon_debug_counter_deps(mode: int):
    """1: counter dependencies in the grouped chain, 0: launch order, -1: the library's rule (default)."""
    _check(lib().muon_debug_counter_deps(int(mode)), "muon_debug_counter_deps")


def muon_debug_half_symmetric(on: int):
    """1: the chain stores G and H as their upper 256-blocks only (default), 0: whole. Same results."""
    _check(lib().muon_debug_half_symmetric(int(on)), "muon_debug_half_symmetric")


def muon_debug_gram_space(mode: int):
    """Gram-space Newton-Schulz path: -1 the library's rule (default), 0 never, 1 wherever the shape allows it."""
    _check(lib().muon_debug_gram_space(int(mode)), "muon_debug_gram_space")


def muon_debug_gram_split(split: int):
    """Contraction slices of the Gram-space fp32 Gram: 1 .. 8 forced, -1 the table and the rule (default)."""
    _check(lib().muon_debug_gram_split(int(split)), "muon_debug_gram_split")


def muon_gram_space_route(A: int, B: int, K: int = 1) -> bool:
    return bool(lib().muon_gram_space_route(int(K), int(A), int(B)))


def muon_check(ws, stream=None) -> int:
    return int(lib().muon_check(ws.data_ptr(), _stream(stream)))


def muon_set_timeout_ns(ns: int):
    lib().muon_set_timeout_ns(int(ns))


def muon_debug_wait_timeout(ws, timeout_ns: int, stream=None):
    _check(lib().muon_debug_wait_timeout(ws.data_ptr(), ws.numel() * ws.element_size(), int(timeout_ns),
                                         _stream(stream)), "muon_debug_wait_timeout")


def muon_debug_timeline(buf, records_per_cta: int):
    """Registers (or, with buf None, unregisters) a device buffer for per-tile GEMM timestamps."""
    if buf is None:
        _check(lib().muon_debug_timeline(None, 0, 0), "muon_debug_timeline")
    else:
        _check(lib().muon_debug_timeline(buf.data_ptr(), buf.numel() * buf.element_size(), records_per_cta),
               "muon_debug_timeline")


def muon_launch_count() -> int:
    return int(lib().muon_launch_count())


def muon_trace_enable(on: bool):
    lib().muon_trace_enable(int(bool(on)))


def muon_trace_collect(cap: int = 65536):
    kinds = (ctypes.c_int32 * cap)()
    ms = (ctypes.c_float * cap)()
    n = int(lib().muon_trace_collect(kinds, ms, cap))
    if n < 0:
        raise MuonError(MUON_ERR_CUDA, "muon_trace_collect")
    return [(muon_kernel_name(kinds[i]), float(ms[i])) for i in range(n)]


def muon_kernel_name(kind: int) -> str:
    return lib().muon_kernel_name(int(kind)).decode()
