"""GB300-native hybrid Muon + AdamW optimizer step.

libmuon (C ABI, CUDA kernels for sm_103a) does the work; this package holds its ctypes binding
(``libmuon``), the build step (``_build``) and the param_groups optimizer (``HybridMuonAdamW``).
"""
from . import libmuon
from .libmuon import MuonError


def __getattr__(name):
    if name == "HybridMuonAdamW":
        from .optim import HybridMuonAdamW
        return HybridMuonAdamW
    raise AttributeError(name)


__all__ = ["libmuon", "MuonError", "HybridMuonAdamW"]
