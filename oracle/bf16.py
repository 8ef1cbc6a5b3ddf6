"""Round float values to bfloat16 (round to nearest, ties to even), returned as float64.

A stored bf16 parameter is part of the method's state when parameters are kept in
bf16 with no fp32 master copy; the oracle rounds its fp64 result the way a bf16 store
does. Written from the bfloat16 format itself: 8 significant bits (1 implicit + 7
stored), the binary32 exponent range, subnormal spacing 2**-133, largest finite value
(2 - 2**-7) * 2**127. The rounding is done once, straight from float64.
Pinned in tests against torch's conversion to bfloat16.
"""
import numpy as np

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
_BF16_SUBNORMAL_SPACING_EXP = -133


def round_bf16(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0)
    xf = x[finite]
    _, e = np.frexp(xf)                                   # xf = m * 2**e, 0.5 <= |m| < 1
    spacing_exp = np.maximum(e - 8, _BF16_SUBNORMAL_SPACING_EXP)
    spacing = np.ldexp(1.0, spacing_exp)
    r = np.round(xf / spacing) * spacing                  # exact scaling; np.round ties to even
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, xf), r)
    out[finite] = r
    return out


def round_f32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to(x, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_bf16(x)
    if dtype == "f32":
        return round_f32(x)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(dtype)
