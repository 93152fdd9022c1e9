"""IEEE float32 helpers for the bit-exact parts of the oracle.

Every operation is one numpy float32 operation, i.e. one correctly rounded
IEEE binary32 add, multiply or divide (numpy never fuses a multiply and an
add).  Test infrastructure only.
"""
from __future__ import annotations

import numpy as np

F = np.float32


def tree_sum_f32(x: np.ndarray) -> np.ndarray:
    """Pairwise float32 sum over the last axis (length a power of two).

    The order is the adjacent-pair tree: at every level element ``2i`` and
    element ``2i+1`` are added.  This is the summation order the bound
    arithmetic fixes (the pages leave the order open; the deterministic
    bounds of "Algorithm Components" 4 need *some* fixed order to be
    reproducible).
    """
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[-1]
    if n & (n - 1):
        raise ValueError("tree_sum_f32 needs a power-of-two length")
    while x.shape[-1] > 1:
        x = x[..., 0::2] + x[..., 1::2]
    return x[..., 0]


# atanh series for log: ln f = 2 (z + z^3/3 + z^5/5 + ...), z = (f-1)/(f+1)
# (Abramowitz & Stegun 4.1.27).  On f in [1/sqrt2, sqrt2], |z| <= 0.1716 and
# the first omitted term (z^11/11) is below 2e-9 relative.
_C3 = F(1.0 / 3.0)
_C5 = F(1.0 / 5.0)
_C7 = F(1.0 / 7.0)
_C9 = F(1.0 / 9.0)
_K2 = F(2.0 / np.log(2.0))        # 2 / ln 2
_SQRT2 = F(np.sqrt(2.0))


def log2_m53_f32(m: np.ndarray) -> np.ndarray:
    """float32 log2(m) for integers m in [1, 2^53] (uint64 array).

    Steps: e = floor(log2 m) from the bit length; the top 24 bits of m give
    the float32 mantissa f in [1, 2) (truncation); f > sqrt2 is halved
    (e += 1); then log2 f = (2/ln2) * atanh-series(z), z = (f-1)/(f+1),
    Horner in z^2 with separate float32 multiplies and adds.
    Returns e + log2 f rounded to float32.
    """
    m = np.asarray(m, dtype=np.uint64)
    if np.any(m == 0):
        raise ValueError("log2 of zero")
    # bit length via float64 frexp is exact for m <= 2^53
    _, ex = np.frexp(m.astype(np.float64))
    e = ex.astype(np.int64) - 1                       # floor(log2 m)
    shift = np.maximum(e - 23, 0)
    top = (m >> shift.astype(np.uint64)).astype(np.float32)   # < 2^24, exact
    f = np.ldexp(top, -(e - shift)).astype(np.float32)        # exact, [1, 2)
    big = f > _SQRT2
    f = np.where(big, f * F(0.5), f).astype(np.float32)
    e = e + big.astype(np.int64)
    z = (f - F(1.0)) / (f + F(1.0))
    z2 = z * z
    p = _C9 * z2
    p = p + _C7
    p = p * z2
    p = p + _C5
    p = p * z2
    p = p + _C3
    p = p * z2
    p = p + F(1.0)
    l2f = (z * p) * _K2
    return e.astype(np.float32) + l2f
