"""Deterministic score bounds from the 4-bit keys (float32, bit-exact).

picx.dev summary, "Algorithm Components" 4: the 4-bit scan (int8 dot
products, AVX-512 VNNI on the pages' CPU) gives deterministic upper bounds
u_i >= s_i for every score s_i = q.k_i / sqrt(d) ("Problem Setup").  The
pages do not print the bound; the one used here follows from the quantiser
(``quantize.py``) and an integer query code:

  per query head and block, with rs = fl(1/sqrt d), qt_c = fl(q_c * rs):
    a_c   = fl(qt_c * Delta_c)
    amax  = max_c |a_c|;  alpha = fl(amax / QM);  inv = fl(QM / amax)
            (alpha = inv = 0 when amax = 0)
    at_c  = clamp(rint(fl(a_c * inv)), -QM, QM)         integer query code
    r_c   = fl(a_c - fl(alpha * at_c))                  its residual
    Bq    = tree(fl(qt_c * m_c))                        offset term
    A1    = tree(|a_c|);  Rp = tree(max(r_c,0));  Rn = tree(max(-r_c,0))
    sk    = fl(A1 * (1/2 + 2^-16))                      key-rounding slack
    hi    = fl(sk + fl(15 * Rp));   lo = fl(sk + fl(15 * Rn))
    Q1    = tree(|qt_c|);  Kabs = max_c fl(|m_c| + 16 Delta_c)
    marg  = fl(fl(fl(fl(Q1 * Kabs) + hi) + lo) * 2^-14)  float32 safety
    b_hi  = fl(fl(Bq + hi) + marg);   b_lo = fl(fl(Bq - lo) - marg)
  per key i of the block, I_i = sum_c at_c * code_ic  (exact integer):
    ubar_i = fl(fl(alpha * I_i) + b_hi),   l_i = fl(fl(alpha * I_i) + b_lo)

``tree`` is the adjacent-pair float32 tree of ``fp32.tree_sum_f32``.
Why it bounds s_i: k_ic = m_c + code_ic Delta_c + e_ic with
|e_ic| <= Delta_c (1/2 + 2^-16), and sum_c a_c code_c = alpha I_i +
sum_c r_c code_c with 0 <= code <= 15; every float32 rounding above is at most
2^-24 relative to a quantity bounded by Q1 * Kabs, far inside marg.
QM = 127 (int8 codes, as for the pages' u8 x s8 dot products).  Option:
two-digit codes, QM = QM_TWO_DIGIT = 127 * 257 (at = 256 hi + lo, two s8
digits), with both residual terms replaced by the closed form
fl(fl(15 d) * fl(alpha * (1/2 + 2^-6))) (see ``query_prep``).
Test infrastructure only.
"""
from __future__ import annotations

import math

import numpy as np

from .fp32 import tree_sum_f32

F = np.float32
QM_DEFAULT = 127
# two signed 8-bit digits per query code: at = 256 hi + lo, |hi|, |lo| <= 127
QM_TWO_DIGIT = 127 * 257
_RES_HALF = F(0.5 + 2.0 ** -6)
_RHO = F(0.5 + 2.0 ** -16)
_MARG = F(2.0 ** -14)


def inv_sqrt_d_f32(d: int) -> np.float32:
    return F(1.0 / math.sqrt(d))


def query_prep(q: np.ndarray, mins: np.ndarray, deltas: np.ndarray,
               QM: int = QM_DEFAULT, levels: int = 15,
               closed_residual: bool = False):
    """Per-block query code for one query head.

    q float32 [d]; mins, deltas float32 [nblk, d]; `levels` the largest key
    code (15 for the 4-bit keys; 255 for the 8-bit refinement codes, whose
    bound is the same construction with 15 -> 255 and 16 -> 256, best with
    a finer query code, QM = 2047: with QM = 127 the query residual term
    levels * sum |r_c| outweighs the 8-bit keys' rounding slack).
    With ``closed_residual`` the two residual trees give way to a closed
    form, meant for fine query codes (QM_TWO_DIGIT): a_c - alpha at_c is
    within 1/2 + 2^-6 of alpha per channel (rint's half step, plus the
    float32 roundings of inv, a_c inv and alpha, each at most QM 2^-23
    relative to alpha), so both residual terms are replaced by
    fl(fl(levels d) * fl(alpha * (1/2 + 2^-6))).
    Returns (at int32 [nblk, d], alpha f32 [nblk], b_hi f32 [nblk],
    b_lo f32 [nblk]).
    """
    assert not closed_residual or QM <= QM_TWO_DIGIT
    q = np.asarray(q, dtype=np.float32)
    d = q.shape[0]
    qt = q * inv_sqrt_d_f32(d)
    a = qt[None, :] * deltas
    amax = np.abs(a).max(axis=1)
    pos = amax > F(0.0)
    safe = np.where(pos, amax, F(1.0)).astype(np.float32)
    alpha = np.where(pos, safe / F(QM), F(0.0)).astype(np.float32)
    inv = np.where(pos, F(QM) / safe, F(0.0)).astype(np.float32)
    at = np.clip(np.rint(a * inv[:, None]), -QM, QM).astype(np.float32)
    Bq = tree_sum_f32(qt[None, :] * mins)
    A1 = tree_sum_f32(np.abs(a))
    sk = A1 * _RHO
    if closed_residual:
        res = F(levels * d) * (alpha * _RES_HALF)
        hi = sk + res
        lo = sk + res
    else:
        r = a - alpha[:, None] * at
        Rp = tree_sum_f32(np.maximum(r, F(0.0)))
        Rn = tree_sum_f32(np.maximum(-r, F(0.0)))
        hi = sk + F(levels) * Rp
        lo = sk + F(levels) * Rn
    Q1 = tree_sum_f32(np.abs(qt))
    Kabs = (np.abs(mins) + F(levels + 1) * deltas).max(axis=1)
    mag = ((Q1 * Kabs) + hi) + lo
    marg = mag * _MARG
    b_hi = (Bq + hi) + marg
    b_lo = (Bq - lo) - marg
    return at.astype(np.int32), alpha, b_hi, b_lo


def key_bounds(codes: np.ndarray, at: np.ndarray, alpha: np.ndarray,
               b_hi: np.ndarray, b_lo: np.ndarray, n: int, T: int = 64):
    """ubar_i and l_i (float32 [n]) for the first n keys of one head.

    codes uint8 [>=n, d] unpacked; at int32 [nblk, d].
    """
    blk = np.arange(n) // T
    I = np.einsum("nd,nd->n", codes[:n].astype(np.int64),
                  at[blk].astype(np.int64))
    # |I| < 2^24 with int8 query codes, so I converts exactly; with
    # two-digit codes it may round (to nearest even), which the margin covers
    aI = alpha[blk] * I.astype(np.float32)
    ubar = aI + b_hi[blk]
    low = aI + b_lo[blk]
    return ubar.astype(np.float32), low.astype(np.float32), I
