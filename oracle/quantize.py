"""4-bit per-block, per-channel key quantiser and value-norm metadata.

picx.dev summary, "Algorithm Components" 4: keys are quantised to 4 bits per
block and per channel (as in KIVI), and the scan over those codes gives
deterministic score bounds.  The pages give neither the block length nor the
rounding rule; the readings taken here:
  * block = T = 64 consecutive token positions, aligned to position 0;
    a partial last block is quantised over the tokens present;
  * per (block, channel c): m_c = min, M_c = max (float32),
    Delta_c = fl((M_c - m_c) / 15), replaced by 1 when it is 0;
    code = clamp(rint(fl(fl(k - m_c) / Delta_c)), 0, 15), ties to even;
  * two codes per byte, the even channel in the low nibble.
Each code satisfies |k - m_c - code * Delta_c| <= Delta_c (1/2 + 2^-16),
the rounding of the float32 ops included (see ``bounds.py``).

Value-norm metadata (not on the pages; needed by the certificate's range
constants): per block, vmax = max_i ||v_i|| over the tokens present, with
||v|| = sqrt of the sequential float32 sum of v_c^2 (c = 0, 1, ...), then
multiplied by (1 + 2^-16) so that it is an upper bound despite rounding.
Test infrastructure only.
"""
from __future__ import annotations

import numpy as np

F = np.float32
T_BLOCK = 64
_VMAX_UP = F(1.0 + 2.0 ** -16)


def _quantize(K: np.ndarray, n: int, T: int, levels: int):
    """Per-block per-channel quantiser with codes 0..levels (the rule in the
    module docstring, with `levels` in place of 15)."""
    K = np.asarray(K, dtype=np.float32)
    d = K.shape[1]
    nblk = (n + T - 1) // T
    codes = np.zeros((nblk * T, d), np.uint8)
    mins = np.zeros((nblk, d), np.float32)
    deltas = np.zeros((nblk, d), np.float32)
    for blk in range(nblk):
        a, b = blk * T, min(blk * T + T, n)
        rows = K[a:b]
        m = rows.min(axis=0)
        M = rows.max(axis=0)
        dl = (M - m) / F(levels)
        dl = np.where(dl == F(0.0), F(1.0), dl).astype(np.float32)
        x = (rows - m[None, :]) / dl[None, :]
        c = np.clip(np.rint(x), 0, levels)
        codes[a:b] = c.astype(np.uint8)
        mins[blk] = m
        deltas[blk] = dl
    return codes, mins, deltas


def quantize_keys(K: np.ndarray, n: int, T: int = T_BLOCK):
    """Quantise the first n rows of K (float32 [>=n, d]) to 4 bits.

    Returns (codes uint8 [nblk*T, d] unpacked, packed uint8 [nblk*T, d/2],
    mins float32 [nblk, d], deltas float32 [nblk, d]).
    Rows at positions >= n get code 0.
    """
    codes, mins, deltas = _quantize(K, n, T, 15)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return codes, packed, mins, deltas


def quantize_keys8(K: np.ndarray, n: int, T: int = T_BLOCK):
    """8-bit codes of the same blocks (picx.dev "Algorithm Components" 4:
    "8-bit refinement" before the exact 16-bit reads; the pages give no
    detail, so the 4-bit rule with 255 levels: Delta8_c = fl((M_c -
    m_c) / 255), code = clamp(rint(fl(fl(k - m_c) / Delta8_c)), 0, 255)).
    Returns (codes uint8 [nblk*T, d], mins, deltas8)."""
    return _quantize(K, n, T, 255)


def value_sq_norms_f32(V: np.ndarray, n: int) -> np.ndarray:
    """||v_i||^2 of the first n value rows as the sequential float32 sum of
    v_c^2 over the channels c = 0, 1, ... (float32 [n]).  The value norms
    enter the Hilbert-space Bernstein bound and the value scale M of the
    certificate (picx.dev "Algorithm Components" 3)."""
    V = np.asarray(V[:n], dtype=np.float32)
    d = V.shape[1]
    ss = np.zeros(V.shape[0], np.float32)
    for c in range(d):
        ss = ss + V[:, c] * V[:, c]
    return ss


def vmax_blocks(V: np.ndarray, n: int, T: int = T_BLOCK) -> np.ndarray:
    """Per-block upper bound on ||v_i|| (float32 [nblk])."""
    ss = value_sq_norms_f32(V, n)
    nrm = np.sqrt(ss).astype(np.float32)
    nblk = (n + T - 1) // T
    out = np.zeros(nblk, np.float32)
    for blk in range(nblk):
        out[blk] = nrm[blk * T:min(blk * T + T, n)].max() * _VMAX_UP
    return out
