"""Pins for the two-digit query codes of the 4-bit bounds (an option of the
oracle's bound construction; picx.dev summary, "Algorithm Components" 4
fixes only that the bounds are deterministic).

The query code per (block, head) is an integer at_c in [-QM, QM] with
QM = 127 * 257, held as two signed 8-bit digits at_c = 256 hi_c + lo_c so
that each digit fits the u8 x s8 integer products of the scan.  The finer
code leaves a residual a_c - alpha at_c within (1/2 + 2^-6) alpha per
channel, so the two residual trees of the int8 construction give way to a
closed form.  The pins: the digit split is exact and in range, the residual
bound holds (also at rounding ties and at the clamp), l <= s <= ubar on
ordinary, outlier-heavy and degenerate inputs, the interval is narrower
than with int8 codes, and the decode step's results do not change.
"""
import math

import numpy as np

import synth
from oracle.bounds import QM_TWO_DIGIT, _RES_HALF, key_bounds, query_prep
from oracle.quantize import quantize_keys
from oracle.step import Params, oracle_decode_group, score_f32

F = np.float32


def _digits(at):
    hi = np.floor_divide(at + 128, 256)
    return hi, at - 256 * hi


def test_digit_split_exact_and_in_range():
    at = np.arange(-QM_TWO_DIGIT, QM_TWO_DIGIT + 1, dtype=np.int64)
    hi, lo = _digits(at)
    assert np.all(256 * hi + lo == at)
    assert hi.min() >= -127 and hi.max() <= 127
    assert lo.min() >= -128 and lo.max() <= 127
    # I = 256 I_hi + I_lo: the split products recombine exactly
    rng = np.random.default_rng(0)
    a = rng.integers(-QM_TWO_DIGIT, QM_TWO_DIGIT + 1, (50, 128))
    codes = rng.integers(0, 16, (50, 128))
    h, l = _digits(a)
    assert np.array_equal(256 * (h * codes).sum(1) + (l * codes).sum(1),
                          (a * codes).sum(1))
    assert np.abs(a * codes).sum(1).max() < 2 ** 31


def _residual_ok(q, mins, deltas):
    at, alpha, _, _ = query_prep(q, mins, deltas, QM_TWO_DIGIT,
                                 closed_residual=True)
    d = q.shape[0]
    qt = (q * F(1.0 / math.sqrt(d))).astype(F)
    a = (qt[None, :] * deltas).astype(np.float64)
    r = a - alpha[:, None].astype(np.float64) * at
    bound = alpha.astype(np.float64)[:, None] * float(_RES_HALF)
    assert np.all(np.abs(r) <= bound), (np.abs(r) / np.maximum(bound, 1e-300)).max()
    assert np.abs(at).max() <= QM_TWO_DIGIT
    return at, alpha


def test_residual_within_closed_form():
    rng = np.random.default_rng(1)
    for trial in range(200):
        d = 128 if trial % 2 else 64
        q = (rng.standard_normal(d) * rng.lognormal(0, 2)).astype(F)
        deltas = rng.lognormal(-2, 1.5, (4, d)).astype(F)
        mins = rng.standard_normal((4, d)).astype(F)
        _residual_ok(q, mins, deltas)
    # exact ties: with amax = QM / 1024, inv = 1024 and alpha = 2^-10
    # exactly, so a_c = (k + 1/2) / 1024 scales to a half step and rint
    # leaves a residual of exactly alpha / 2; the first channel is amax
    # itself (the clamp)
    d = 64
    deltas = np.ones((1, d), F)
    a = (np.arange(d, dtype=np.float64) * 97.0 - 3000.0 + 0.5) / 1024.0
    a[0] = QM_TWO_DIGIT / 1024.0
    q = (a * 8.0).astype(F)               # qt = q / sqrt(64) = a exactly
    at, alpha = _residual_ok(q, np.zeros((1, d), F), deltas)
    assert alpha[0] == F(2.0 ** -10) and at[0, 0] == QM_TWO_DIGIT
    r = a[1:] - float(alpha[0]) * at[0, 1:]
    assert np.all(np.abs(r) == 2.0 ** -11)
    q = np.zeros(d, F)
    q[0] = 1.0
    q[1] = -1.0
    q[2] = F(0.5) + F(2.0 ** -20)
    _residual_ok(q, np.zeros((1, d), F), deltas)


def _check(q, K, n):
    codes, _, mins, deltas = quantize_keys(K, n)
    s = K[:n].astype(np.float64) @ q.astype(np.float64) / math.sqrt(q.shape[0])
    s32, _ = score_f32(q, K[:n])
    out = []
    for two in (False, True):
        if two:
            at, al, bh, bl = query_prep(q, mins, deltas, QM_TWO_DIGIT,
                                        closed_residual=True)
        else:
            at, al, bh, bl = query_prep(q, mins, deltas)
        ub, lo, _ = key_bounds(codes, at, al, bh, bl, n)
        assert np.all(lo.astype(np.float64) <= s) and np.all(ub >= s)
        assert np.all(ub >= s32) and np.all(lo <= s32)
        out.append((ub.astype(np.float64) - lo).mean())
    return out


def test_bounds_hold_and_are_narrower():
    w = synth.workload("llama16k", B=1, n=2000, Hq=8, Hkv=2)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, 0)
    ratios = []
    for g in range(w.Hkv):
        for h in range(w.G):
            w8, w2 = _check(q[0, g * w.G + h], K[0, g], w.n)
            ratios.append(w2 / w8)
    # on this recipe the residual term is about a third of the key-rounding
    # slack with int8 codes; two digits remove nearly all of it
    assert max(ratios) < 0.9 and min(ratios) > 0.6, ratios


def test_bounds_hold_on_adversarial_inputs():
    rng = np.random.default_rng(7)
    d = 128
    K = rng.standard_normal((256, d)).astype(F)
    K[:, 3] = 1e4 + K[:, 3]
    K[:, 9] *= 1000.0
    q = rng.standard_normal(d).astype(F)
    q[3] = 1e-3
    _check(q, K, 256)
    _check(np.zeros(d, F), K, 256)
    _check(q, np.tile(K[:1], (130, 1)), 130)
    # large |I|: every code at 15 and a query at the clamp in every channel
    K2 = np.zeros((64, d), F)
    K2[0] = 1.0
    _check(np.ones(d, F) * F(3.0), K2, 64)


def test_decode_step_results_unchanged():
    w = synth.workload("llama16k", B=1, n=3000, Hq=8, Hkv=2)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, 0)
    seed = int(synth.step_seeds(w, 0)[0])
    G = w.G
    fewer = 0
    for g in range(w.Hkv):
        args = (q[0, g * G:(g + 1) * G], K[0, g], V[0, g], w.n, seed, g)
        a = oracle_decode_group(*args, Params(w.eps, w.delta, w.r))
        b = oracle_decode_group(*args, Params(w.eps, w.delta, w.r,
                                              two_digit=True))
        assert np.array_equal(a.o, b.o) and np.array_equal(a.beta, b.beta)
        assert np.array_equal(a.level, b.level)
        assert np.array_equal(a.values_read, b.values_read)
        fewer += int(a.keys_read.sum() - b.keys_read.sum())
    assert fewer > 0
