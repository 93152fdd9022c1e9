"""Pins for the 4-bit quantiser and the deterministic score bounds.

picx.dev summary, "Algorithm Components" 4: 4-bit per-block per-channel key
codes give deterministic upper bounds u_i >= s_i for every score.  The pins
check the defining inequalities against float64 scores on ordinary,
outlier-heavy and degenerate inputs, the integer dot product by brute force,
and the grid size J = ceil(r log2 |P|) by exact integer comparison.
"""
import math

import numpy as np
import pytest

import synth
from oracle.bounds import key_bounds, query_prep
from oracle.quantize import quantize_keys, value_sq_norms_f32, vmax_blocks
from oracle.step import grid_J, score_f32, cstar_lower_f32


def _exact_scores(q, K):
    return K.astype(np.float64) @ q.astype(np.float64) / math.sqrt(q.shape[0])


def _check_bounds(q, K, n, QM=127):
    codes, packed, mins, deltas = quantize_keys(K, n)
    at, alpha, b_hi, b_lo = query_prep(q, mins, deltas, QM)
    ub, lo, I = key_bounds(codes, at, alpha, b_hi, b_lo, n)
    s = _exact_scores(q, K[:n])
    assert np.all(lo.astype(np.float64) <= s), (s - lo).min()
    assert np.all(ub.astype(np.float64) >= s), (ub - s).min()
    # the float32 rescoring used on the device stays inside the bounds too
    s32, _ = score_f32(q, K[:n])
    assert np.all(ub >= s32) and np.all(lo <= s32)
    assert np.abs(at).max() <= QM
    return ub, lo, s


def test_quantizer_error_bound_and_codes():
    rng = np.random.default_rng(0)
    n, d = 1000, 64
    K = (rng.standard_normal((n, d)) * rng.lognormal(0, 2, d)).astype(
        np.float32)
    codes, packed, mins, deltas = quantize_keys(K, n)
    assert codes.max() <= 15
    blk = np.arange(n) // 64
    recon = mins[blk].astype(np.float64) + codes[:n] * deltas[blk].astype(
        np.float64)
    err = np.abs(K.astype(np.float64) - recon)
    assert np.all(err <= deltas[blk] * (0.5 + 2.0 ** -16))
    # packing: low nibble = even channel
    assert np.array_equal(packed[:n] & 15, codes[:n, 0::2])
    assert np.array_equal(packed[:n] >> 4, codes[:n, 1::2])
    # partial last block: 1000 = 15*64 + 40 rows
    assert mins.shape[0] == 16
    assert np.array_equal(mins[15], K[960:1000].min(axis=0))


def test_quantizer_constant_channel_and_tiny_range():
    K = np.ones((64, 8), np.float32) * 3.0
    K[:, 1] = np.linspace(0, 1e-44, 64, dtype=np.float32)  # subnormal range
    codes, _, mins, deltas = quantize_keys(K, 64)
    assert deltas[0, 0] == 1.0 and np.all(codes[:, 0] == 0)
    assert np.all(np.isfinite(deltas))


def test_vmax_is_upper_bound():
    rng = np.random.default_rng(3)
    V = (rng.standard_normal((300, 128)) * 7).astype(np.float32)
    vm = vmax_blocks(V, 300)
    nrm = np.linalg.norm(V.astype(np.float64), axis=1)
    for b in range(5):
        assert vm[b] >= nrm[b * 64:(b + 1) * 64].max()
        assert vm[b] <= nrm[b * 64:(b + 1) * 64].max() * (1 + 1e-4)


def test_value_sq_norms_exact_cases_and_error():
    # small integers: every partial sum is exact in float32
    V = np.array([[3, 4, 0, 0], [1, 1, 1, 1], [0, 0, 0, 12]], np.float32)
    assert value_sq_norms_f32(V, 3).tolist() == [25.0, 4.0, 144.0]
    assert value_sq_norms_f32(V, 2).shape == (2,)
    # against float64 within the sequential-sum error bound d * 2^-24
    rng = np.random.default_rng(7)
    W = (rng.standard_normal((200, 128)) * 5).astype(np.float32)
    ss = value_sq_norms_f32(W, 200).astype(np.float64)
    ref = (W.astype(np.float64) ** 2).sum(axis=1)
    assert np.all(np.abs(ss - ref) <= 128 * 2.0 ** -24 * ref)
    # the block bound is built from the same sums
    vm = vmax_blocks(W, 200)
    for b in range(4):
        top = np.sqrt(ss[b * 64:(b + 1) * 64].astype(np.float32)).max()
        assert vm[b] == np.float32(top) * np.float32(1 + 2.0 ** -16)


def test_integer_dot_brute_force():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((70, 64)).astype(np.float32)
    q = rng.standard_normal(64).astype(np.float32)
    codes, _, mins, deltas = quantize_keys(K, 70)
    at, alpha, b_hi, b_lo = query_prep(q, mins, deltas)
    _, _, I = key_bounds(codes, at, alpha, b_hi, b_lo, 70)
    for i in (0, 13, 63, 64, 69):
        ref = sum(int(at[i // 64, c]) * int(codes[i, c]) for c in range(64))
        assert I[i] == ref


@pytest.mark.parametrize("name", ["tiny", "llama16k"])
def test_bounds_on_workloads(name):
    w = synth.workload(name, B=1, n=700, Hq=8, Hkv=2)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, 0, K=K)
    for g in range(w.Hkv):
        for h in range(w.G):
            _check_bounds(q[0, g * w.G + h], K[0, g], w.n)


def test_bounds_adversarial_inputs():
    rng = np.random.default_rng(7)
    d = 128
    # huge outlier channels, offsets far from zero, near-cancelling scores
    K = rng.standard_normal((256, d)).astype(np.float32)
    K[:, 3] = 1e4 + K[:, 3]
    K[:, 9] *= 1000.0
    q = rng.standard_normal(d).astype(np.float32)
    q[3] = 1e-3
    _check_bounds(q, K, 256)
    # zero query: every score is 0 and both bounds equal 0
    ub, lo, s = _check_bounds(np.zeros(d, np.float32), K, 256)
    assert np.all(ub == 0) and np.all(lo == 0)
    # all-equal keys
    _check_bounds(q, np.tile(K[:1], (130, 1)), 130)
    # tiny magnitudes
    _check_bounds(q * 1e-20, K * 1e-10, 256)


@pytest.mark.parametrize("QM", [7, 127, 2047])
def test_bounds_any_query_code_width(QM):
    rng = np.random.default_rng(11)
    K = (rng.standard_normal((512, 64)) * 3).astype(np.float32)
    q = rng.standard_normal(64).astype(np.float32)
    ub, lo, s = _check_bounds(q, K, 512, QM)
    if QM == 2047:
        ub8, _, _ = _check_bounds(q, K, 512, 127)
        assert np.mean(ub - s) < np.mean(ub8 - s)   # finer code: tighter


def test_cstar_lower_bound():
    rng = np.random.default_rng(5)
    for _ in range(20):
        K = (rng.standard_normal((200, 128)) * rng.lognormal(0, 1)).astype(
            np.float32)
        q = rng.standard_normal(128).astype(np.float32)
        cb = cstar_lower_f32(q, K)
        cs = _exact_scores(q, K).max()
        assert cb <= cs and cs - cb < 1e-2 * (1 + abs(cs))


@pytest.mark.parametrize("P,r", [(1, 2), (2, 2), (3, 2), (1984, 2),
                                 (16320, 2), (131008, 4), (1 << 17, 4),
                                 ((1 << 17) + 1, 4), (1048512, 2), (5, 3)])
def test_grid_J(P, r):
    J = grid_J(P, r)
    if P <= 1:
        assert J == 0
        return
    # smallest integer with 2^J >= P^r, i.e. tau_J = 2^(-J/r) <= 1/|P|
    assert 2 ** J >= P ** r and 2 ** (J - 1) < P ** r
    if P & (P - 1):
        assert J == math.ceil(r * math.log2(P))
    else:
        assert J == r * (P.bit_length() - 1)


def test_bound_tight_for_aligned_key_rounding():
    # Worst case for the key-rounding slack: every channel of the probe key
    # sits just below / above a rounding midpoint, with the rounding error's
    # sign matching the query's sign, so q.e reaches ~ sum |q_c| Delta_c / 2.
    rng = np.random.default_rng(13)
    d = 64
    q = rng.standard_normal(d).astype(np.float32)
    K = np.zeros((64, d), np.float32)
    K[1] = 15.0                                  # m_c = 0, Delta_c = 1
    K[2] = np.where(q > 0, 7.5 - 2 ** -7, 7.5 + 2 ** -7).astype(np.float32)
    ub, lo, s = _check_bounds(q, K, 64)
    slack = ub[2] - s[2]
    # the excess of s over the code-estimate is ~ 0.49 sum |q_c| / sqrt(d):
    # the bound has to carry nearly all of its key-rounding slack
    assert slack < 0.1 * np.abs(q).sum() / 8.0


def test_bound_tight_for_aligned_query_residual():
    # Worst case for the query-code residual: codes 15 where the residual
    # r_c = a_c - alpha at_c is positive and 0 where it is negative.
    rng = np.random.default_rng(17)
    d = 64
    q = (rng.standard_normal(d) * np.linspace(0.2, 3, d)).astype(np.float32)
    K = np.zeros((64, d), np.float32)
    K[1] = 15.0                                   # m_c = 0, Delta_c = 1
    codes, _, mins, deltas = quantize_keys(K, 64)
    at, alpha, b_hi, b_lo = query_prep(q, mins, deltas, 7)
    qt = (q * np.float32(1 / 8.0)).astype(np.float32)
    r = qt * deltas[0] - alpha[0] * at[0].astype(np.float32)
    K[2] = np.where(r > 0, 15.0, 0.0).astype(np.float32)
    K[3] = np.where(r < 0, 15.0, 0.0).astype(np.float32)
    ub, lo, s = _check_bounds(q, K, 64, QM=7)
    # codes are exact here (no key rounding): the bound's excess over s is
    # its key-rounding slack (sum |qt_c| Delta_c / 2) plus the float32
    # margin (2^-14 of a magnitude ~ 18 sum |qt_c|) only
    tol = 0.5 * np.abs(qt).sum() * (1 + 3e-3)
    assert ub[2] - s[2] <= tol
    assert s[3] - lo[3] <= tol


# ----------------------------------------------------- 8-bit refinement codes

QM8 = 2047

def test_quantizer8_error_bound_and_codes():
    # the 8-bit codes of the same blocks: 0..255 and |k - m - code Delta8|
    # <= Delta8 (1/2 + 2^-16), Delta8 = (max - min) / 255
    from oracle.quantize import quantize_keys8
    rng = np.random.default_rng(3)
    n, d = 1000, 64
    K = (rng.normal(size=(n, d)) * rng.lognormal(0, 1, d)).astype(np.float32)
    codes, mins, deltas = quantize_keys8(K, n)
    assert codes.max() <= 255
    blk = np.arange(n) // 64
    err = np.abs(K.astype(np.float64) - mins[blk] - codes[:n] * deltas[blk].astype(np.float64))
    assert np.all(err <= deltas[blk] * (0.5 + 2.0 ** -16))
    nf = n // 64
    Kb = K[:nf * 64].reshape(nf, 64, d)
    span = Kb.max(axis=1) - Kb.min(axis=1)
    assert np.allclose(deltas[:nf], span / 255.0, rtol=1e-6)


@pytest.mark.parametrize("regime", ["llama", "outliers"])
def test_bounds8_hold_and_are_tighter(regime):
    # the same bound construction on 8-bit codes (15 -> 255) holds for every
    # key and is an order of magnitude narrower than the 4-bit one
    from oracle.quantize import quantize_keys8
    rng = np.random.default_rng(4)
    n, d = 1500, 128
    K = rng.normal(size=(n, d)).astype(np.float32)
    if regime == "outliers":
        K[:, :4] *= 8.0
    q = (rng.normal(size=d) * 3.0).astype(np.float32)
    s = _exact_scores(q, K)
    c4, _, m4, d4 = quantize_keys(K, n)
    at4, al4, bh4, bl4 = query_prep(q, m4, d4)
    u4, l4, _ = key_bounds(c4, at4, al4, bh4, bl4, n)
    c8, m8, d8 = quantize_keys8(K, n)
    # 12-bit query codes (QM 2047): with int8 ones the query residual term,
    # 255 x sum |r_c|, would dominate the 8-bit keys' rounding slack
    at8, al8, bh8, bl8 = query_prep(q, m8, d8, QM=QM8, levels=255)
    u8, l8, I8 = key_bounds(c8, at8, al8, bh8, bl8, n)
    assert np.abs(I8).max() < 2 ** 24          # exact in float32
    assert np.all(u8.astype(np.float64) >= s) and np.all(l8.astype(np.float64) <= s)
    # brute-force integer dot products
    blk = np.arange(n) // 64
    for i in (0, 77, n - 1):
        assert I8[i] == int(np.dot(c8[i].astype(np.int64), at8[blk[i]].astype(np.int64)))
    w4 = float(np.mean(u4 - l4))
    w8 = float(np.mean(u8 - l8))
    assert w8 < w4 / 12.0, (w4, w8)


def test_refined_bound_level_stays_below_the_exact_level():
    # refinement: the bound level from min(ubar4, ubar8) is at least the
    # 4-bit bound level and never above the exact level, so a key it drops
    # cannot enter the sample at that level; on a peaked head it drops most
    # of the keys the 4-bit bound keeps at the stop level
    from oracle.quantize import quantize_keys8
    from oracle.step import Params, bound_levels_f32, oracle_decode_group
    w = synth.workload("llama16k", B=1, n=3000, Hq=4, Hkv=1)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, 0)
    seed = int(synth.step_seeds(w, 0)[0])
    res = oracle_decode_group(q[0], K[0, 0], V[0, 0], w.n, seed, 0,
                              Params(w.eps, w.delta, w.r))
    P = w.n - 64
    c8, m8, d8 = quantize_keys8(K[0, 0, :w.n], w.n)
    kept4 = kept8 = 0
    for h in range(w.G):
        det = res.detail[h]
        at8, al8, bh8, bl8 = query_prep(q[0, h], m8, d8, QM=QM8, levels=255)
        u8, _, _ = key_bounds(c8, at8, al8, bh8, bl8, w.n)
        u = np.minimum(det["ubar"][:P], u8[:P])
        jb8 = np.minimum(bound_levels_f32(u, det["cb"], det["t"], w.r), res.J + 1)
        jl = np.minimum(det["jl"], res.J + 1)
        assert np.all(jb8 >= np.minimum(det["jbar"], res.J + 1))
        assert np.all(jb8 <= jl)
        L = min(int(res.level[h]), res.J)
        kept4 += int((det["jbar"] <= L).sum())
        kept8 += int((jb8 <= L).sum())
    assert kept8 < kept4
