"""Pins for the per-level sums of the estimate and for the constant of the
Hilbert-space Bernstein (Pinelis) bound.

picx.dev summary, "Algorithm Components" 2 (Horvitz-Thompson estimate:
window keys exact, heavy keys w_i >= tau exact, light keys sampled with
probability w_i / tau and weighted by tau) and 3 (the centred numerator Z_c,
its Hilbert-space Bernstein bound zeta, the variance proxy G).

``level_sums`` feeds every certificate quantity: D_B, N_B, H_B over heavy
keys, and k, S1, S2, Gs over light sampled keys with Gs centred on the
level's deterministic centre c_j = (N_R + N_B) / (D_R + D_B).  It is pinned
here by a pool small enough to sum by hand (the expected values are written
out as numbers), and by a per-key event formulation on random pools: each
key enters the light sums at its inclusion level and leaves them at its
heavy level, where it enters the heavy sums.
"""
import math

import numpy as np
import pytest

from oracle.certificate import MEASURE_VALUE, certificate_levels
from oracle.step import level_sums

# ---------------------------------------------------------------- by hand
#
# Four pool keys, d = 2, levels 0..2.
#   key  w     v         jl  hl
#   0    0.9   ( 1, 0)   0   1
#   1    0.3   ( 0, 2)   1   3
#   2    0.05  ( 1, 1)   2   4
#   3    0.6   (-1, 1)   0   2
# Window: D_R = 1, N_R = (0.5, 0.5).
# Level 0: heavy {} ; light sampled {0, 3}; c_0 = (0.5, 0.5)
#   k = 2, S1 = (0, 1), S2 = 1 + 2 = 3,
#   Gs = |(0.5,-0.5)|^2 + |(-1.5,0.5)|^2 = 0.5 + 2.5 = 3
# Level 1: heavy {0}: D_B = 0.9, N_B = (0.9, 0), H_B = 0.9 * 1 = 0.9
#   light sampled {1, 3}: k = 2, S1 = (-1, 3), S2 = 4 + 2 = 6
#   c_1 = (1.4, 0.5) / 1.9 = (14/19, 5/19)
#   Gs = |(-14/19, 33/19)|^2 + |(-33/19, 14/19)|^2 = 2 * 1285/361 = 2570/361
# Level 2: heavy {0, 3}: D_B = 1.5, N_B = (0.3, 0.6), H_B = 0.9 + 0.6*2 = 2.1
#   light sampled {1, 2}: k = 2, S1 = (1, 3), S2 = 4 + 2 = 6
#   c_2 = (0.8, 1.1) / 2.5 = (0.32, 0.44)
#   Gs = |(-0.32, 1.56)|^2 + |(0.68, 0.56)|^2 = 2.536 + 0.776 = 3.312
# Sampled keys (jl <= j): 2, 3, 4.

_W = np.array([0.9, 0.3, 0.05, 0.6])
_V = np.array([[1.0, 0.0], [0.0, 2.0], [1.0, 1.0], [-1.0, 1.0]])
_JL = np.array([0, 1, 2, 0])
_HL = np.array([1, 3, 4, 2])
_DR, _NR = 1.0, np.array([0.5, 0.5])

_HAND = {
    "k": [2.0, 2.0, 2.0],
    "S1": [[0.0, 1.0], [-1.0, 3.0], [1.0, 3.0]],
    "S2": [3.0, 6.0, 6.0],
    "Gs": [3.0, 2570.0 / 361.0, 3.312],
    "D_B": [0.0, 0.9, 1.5],
    "N_B": [[0.0, 0.0], [0.9, 0.0], [0.3, 0.6]],
    "H_B": [0.0, 0.9, 2.1],
    "n_sampled": [2.0, 3.0, 4.0],
}


def test_level_sums_hand_example():
    got = level_sums(_JL, _HL, _W, _V, _DR, _NR, 3)
    for key, want in _HAND.items():
        np.testing.assert_allclose(got[key], np.array(want), rtol=0,
                                   atol=1e-12, err_msg=key)


def test_hand_example_separates_plausible_mistakes():
    # The hand values differ from what a plausible mistake would give, by
    # far more than the 1e-12 of the pin above: Gs centred on 0 (= S2), Gs
    # centred on the estimate o_hat instead of c_j, H_B without ||v||^2
    # (= D_B), S2 summed over heavy keys too, a heavy set that counts a key
    # already at level hl - 1.
    tau = np.array([1.0, 2 ** -0.5, 0.5])          # r = 2
    k = np.array(_HAND["k"])
    S1 = np.array(_HAND["S1"])
    DB = np.array(_HAND["D_B"])
    NB = np.array(_HAND["N_B"])
    Dh = _DR + DB + tau * k
    oh = (_NR[None, :] + NB + tau[:, None] * S1) / Dh[:, None]
    wrong_gs_ohat = []
    for j in range(3):
        light = (_JL <= j) & (_HL > j)
        wrong_gs_ohat.append(((_V[light] - oh[j]) ** 2).sum())
    vn2 = (_V * _V).sum(1)
    wrong = {
        "Gs": [np.array(_HAND["S2"]), np.array(wrong_gs_ohat)],
        "H_B": [np.array(_HAND["D_B"])],
        "S2": [np.array([(vn2 * (_JL <= j)).sum() for j in range(3)])],
        "D_B": [np.array([_W[_HL <= j + 1].sum() for j in range(3)])],
    }
    for key, variants in wrong.items():
        for v in variants:
            assert np.max(np.abs(v - np.array(_HAND[key]))) > 0.05, key


# -------------------------------------------------- event formulation

def _sums_by_events(jl, hl, w, V, D_R, N_R, nL):
    """The same sums built key by key: a light key adds (1, v, ||v||^2) from
    its inclusion level until its heavy level; from the heavy level on it
    adds (w, w v, w ||v||^2) to the heavy sums.  Per-level increments, then
    a running total over the levels; Gs expanded about the level's centre
    as sum ||v||^2 - 2 c.sum v + k ||c||^2 from the light running totals."""
    d = V.shape[1]
    dk = np.zeros(nL)
    dS1 = np.zeros((nL, d))
    dS2 = np.zeros(nL)
    dDB = np.zeros(nL)
    dNB = np.zeros((nL, d))
    dHB = np.zeros(nL)
    dns = np.zeros(nL)
    for i in range(len(w)):
        v = V[i]
        q = float(v @ v)
        a, h = int(jl[i]), int(hl[i])
        if a < nL:
            dns[a] += 1
        if a < h and a < nL:
            dk[a] += 1
            dS1[a] += v
            dS2[a] += q
        if a < h and h < nL:
            dk[h] -= 1
            dS1[h] -= v
            dS2[h] -= q
        if h < nL:
            dDB[h] += w[i]
            dNB[h] += w[i] * v
            dHB[h] += w[i] * q
    out = {"k": np.cumsum(dk), "S1": np.cumsum(dS1, axis=0),
           "S2": np.cumsum(dS2), "D_B": np.cumsum(dDB),
           "N_B": np.cumsum(dNB, axis=0), "H_B": np.cumsum(dHB),
           "n_sampled": np.cumsum(dns)}
    c = (N_R[None, :] + out["N_B"]) / (D_R + out["D_B"])[:, None]
    out["Gs"] = (out["S2"] - 2.0 * (c * out["S1"]).sum(1)
                 + out["k"] * (c * c).sum(1))
    return out


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_level_sums_match_event_formulation(seed):
    rng = np.random.default_rng(seed)
    n, d, nL = 300, 8, 12
    w = rng.uniform(0.0, 1.0, n) ** 3
    V = rng.normal(0, 1, (n, d)) * rng.lognormal(0, 0.5, (n, 1))
    hl = rng.integers(0, nL + 3, n)
    jl = np.minimum(hl, rng.integers(0, nL + 3, n))     # jl <= hl
    # some keys never sampled within the grid
    jl[rng.random(n) < 0.2] = nL + 5
    hl = np.maximum(hl, jl)
    D_R = 0.7
    N_R = rng.normal(0, 1, d) * 0.5
    got = level_sums(jl, hl, w, V, D_R, N_R, nL)
    ref = _sums_by_events(jl, hl, w, V, D_R, N_R, nL)
    for key in ("k", "S1", "S2", "D_B", "N_B", "H_B", "n_sampled"):
        np.testing.assert_allclose(got[key], ref[key], rtol=0, atol=1e-10,
                                   err_msg=key)
    np.testing.assert_allclose(got["Gs"], ref["Gs"], rtol=1e-11, atol=1e-9)


# ------------------------------------------------------ Pinelis constant
#
# Z_c = sum_A (tau X_i - w_i)(v_i - c) with X_i ~ Bernoulli(w_i / tau).  In
# one dimension with every v_i - c = 1 and every w_i = p tau, Z_c =
# tau (X - m p), X ~ Binomial(m, p), whose law is known exactly.  For m p
# large the sum is nearly Gaussian and at a small budget delta_e the
# Bernstein form zeta = sqrt(2 sigma^2 L_z) + (2/3) b L_z has little slack:
# with the oracle's L_z = ln(2 / delta_e) the exact probability that
# |Z_c| > zeta is a few per cent of delta_e, while a log term 20 % smaller
# already exceeds 2 delta_e and one 35 % smaller exceeds 50 delta_e; a
# log term 50 % larger drops the probability below 1e-6 delta_e.  zeta is
# taken from the oracle's certificate, with its own G_hi from each outcome's
# observed G_hat, so the probability covers the G event as well (allowed:
# delta_e) and the Pinelis event (delta_e).

def _exact_zeta_miss(delta_e, m, p, tau=0.5, width=16.0):
    from scipy.stats import binom
    lam = m * p
    sd = math.sqrt(lam * (1.0 - p))
    k = np.arange(max(0, math.floor(lam - width * sd)),
                  math.ceil(lam + width * sd) + 1, dtype=np.float64)
    pmf = binom.pmf(k, m, p)
    S = len(k)
    # window: D_R tiny, N_R = 0, so the centre c = 0; |v| = 1 = Vmax, R_c = 1
    res = certificate_levels(
        np.full(S, tau), k, k[:, None].copy(), k.copy(), k.copy(),
        np.zeros(S), np.zeros((S, 1)), np.zeros(S), 1e-3, np.zeros(1), 0.0,
        1.0, delta_e, 0.05, MEASURE_VALUE)
    Z = np.abs(tau * (k - lam))
    return float(pmf[Z > res["zeta"]].sum()), float(1.0 - pmf.sum())


@pytest.mark.parametrize("delta_e", [1e-9, 1e-12])
def test_pinelis_constant_exact_tail(delta_e):
    pytest.importorskip("scipy")
    miss, lost = _exact_zeta_miss(delta_e, m=10 ** 8, p=0.01)
    assert lost < 1e-14                 # the window holds the whole law
    assert miss <= 2.0 * delta_e        # valid (G event + Pinelis event)
    assert miss >= 0.005 * delta_e      # and not grossly over-wide
