"""Pins for the confidence events, the output bound beta and coverage.

picx.dev summary, "Algorithm Components" 3 (Chernoff interval on the
Poisson-binomial count, Hilbert-space Bernstein bound on the centred
numerator Z_c, beta = (zeta + ||o_hat - c|| dD) / (D_hat - dD)) and Theorem 4
(Pr[certified and error > eps] <= delta).  Probabilities are computed
exactly: Poisson-binomial laws by dynamic programming, and every event by
enumerating all 2^m samples of a small light set.
"""
import itertools
import math

import numpy as np
import pytest

import synth
from oracle.certificate import (MEASURE_CLT, MEASURE_DENOM, MEASURE_OUTPUT,
                                MEASURE_VALUE, clt_quantile,
                                certificate_levels, chernoff_interval)
from oracle.step import Params, dense_attention, oracle_decode_group


def _poisson_binomial_pmf(p):
    pmf = np.zeros(len(p) + 1)
    pmf[0] = 1.0
    for pi in p:
        pmf[1:] = pmf[1:] * (1 - pi) + pmf[:-1] * pi
        pmf[0] *= (1 - pi)
    return pmf


@pytest.mark.parametrize("delta_e", [0.3, 0.1, 0.01])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_chernoff_interval_exact_coverage(delta_e, seed):
    rng = np.random.default_rng(seed)
    m = 30
    for scale in (0.05, 0.3, 0.9):
        p = np.clip(rng.uniform(0, 2 * scale, m), 1e-6, 1.0)
        mu = p.sum()
        pmf = _poisson_binomial_pmf(p)
        k = np.arange(m + 1, dtype=np.float64)
        lo, hi = chernoff_interval(k, math.log(2.0 / delta_e))
        cover = pmf[(lo <= mu) & (mu <= hi)].sum()
        assert cover >= 1.0 - delta_e
        # the interval always contains the observed count
        assert np.all(lo <= k) and np.all(k <= hi)


def test_chernoff_zero_count():
    lo, hi = chernoff_interval(np.array([0.0]), 5.0)
    assert lo[0] == 0.0 and hi[0] == 5.0


def _enumerate(m=12, d=3, seed=0, tau=0.5, delta_e=0.1):
    """All 2^m samples of a light set A with exact probabilities, plus the
    oracle's certificate quantities for each sample."""
    rng = np.random.default_rng(seed)
    w = rng.uniform(0.02, 0.98, m) * tau            # light: w < tau
    v = rng.normal(0, 1, (m, d)) * rng.lognormal(0, 0.5, (m, 1))
    c = rng.normal(0, 0.3, d)                      # fixed centre
    pi = w / tau
    X = np.array(list(itertools.product([0, 1], repeat=m)), dtype=np.float64)
    prob = np.prod(np.where(X > 0, pi, 1 - pi), axis=1)
    S = len(X)
    vn2 = (v * v).sum(axis=1)
    gc = ((v - c) ** 2).sum(axis=1)
    Vmax = float(np.sqrt(vn2.max())) * (1 + 1e-12)
    # window that fixes the centre: D_R = 1, N_R = c, no heavy keys
    D_R, N_R, H_R = 1.0, c.copy(), float(c @ c)
    res = certificate_levels(
        np.full(S, tau), X.sum(1), X @ v, X @ gc, X @ vn2, np.zeros(S),
        np.zeros((S, d)), np.zeros(S), D_R, N_R, H_R, Vmax, delta_e, 0.05,
        MEASURE_VALUE)
    truth = {"G_A": (w * gc).sum(), "H_A": (w * vn2).sum(),
             "D": D_R + w.sum(), "N": N_R + w @ v,
             "Z": (tau * X - w[None, :]) @ (v - c[None, :])}
    return X, prob, res, truth, w, v, c, tau


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("delta_e", [0.2, 0.05])
def test_bernstein_events_by_enumeration(seed, delta_e):
    X, prob, res, tr, w, v, c, tau = _enumerate(seed=seed, delta_e=delta_e)
    # G_hi is an upper confidence bound on G_A(c)
    assert prob[tr["G_A"] > res["G_hi"]].sum() <= delta_e
    # ||Z_c|| <= zeta fails only on the G event or the Pinelis event
    zn = np.linalg.norm(tr["Z"], axis=1)
    assert prob[zn > res["zeta"]].sum() <= 2 * delta_e
    # H_lo is a lower confidence bound on H_A
    assert prob[tr["H_A"] < res["H_lo"]].sum() <= delta_e
    # Chernoff: |D_hat - D| <= dD
    assert prob[np.abs(res["D_hat"] - tr["D"]) > res["dD"]].sum() <= delta_e
    # the output bound: ||o_hat - o|| <= beta outside the four events
    o = tr["N"] / tr["D"]
    err = np.linalg.norm(res["o_hat"] - o[None, :], axis=1)
    assert prob[err > res["beta"]].sum() <= 4 * delta_e


def test_beta_algebra_identity():
    # o - o_hat = [(o_hat - c)(D_hat - D) - Z_c] / D for every sample, with
    # Z_c = sum_A (tau X_i - w_i)(v_i - c) exactly as the pages define it
    X, prob, res, tr, w, v, c, tau = _enumerate(seed=5)
    o = tr["N"] / tr["D"]
    lhs = o[None, :] - res["o_hat"]
    rhs = ((res["o_hat"] - c[None, :]) * (res["D_hat"] - tr["D"])[:, None]
           - tr["Z"]) / tr["D"]
    assert np.allclose(lhs, rhs, rtol=0, atol=1e-12)
    # hence beta bounds the error whenever |D_hat - D| <= dD and
    # ||Z_c|| <= zeta
    ok = (np.abs(res["D_hat"] - tr["D"]) <= res["dD"]) & \
         (np.linalg.norm(tr["Z"], axis=1) <= res["zeta"])
    err = np.linalg.norm(lhs, axis=1)
    assert np.all(err[ok] <= res["beta"][ok] * (1 + 1e-12))
    # and beta dominates the derivation's intermediate bound
    # (||o_hat - c|| |D_hat - D| + ||Z_c||) / D on those samples
    inter = (np.linalg.norm(res["o_hat"] - c[None, :], axis=1)
             * np.abs(res["D_hat"] - tr["D"])
             + np.linalg.norm(tr["Z"], axis=1)) / tr["D"]
    assert np.all(inter[ok] <= res["beta"][ok] * (1 + 1e-12))


def _coverage(name, n, measure, eps, steps, delta):
    w = synth.workload(name, B=1, n=n)
    K, V, meta = synth.kv_numpy(w)
    viol = 0
    errs = []
    fell_back = 0
    for st in range(steps):
        q = synth.q_numpy(w, meta, st, K=K)
        p = Params(eps, delta, 2, measure=measure)
        res = oracle_decode_group(q[0, :1], K[0, 0], V[0, 0], n, 1000 + st, 0, p,
                                  keep_detail=False)
        o, s = dense_attention(q[0, 0], K[0, 0, :n], V[0, 0, :n])
        a = np.exp(s - s.max())
        a /= a.sum()
        Vd = V[0, 0, :n].astype(np.float64)
        if measure == MEASURE_VALUE:
            scale = math.sqrt(a @ (Vd * Vd).sum(axis=1))
        else:
            scale = np.linalg.norm(o)
        e = np.linalg.norm(res.o[0] - o) / scale
        if res.level[0] <= res.J:
            errs.append(e)
            if measure != MEASURE_DENOM and e > eps:
                viol += 1
        else:
            fell_back += 1
    return viol, np.array(errs), fell_back


@pytest.mark.parametrize("measure", [MEASURE_VALUE, MEASURE_OUTPUT])
def test_certificate_coverage(measure):
    # Theorem 4: Pr[certified and error > eps] <= delta.  Over 150 fresh
    # queries and perturbations the violation count must stay under the
    # 99.9% binomial quantile for rate delta (the pages observed none).
    delta, steps = 0.05, 150
    viol, errs, fb = _coverage("tiny", 1024, measure, 0.05, steps, delta)
    assert viol <= delta * steps + 3.1 * math.sqrt(delta * steps)
    assert len(errs) > 0 and errs.max() <= 1.0


def _light_set_mc(m, d, seed, tau, n_mc, c_shift=0.0):
    rng = np.random.default_rng(seed)
    w = rng.uniform(0.05, 0.95, m) * tau
    v = rng.normal(0, 1, (m, d)) + c_shift
    c = np.zeros(d)
    return w, v, c


@pytest.mark.parametrize("delta_e", [0.05, 0.01])
def test_chernoff_dD_large_count(delta_e):
    # Gaussian regime (mu ~ 300): the relative-entropy interval is nearly
    # tight, so a narrower interval (smaller log term) would miss too often.
    rng = np.random.default_rng(9)
    m, tau = 1200, 0.5
    w = rng.uniform(0.05, 0.45, m) * tau
    p = w / tau
    pmf = _poisson_binomial_pmf(p)
    k = np.arange(m + 1, dtype=np.float64)
    S = m + 1
    d = 1
    res = certificate_levels(
        np.full(S, tau), k, np.zeros((S, d)), np.zeros(S), np.zeros(S),
        np.zeros(S), np.zeros((S, d)), np.zeros(S), 1.0, np.zeros(d), 0.0,
        1.0, delta_e, 0.05, MEASURE_VALUE)
    D = 1.0 + w.sum()
    miss = pmf[np.abs(res["D_hat"] - D) > res["dD"]].sum()
    assert miss <= delta_e
    assert miss >= delta_e / 200          # not grossly over-wide either


@pytest.mark.parametrize("d,c_shift", [(1, 0.0), (8, 0.0), (1, 3.0)])
def test_numerator_bound_monte_carlo(d, c_shift):
    # Many light keys (m = 400): Bernstein/Pinelis and the beta bound are
    # close to tight; a halved zeta or a dropped ||o_hat - c|| dD term fails.
    m, tau, n_mc, delta_e = 400, 0.25, 40000, 0.05
    w, v, c = _light_set_mc(m, d, 21 + d, tau, n_mc, c_shift)
    rng = np.random.default_rng(4)
    X = (rng.random((n_mc, m)) < (w / tau)[None, :]).astype(np.float64)
    vn2 = (v * v).sum(axis=1)
    gc = ((v - c) ** 2).sum(axis=1)
    Vmax = float(np.sqrt(vn2.max())) * (1 + 1e-12)
    D_R = 0.5
    N_R = c * D_R
    res = certificate_levels(
        np.full(n_mc, tau), X.sum(1), X @ v, X @ gc, X @ vn2,
        np.zeros(n_mc), np.zeros((n_mc, d)), np.zeros(n_mc), D_R, N_R,
        D_R * float(c @ c), Vmax, delta_e, 0.05, MEASURE_VALUE)
    Z = (tau * X - w[None, :]) @ (v - c[None, :])
    zn = np.linalg.norm(Z, axis=1)
    G_A = (w * gc).sum()
    H_A = (w * vn2).sum()
    se = 4 * math.sqrt(delta_e / n_mc)
    assert (zn > res["zeta"]).mean() <= 2 * delta_e + se
    assert (G_A > res["G_hi"]).mean() <= delta_e + se
    assert (H_A < res["H_lo"]).mean() <= delta_e + se
    D = D_R + w.sum()
    o = (N_R + w @ v) / D
    err = np.linalg.norm(res["o_hat"] - o[None, :], axis=1)
    assert (err > res["beta"]).mean() <= 4 * delta_e + se
    if c_shift == 0.0:
        # centred on the mean: the bound is informative, not vacuous
        assert np.median(res["beta"]) < 20 * np.median(err)


@pytest.mark.parametrize("delta_e", [0.02, 0.01])
def test_bernstein_near_tight_regime(delta_e):
    # One-dimensional values v = +-1 (70 % +1) around c = 0 and small
    # inclusion probabilities: Var Z_c ~ tau G_A and the G_hat terms sit at
    # their range bound, so the Bernstein / Pinelis constants are nearly
    # attained (a zeta or G_hi too small by a factor 2 fails), and Z_c and
    # D_hat - D move together, so beta must carry its ||o_hat - c|| dD term.
    rng = np.random.default_rng(31)
    m, d, tau, n_mc = 3000, 1, 0.5, 20000
    w = rng.uniform(0.01, 0.1, m) * tau
    v = np.where(rng.random(m) < 0.7, 1.0, -1.0)[:, None]
    c = np.zeros(d)
    D_R = 1e-3
    miss_z = miss_g = miss_b = bad_inter = 0
    G_A = w.sum()
    D = D_R + w.sum()
    o = (w @ v) / D
    for chunk in range(n_mc // 2000):
        X = (rng.random((2000, m)) < (w / tau)[None, :]).astype(np.float64)
        k = X.sum(1)
        res = certificate_levels(
            np.full(2000, tau), k, X @ v, k.copy(), k.copy(), np.zeros(2000),
            np.zeros((2000, d)), np.zeros(2000), D_R, c * D_R, 0.0,
            1.0 + 1e-12, delta_e, 0.05, MEASURE_VALUE)
        Z = (tau * X - w[None, :]) @ v
        zn = np.linalg.norm(Z, axis=1)
        miss_z += (zn > res["zeta"]).sum()
        miss_g += (G_A > res["G_hi"]).sum()
        err = np.linalg.norm(res["o_hat"] - o[None, :], axis=1)
        miss_b += (err > res["beta"]).sum()
        dev = np.abs(res["D_hat"] - D)
        ok = (dev <= res["dD"]) & (zn <= res["zeta"])
        inter = (np.linalg.norm(res["o_hat"] - c[None, :], axis=1) * dev
                 + zn) / D
        bad_inter += (inter[ok] > res["beta"][ok] * (1 + 1e-12)).sum()
    se = 4 * math.sqrt(delta_e / n_mc)
    assert miss_z / n_mc <= 2 * delta_e + se
    assert miss_g / n_mc <= delta_e + se
    assert miss_b / n_mc <= 4 * delta_e + se
    assert bad_inter == 0


@pytest.mark.parametrize("delta", [0.05, 0.2])
def test_clt_estimate_coverage_monte_carlo(delta):
    # The uncertified comparison rule: beta_clt = z sqrt(tau G_hat) / D_hat
    # with z the two-sided normal quantile.  With small inclusion
    # probabilities Var Z_c = tau G_A and, for scalar values centred on c,
    # o_hat - o ~ -Z_c / D, so P(|o_hat - o| <= beta_clt) ~ 1 - delta.  A
    # dropped square root, tau or quantile moves the coverage far off.
    m, tau, n_mc, d = 2000, 0.25, 40000, 1
    rng = np.random.default_rng(31)
    w = rng.uniform(0.005, 0.03, m) * tau
    v = rng.normal(0, 1, (m, d))
    c = np.zeros(d)
    X = (rng.random((n_mc, m)) < (w / tau)[None, :]).astype(np.float64)
    vn2 = (v * v).sum(axis=1)
    gc = ((v - c) ** 2).sum(axis=1)
    D_R = 5.0
    N_R = c * D_R
    J1 = 7                                # levels of the certified rule
    res = certificate_levels(
        np.full(n_mc, tau), X.sum(1), X @ v, X @ gc, X @ vn2,
        np.zeros(n_mc), np.zeros((n_mc, d)), np.zeros(n_mc), D_R, N_R,
        0.0, float(np.sqrt(vn2.max())), delta / (4.0 * J1), 0.05,
        MEASURE_CLT, delta=delta)
    D = D_R + w.sum()
    o = (N_R + w @ v) / D
    err = np.linalg.norm(res["o_hat"] - o[None, :], axis=1)
    cover = (err <= res["beta"]).mean()
    assert abs(cover - (1.0 - delta)) <= 0.02, cover
    assert abs(clt_quantile(0.05) - 1.959964) < 1e-5
    # the certified bound at the same level is wider
    cert = certificate_levels(
        np.full(n_mc, tau), X.sum(1), X @ v, X @ gc, X @ vn2,
        np.zeros(n_mc), np.zeros((n_mc, d)), np.zeros(n_mc), D_R, N_R,
        0.0, float(np.sqrt(vn2.max())), delta / (4.0 * J1), 0.05,
        MEASURE_VALUE)
    assert np.median(res["beta"]) < np.median(cert["beta"])


def test_clt_rule_stops_no_later_than_certificate():
    # on the same draws the uncertified rule stops at or before the
    # certified stop level (its bound is narrower at every level)
    w = synth.workload("llama16k", n=3000, Hq=8, Hkv=2)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, 0)
    seed = int(synth.step_seeds(w, 0)[0])
    for g in range(w.Hkv):
        qs = q[0, g * w.G:(g + 1) * w.G]
        a = oracle_decode_group(qs, K[0, g], V[0, g], w.n, seed, g,
                                Params(w.eps, w.delta, w.r), keep_detail=False)
        b = oracle_decode_group(qs, K[0, g], V[0, g], w.n, seed, g,
                                Params(w.eps, w.delta, w.r, measure=MEASURE_CLT),
                                keep_detail=False)
        assert np.all(b.level <= a.level)
        assert np.all(b.values_read <= a.values_read)


def test_certificate_coverage_per_head_draws():
    # one perturbation draw per query head (instead of one per KV group):
    # each head's certificate is the same construction on its own sample,
    # so Theorem 4 holds per head; 4 heads x 60 fresh steps at 1024 tokens
    w = synth.workload("llama16k", B=1, n=1024, Hq=4, Hkv=1)
    K, V, meta = synth.kv_numpy(w)
    Vd = V[0, 0].astype(np.float64)
    viol, heads, differ = 0, 0, 0
    for st in range(60):
        q = synth.q_numpy(w, meta, st, K=K)
        p = Params(w.eps, w.delta, w.r, per_head=True)
        res = oracle_decode_group(q[0], K[0, 0], V[0, 0], w.n, 500 + st, 0, p)
        ts = [d["t"] for d in res.detail]
        differ += int(not np.array_equal(ts[0], ts[1]))
        for h in range(w.G):
            o, s_ = dense_attention(q[0, h], K[0, 0], V[0, 0])
            a = np.exp(s_ - s_.max())
            a /= a.sum()
            M = math.sqrt(a @ (Vd * Vd).sum(axis=1))
            heads += 1
            if res.level[h] <= res.J and np.linalg.norm(res.o[h] - o) > w.eps * M:
                viol += 1
    assert differ == 60
    assert viol <= w.delta * heads + 3.1 * math.sqrt(w.delta * heads)
