"""Pins for perturbed threshold sampling and the Horvitz-Thompson estimates.

picx.dev summary, "Theoretical Foundation": key i passes the perturbed
threshold s_i - c* + E_i >= log tau with probability min(1, w_i / tau)
(threshold PPS sampling), a lower tau only adds keys (the samples nest),
and the Horvitz-Thompson estimates are unbiased
(Theorem 1: E D_hat = D, E N_hat = N, Var D_hat <= tau D_A).  These tests run
the oracle's own level and sum routines over many step seeds.
"""
import math

import numpy as np
import pytest

import synth
from oracle.hashing import perturb_t
from oracle.step import (Params, exact_levels, level_sums,
                         oracle_decode_group, dense_attention)


def _seeds_t(n_seeds, pool, g=0, base=1000):
    return np.stack([perturb_t(base + s, g, np.arange(pool))
                     for s in range(n_seeds)])


def test_inclusion_law_monte_carlo():
    rng = np.random.default_rng(0)
    pool, r, N = 16, 2, 40000
    sp = rng.normal(0.0, 1.5, pool)
    c_star = sp.max() + 0.3            # the maximum sits in the window
    t = _seeds_t(N, pool)
    jl, hl = exact_levels(sp, c_star, t, r)
    w = np.exp(sp - c_star)
    for j in range(0, 12):
        tau = 2.0 ** (-j / r)
        p = np.minimum(1.0, w / tau)
        freq = (jl <= j).mean(axis=0)
        sd = np.sqrt(np.maximum(p * (1 - p), 1e-12) / N)
        assert np.all(np.abs(freq - p) <= 4.5 * sd + 1.0 / N), (j, freq, p)
        # heavy keys (w >= tau) are always sampled
        assert np.all((jl <= j)[:, w >= tau])


def test_samples_are_nested():
    rng = np.random.default_rng(1)
    pool, r = 200, 3
    sp = rng.normal(0.0, 2.0, pool)
    t = _seeds_t(50, pool)
    jl, hl = exact_levels(sp, sp.max(), t, r)
    for j in range(20):
        assert np.all((jl <= j) <= (jl <= j + 1))
        assert np.all((hl <= j) <= (hl <= j + 1))
        # heavy implies sampled
        assert np.all((hl <= j) <= (jl <= j))


def test_unbiased_estimates_and_variance_bound():
    rng = np.random.default_rng(2)
    pool, d, r, N = 40, 4, 2, 20000
    sp = rng.normal(0.0, 1.0, pool)
    win_s = rng.normal(0.0, 1.0, 8)
    c_star = max(sp.max(), win_s.max())
    Vp = rng.normal(0.0, 1.0, (pool, d))
    Vw = rng.normal(0.0, 1.0, (8, d))
    w = np.exp(sp - c_star)
    ww = np.exp(win_s - c_star)
    D_R, N_R = ww.sum(), ww @ Vw
    D = D_R + w.sum()
    Nv = N_R + w @ Vp
    t = _seeds_t(N, pool, base=77)
    jl, hl = exact_levels(sp, c_star, t, r)
    levels = [0, 2, 5, 9]
    Dh = np.zeros((N, len(levels)))
    Nh = np.zeros((N, len(levels), d))
    for s in range(N):
        sums = level_sums(jl[s], hl[s], w, Vp, D_R, N_R, 10)
        for a, j in enumerate(levels):
            tau = 2.0 ** (-j / r)
            Dh[s, a] = D_R + sums["D_B"][j] + tau * sums["k"][j]
            Nh[s, a] = N_R + sums["N_B"][j] + tau * sums["S1"][j]
    for a, j in enumerate(levels):
        tau = 2.0 ** (-j / r)
        sd = Dh[:, a].std() / math.sqrt(N)
        assert abs(Dh[:, a].mean() - D) <= 5 * sd + 1e-12
        sdn = Nh[:, a].std(axis=0) / math.sqrt(N)
        assert np.all(np.abs(Nh[:, a].mean(axis=0) - Nv) <= 5 * sdn + 1e-12)
        D_A = w[w < tau].sum()
        # Theorem 1: Var D_hat <= tau D_A (sampling error of a variance
        # estimate: 5 * sqrt(2/N) relative)
        assert Dh[:, a].var() <= tau * D_A * (1 + 5 * math.sqrt(2.0 / N)) \
            + 1e-15


def _group(name="tiny", n=700, seed_step=0, **over):
    w = synth.workload(name, B=1, n=n, **over)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, seed_step, K=K)
    return w, K, V, q


@pytest.mark.parametrize("name,n", [("tiny", 700), ("llama16k", 1500)])
def test_candidate_invariants(name, n):
    over = {} if name == "tiny" else {"Hq": 8, "Hkv": 2}
    w, K, V, q = _group(name, n, **over)
    p = Params(w.eps, w.delta, w.r)
    for g in range(w.Hkv):
        for seed in (3, 4, 5):
            res = oracle_decode_group(q[0, g * w.G:(g + 1) * w.G], K[0, g],
                                      V[0, g], n, seed, g, p)
            J = res.J
            for det in res.detail:
                jbar, jl, hl = det["jbar"], det["jl"], det["hl"]
                # the bound level never exceeds the exact level ...
                assert np.all(jbar <= jl)
                # ... so every key sampled up to J is a candidate
                assert np.all(det["cand"][jl <= J])
                # exact maximum over the small set is the global maximum
                assert det["c_star"] == det["s"].max()
                assert det["cb"] <= det["c_star"]
                assert det["c_lo"] <= det["c_star"] <= det["c_hi"]


def test_dense_when_pool_empty():
    w, K, V, q = _group("tiny", 64)
    res = oracle_decode_group(q[0], K[0, 0], V[0, 0], 64, 9, 0,
                              Params(0.05, 0.01, 2))
    o, _ = dense_attention(q[0, 0], K[0, 0, :64], V[0, 0, :64])
    assert np.allclose(res.o[0], o, rtol=0, atol=1e-12)
    assert res.beta[0] == 0 and res.level[0] == 0
    assert res.keys_read[0] == 64 and res.values_read[0] == 64


def test_exact_when_grid_passes_every_weight():
    # extend the grid until tau_J is below every weight: the sample is the
    # whole pool, all keys heavy, and o_hat at level J is dense attention
    w, K, V, q = _group("tiny", 400)
    n = 400
    s = K[0, 0, :n].astype(np.float64) @ q[0, 0].astype(np.float64) / 8.0
    wmin = np.exp(s - s.max()).min()
    J = int(math.ceil(-2 * math.log2(wmin))) + 1
    res = oracle_decode_group(q[0], K[0, 0], V[0, 0], n, 11, 0,
                              Params(0.05, 0.01, 2, J_override=J))
    det = res.detail[0]
    o, _ = dense_attention(q[0, 0], K[0, 0, :n], V[0, 0, :n])
    oJ = det["cert"]["o_hat"][J]
    assert np.allclose(oJ, o, rtol=1e-12, atol=1e-12)
    assert det["k"][J] == 0 and np.all(det["hl"] <= J)
