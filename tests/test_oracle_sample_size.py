"""Pins for Theorem 2 (the sample size it needs does not grow with n).

picx.dev summary, "Theoretical Contributions", Theorem 2: with the
threshold set to tau = D/m, the estimate is within

    (sigma_v sqrt(2L/m) + 2 R_o L/(3m)) / (1 - eta)

of the exact output with probability at least 1 - delta, where L = ln(4/delta),
eta = sqrt(2L/m) + L/(3m) and sigma_v^2 = M^2 - ||o||^2; the sample it reads
has about m values whatever the context length.  The page leaves R_o open;
these tests read it as the largest distance of a pool value from the exact
output, max_i ||v_i - o|| (the range of the centred terms the estimate sums).

The checks run the oracle's own levels, per-level sums and certificate
routine over many step seeds and compare with quantities computed from the
definitions: the exact output, the value scale M and the weights w_i.
"""
import math

import numpy as np

from oracle.certificate import certificate_levels
from oracle.hashing import perturb_t
from oracle.step import Params, exact_levels, level_sums, oracle_decode_group

DELTA = 0.1
R = 4


def _head(rng, pool, d=8, win=16):
    """Scores with a moderate spread and Gaussian values; the exact output
    o, the value scale M^2 = sum w ||v||^2 / D and the window sums."""
    sp = rng.normal(0.0, 2.0, pool)
    sw = rng.normal(0.0, 2.0, win)
    c_star = max(sp.max(), sw.max())
    Vp = rng.normal(0.3, 1.0, (pool, d))
    Vw = rng.normal(0.3, 1.0, (win, d))
    w = np.exp(sp - c_star)
    ww = np.exp(sw - c_star)
    D_R, N_R, H_R = ww.sum(), ww @ Vw, ww @ (Vw * Vw).sum(axis=1)
    D = D_R + w.sum()
    o = (N_R + w @ Vp) / D
    M2 = (H_R + w @ (Vp * Vp).sum(axis=1)) / D
    return dict(sp=sp, c_star=c_star, Vp=Vp, w=w, D_R=D_R, N_R=N_R, H_R=H_R,
                D=D, o=o, M2=M2)


def _theorem2_bound(h, m):
    L = math.log(4.0 / DELTA)
    eta = math.sqrt(2.0 * L / m) + L / (3.0 * m)
    assert eta < 1.0
    sigma_v = math.sqrt(h["M2"] - h["o"] @ h["o"])
    R_o = np.linalg.norm(h["Vp"] - h["o"][None, :], axis=1).max()
    return (sigma_v * math.sqrt(2.0 * L / m) + 2.0 * R_o * L / (3.0 * m)) \
        / (1.0 - eta)


def _estimates_at(h, j, n_seeds, base):
    """The oracle's o_hat and sample size at grid level j, one per seed."""
    pool = len(h["sp"])
    t = np.stack([perturb_t(base + s, 3, np.arange(pool))
                  for s in range(n_seeds)])
    jl, hl = exact_levels(h["sp"], h["c_star"], t, R)
    taus = 2.0 ** (-np.arange(j + 1) / R)
    err = np.zeros(n_seeds)
    size = np.zeros(n_seeds)
    for s in range(n_seeds):
        S = level_sums(jl[s], hl[s], h["w"], h["Vp"], h["D_R"], h["N_R"],
                       j + 1)
        cert = certificate_levels(taus, S["k"], S["S1"], S["Gs"], S["S2"],
                                  S["D_B"], S["N_B"], S["H_B"], h["D_R"],
                                  h["N_R"], h["H_R"], 1.0, 1e-3, 0.1)
        err[s] = np.linalg.norm(cert["o_hat"][j] - h["o"])
        size[s] = S["n_sampled"][j]
    return err, size


def test_theorem2_error_bound_and_sample_size():
    """At tau = D/m (m taken where the grid puts tau), the error exceeds the
    Theorem 2 bound in at most a delta fraction of seeds, and the sample
    holds sum_i min(1, w_i/tau) <= m keys on average, at a pool of 1000 and
    of 8000 keys alike."""
    rng = np.random.default_rng(7)
    n_seeds = 500
    for pool in (1000, 8000):
        h = _head(rng, pool)
        for m_target in (64, 256):
            j = math.ceil(R * math.log2(m_target / h["D"]))
            tau = 2.0 ** (-j / R)
            m = h["D"] / tau
            bound = _theorem2_bound(h, m)
            err, size = _estimates_at(h, j, n_seeds, base=5000 + pool)
            sd = math.sqrt(DELTA * (1 - DELTA) / n_seeds)
            assert (err > bound).mean() <= DELTA + 3 * sd, (pool, m, bound)
            # expected sample size: sum of inclusion probabilities, <= m
            p = np.minimum(1.0, h["w"] / tau)
            assert p.sum() <= m
            sd_n = math.sqrt((p * (1 - p)).sum() / n_seeds)
            assert abs(size.mean() - p.sum()) <= 4.5 * sd_n + 1e-9, \
                (pool, m, size.mean(), p.sum())


def test_theorem2_error_shrinks_with_m():
    """Quadrupling m halves the sigma_v term of the bound; the empirical
    error quantile must fall with it (by well over a third here)."""
    rng = np.random.default_rng(8)
    h = _head(rng, 4000)
    q = []
    for m_target in (64, 1024):
        j = math.ceil(R * math.log2(m_target / h["D"]))
        err, _ = _estimates_at(h, j, 300, base=9000)
        q.append(np.quantile(err, 1 - DELTA))
    assert q[1] < 0.5 * q[0], q


def test_certified_stop_reads_sublinear_values():
    """The certified stop level's sample does not grow in proportion to the
    context: four times the pool (same score and value laws) reads well
    under four times the values.  (It still grows a little: the grid's
    last level J and with it the per-event budget depend on the pool, and
    the level steps are discrete.)"""
    rng = np.random.default_rng(5)
    d = 64
    reads = {}
    for n in (4096, 16384):
        K = rng.normal(0.0, 1.0, (n, d)).astype(np.float32)
        V = (rng.normal(0.0, 1.0, (n, d)) *
             np.exp(rng.normal(0.0, 0.5, (n, 1)))).astype(np.float32)
        q = (rng.normal(0.0, 1.0, (2, d)) * 1.6).astype(np.float32)
        tot = 0
        for seed in (11, 12):
            res = oracle_decode_group(q, K, V, n, seed, 0,
                                      Params(0.1, 0.05, 2), keep_detail=False)
            assert np.all(res.level <= res.J)
            tot += int(res.values_read.sum())
        reads[n] = tot
    assert reads[16384] < 2.5 * reads[4096], reads
