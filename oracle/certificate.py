"""Per-level confidence events and the output-error certificate (float64).

picx.dev summary, "Algorithm Components" 3 (anytime-valid certificates) and
"Theoretical Contributions" (Theorems 1, 2, 4).  On the grid
tau_j = 2^(-j/r) each level gets failure budget delta_e per event; the pages
print the divisor garbled ("delta/((J+1) e-dot)"), read here as the number of
confidence events per level, 4:  delta_e = delta / (4 (J + 1)).  The events:

 1. Chernoff interval for the Poisson-binomial sample count k (two-sided,
    delta_e/2 per side): mu_lo <= mu <= mu_hi solve
    mu - k + k ln(k/mu) = ln(2/delta_e)  (relative-entropy form; k = 0 gives
    mu_lo = 0, mu_hi = ln(2/delta_e)).  Then |D_hat - D| <= dD with
    dD = tau * max(k - mu_lo, mu_hi - k).
 2. Upper bound G_hi on G_A(c) = sum_A w_i ||v_i - c||^2 from a one-sided
    Bernstein bound on G_hat = tau sum_{S cap A} ||v_i - c||^2 (terms in
    [0, tau R_c^2], variance <= tau R_c^2 G_A), L = ln(1/delta_e):
    G_hi = ((a + sqrt(a^2 + 4 (G_hat + (2/3) tau R_c^2 L))) / 2)^2,
    a = sqrt(2 tau R_c^2 L).
 3. Hilbert-space Bernstein (Pinelis form) on the centred numerator
    Z_c = sum_A (tau X_i - w_i)(v_i - c): ||Z_c|| <= zeta with
    zeta = sqrt(2 tau G_hi L_z) + (2/3) tau R_c L_z,  L_z = ln(2/delta_e),
    summand norm <= b = tau R_c, variance <= tau G_A (Theorem 1).
 4. (value scale only) lower bound on H_A = sum_A w_i ||v_i||^2 from
    H_hat = tau S2:  H_lo = ((-a' + sqrt(a'^2 + 4 (H_hat - (2/3) tau V^2 L)))
    / 2)^2 when the bracket is positive, else 0; a' = sqrt(2 tau V^2 L).

Centre c = (N_R + N_B) / (D_R + D_B): the deterministic part of the estimate
(window and heavy keys), independent of the perturbations.  R_c = V + ||c||
with V = largest per-block value norm bound over the pool.

Output bound (picx.dev, "Algorithm Components" 3):
    beta = (zeta + ||o_hat - c|| dD) / (D_hat - dD),  +inf if D_hat <= dD.
It follows from o - o_hat = [(o_hat - c)(D_hat - D) - Z_c] / D.

Certified (the stopping rule: a head ends at its lowest certified level), with the scale
replaced by a lower confidence bound so the claim is relative to the truth:
    value  (||o_hat - o|| <= eps M):   beta <= eps * M_lo,
           M_lo = sqrt((H_R + H_B + H_lo) / D_hi), D_hi = D_RB + tau mu_hi;
    output (||o_hat - o|| <= eps ||o||): beta (1 + eps) <= eps ||o_hat||;
    denom  (|D_hat - D| <= eps D):       dD <= eps (D_hat - dD);
and always D_hat > dD.

Uncertified comparison mode (picx.dev "Theoretical Contributions": certified
runs read 1.8-3.5x more keys than uncertified CLT rules): MEASURE_CLT stops
at the first level where a normal-approximation error estimate meets the
target,
    beta_clt = z sqrt(tau G_hat) / D_hat,   z = Phi^-1(1 - delta/2),
    (tau G_hat estimates Var Z_c = sum_A tau w_i (1 - w_i/tau) ||v_i - c||^2)
    stop iff D_hat > 0 and beta_clt <= eps M_hat,
    M_hat = sqrt((H_R + H_B + tau S2) / D_hat)  (plug-in value scale).
It carries no guarantee; it is the baseline the certificate is compared with.
Test infrastructure only.
"""
from __future__ import annotations

import math
from statistics import NormalDist

import numpy as np

MEASURE_VALUE, MEASURE_OUTPUT, MEASURE_DENOM, MEASURE_CLT = 0, 1, 2, 3


def clt_quantile(delta: float) -> float:
    """z = Phi^-1(1 - delta/2), the two-sided normal quantile."""
    return NormalDist().inv_cdf(1.0 - delta / 2.0)


def chernoff_interval(k: np.ndarray, Lz: float, iters: int = 200):
    """[mu_lo, mu_hi] for observed counts k (float64 arrays), by bisection."""
    k = np.asarray(k, dtype=np.float64)
    lo_out = np.zeros_like(k)
    hi_out = np.full_like(k, Lz)
    pos = k > 0
    if np.any(pos):
        kk = k[pos]

        def f(mu):
            return mu - kk + kk * np.log(kk / mu)

        # lower root in (0, k]: f decreases from +inf to 0
        a = np.zeros_like(kk)
        b = kk.copy()
        for _ in range(iters):
            mid = 0.5 * (a + b)
            big = f(np.maximum(mid, 1e-300)) > Lz
            a = np.where(big, mid, a)
            b = np.where(big, b, mid)
        lo_out[pos] = a                      # outer end of the bracket
        # upper root in [k, inf): f increases from 0
        a = kk.copy()
        b = kk + Lz + np.sqrt(2.0 * kk * Lz) + 2.0 * Lz + 1.0
        while np.any(f(b) <= Lz):
            b = np.where(f(b) <= Lz, 2.0 * b, b)
        for _ in range(iters):
            mid = 0.5 * (a + b)
            small = f(mid) <= Lz
            a = np.where(small, mid, a)
            b = np.where(small, b, mid)
        hi_out[pos] = b                      # outer end of the bracket
    return lo_out, hi_out


def certificate_levels(tau, k, S1, Gsum, S2, D_B, N_B, H_B, D_R, N_R, H_R,
                       Vmax, delta_e, eps, measure=MEASURE_VALUE, delta=None):
    """Certificate quantities at every level (all float64).

    Per-level inputs (leading axis = level): tau, k (light sampled count),
    S1 [.., d] (sum of v over light sampled), Gsum (sum of ||v - c_j||^2 over
    light sampled, with c_j the level's centre), S2 (sum of ||v||^2 over light
    sampled), D_B, N_B [.., d], H_B (heavy sums).  Window sums D_R, N_R [d],
    H_R.  Returns a dict of per-level arrays: D_hat, o_hat, dD, c, beta,
    scale_lo, certified.  delta (the per-step failure probability) is used
    only by MEASURE_CLT, whose quantile takes no union bound over levels.
    """
    L = math.log(1.0 / delta_e)
    Lz = math.log(2.0 / delta_e)
    tau = np.asarray(tau, np.float64)
    k = np.asarray(k, np.float64)
    D_RB = D_R + D_B
    D_hat = D_RB + tau * k
    N_hat = N_R[None, :] + N_B + tau[:, None] * S1
    o_hat = N_hat / D_hat[:, None]
    mu_lo, mu_hi = chernoff_interval(k, Lz)
    dD = tau * np.maximum(k - mu_lo, mu_hi - k)
    D_hi = D_RB + tau * mu_hi
    c = (N_R[None, :] + N_B) / D_RB[:, None]
    cn = np.linalg.norm(c, axis=1)
    Rc = Vmax + cn
    G_hat = tau * Gsum
    a = np.sqrt(2.0 * tau * Rc * Rc * L)
    G_hi = ((a + np.sqrt(a * a + 4.0 * (G_hat + (2.0 / 3.0) * tau * Rc * Rc
                                        * L))) / 2.0) ** 2
    zeta = np.sqrt(2.0 * tau * G_hi * Lz) + (2.0 / 3.0) * tau * Rc * Lz
    pos = D_hat > dD
    ocn = np.linalg.norm(o_hat - c, axis=1)
    beta = np.where(pos, (zeta + ocn * dD) / np.where(pos, D_hat - dD, 1.0),
                    np.inf)
    if measure == MEASURE_VALUE:
        H_hat = tau * S2
        ap = np.sqrt(2.0 * tau * Vmax * Vmax * L)
        br = H_hat - (2.0 / 3.0) * tau * Vmax * Vmax * L
        H_lo = np.where(br > 0, ((-ap + np.sqrt(ap * ap + 4.0 *
                                                np.maximum(br, 0.0))) / 2.0) ** 2,
                        0.0)
        M_lo = np.sqrt((H_R + H_B + H_lo) / D_hi)
        extra = {"H_lo": H_lo}
        scale = M_lo
        cert = pos & (beta <= eps * M_lo)
    elif measure == MEASURE_OUTPUT:
        onorm = np.linalg.norm(o_hat, axis=1)
        extra = {}
        scale = onorm
        cert = pos & (beta * (1.0 + eps) <= eps * onorm)
    elif measure == MEASURE_DENOM:
        extra = {}
        scale = D_hat - dD
        cert = pos & (dD <= eps * (D_hat - dD))
    elif measure == MEASURE_CLT:
        z = clt_quantile(delta)
        beta = z * np.sqrt(tau * np.maximum(G_hat, 0.0)) / D_hat
        M_hat = np.sqrt((H_R + H_B + tau * S2) / D_hat)
        extra = {"M_hat": M_hat}
        scale = M_hat
        cert = (D_hat > 0) & (beta <= eps * M_hat)
    else:
        raise ValueError("unknown measure")
    return {"D_hat": D_hat, "o_hat": o_hat, "dD": dD, "c": c, "beta": beta,
            "scale_lo": scale, "certified": cert, "mu_lo": mu_lo,
            "mu_hi": mu_hi, "G_hi": G_hi, "zeta": zeta, "D_hi": D_hi,
            **extra}
