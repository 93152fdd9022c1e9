"""One certified sparse decode-attention step for one (sequence, KV head).

picx.dev summary, "Methodology / Problem Setup": scores s_i = q.k_i/sqrt(d),
c* = max_i s_i, weights w_i = exp(s_i - c*), D = sum w_i, N = sum w_i v_i,
o = N / D.  "Algorithm Components" 1-4 and Theorem 4 give the steps taken
below, in this order, separately for each query head h of the group (the
4-bit codes and the perturbations are shared by the group; readsearch.ai
"Abstract"):

 1. Window R = the last 64 positions, read exactly; pool P = the rest.
    With |P| = 0 the step is dense attention (beta = 0, level 0).
 2. 4-bit bounds ubar_i >= s_i >= l_i for every key (``bounds.py``; int8
    query codes, or two-digit codes with ``Params.two_digit``: the bounds
    change, the results below do not); c*_lo = max_i l_i.
 3. Exact maximum: c* = max of s_i over R and the pool keys with
    ubar_i >= c*_lo (the exact-maximum step of "Algorithm Components" 4).
 4. Perturbations t_i = -log2 u_i (``hashing.py``).
 5. Grid tau_j = 2^(-j/r), j = 0..J with J = ceil(r log2 |P|) (tau_J <= 1/|P|),
    budget delta_e = delta / (4 (J+1)) per confidence event.
 6. Candidates, grouped by the lowest level that could include them: the bound
    level jbar_i = max(0, ceil(-r xbar_i)) with
        xbar_i = fl(fl(fl(ubar_i - cb) * log2e) + t_i)   (float32),
        jbar_i = max(0, ceil(fl(fl(-r * xbar_i) - 2^-10))),
    where cb <= c* is the float32 certified lower bound of the exact maximum
    from the float32 rescoring of step 3 (see ``cstar_lower_f32``).  Key i is
    a candidate iff jbar_i <= J.  jbar_i never exceeds the exact level j_i.
 7. Exact levels of candidates (float64): x_i = (s_i - c*) log2 e + t_i,
    j_i = max(0, ceil(-r x_i)): i in S(tau_j) iff j_i <= j, i.e.
    s_i - c* + E_i >= log tau_j (ties included).  Heavy level
    h_i = max(0, ceil(-r (s_i - c*) log2 e)): w_i >= tau_j iff h_i <= j.
 8. Per level: window, heavy (B_j = {h_i <= j}) and light sampled
    (S cap A_j = {j_i <= j < h_i}) sums; Horvitz-Thompson estimates
    D_hat = D_R + D_B + tau k, N_hat = N_R + N_B + tau sum_{S cap A} v;
    certificate (``certificate.py``).
 9. Stop at the first certified level j*; return o_hat, beta, j*.  No
    certified level up to J: exact attention, beta = 0, level J + 1.
10. keys_read = 64 + |exact-max set of the pool U {candidates with
    jbar_i <= j*}|;  values_read = 64 + |S(tau_j*)|.

Optional 8-bit refinement ("Algorithm Components" 4: an 8-bit stage before
the exact 16-bit reads; ``Params.refine8``): each candidate with
jbar_i <= j* also gets the bound ubar8_i from 8-bit codes of the same blocks
(``quantize_keys8``, query codes with QM8 levels), and the refined level
jref_i = max(0, ceil(...)) of step 6 with min(ubar_i, ubar8_i) in place of
ubar_i.  jbar_i <= jref_i <= j_i, so the sample, the estimates, the stop
level and the outputs are unchanged; only keys_read shrinks, to 64 + |exact-
max set U {candidates with jref_i <= j*}|, and the step also reads the 8-bit
rows of the candidates with jbar_i <= j* outside the exact-max set
(``rows8``).

Test infrastructure only.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

from .bounds import (QM_DEFAULT, QM_TWO_DIGIT, key_bounds, query_prep,
                     inv_sqrt_d_f32)
from .certificate import MEASURE_VALUE, certificate_levels
from .fp32 import tree_sum_f32
from .hashing import head_stream, perturb_t
from .quantize import T_BLOCK, quantize_keys, quantize_keys8, vmax_blocks

F = np.float32
WINDOW = 64
LOG2E_F32 = F(1.0 / math.log(2.0))
_CB_MARG = F(2.0 ** -13)
_LVL_SHIFT = F(2.0 ** -10)
NEAR_BAND = 1e-5            # nats, in perturbed log-score


@dataclasses.dataclass
class Params:
    eps: float = 0.05
    delta: float = 0.05
    r: int = 2
    measure: int = MEASURE_VALUE
    J_override: int = -1
    QM: int = QM_DEFAULT
    per_head: bool = False      # one perturbation draw per query head
    two_digit: bool = False     # query codes of two s8 digits (QM_TWO_DIGIT)
                                # with the closed-form residual term
    refine8: bool = False       # 8-bit refinement before the bf16 reads
    QM8: int = 2047             # query code range of the 8-bit bounds


def grid_J(pool: int, r: int) -> int:
    """J = ceil(r log2 |P|): the smallest j with 2^j >= |P|^r (exact)."""
    if pool <= 1:
        return 0
    target = pool ** r
    j = 0
    while (1 << j) < target:
        j += 1
    return j


def dense_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """Exact softmax attention in float64 ("Problem Setup")."""
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    s = K @ q / math.sqrt(q.shape[0])
    w = np.exp(s - s.max())
    return (w @ V) / w.sum(), s


def score_f32(q: np.ndarray, Krows: np.ndarray):
    """float32 rescoring of rows: products fl(q_c k_c), adjacent-pair tree
    sum, times fl(1/sqrt d).  Also the tree sum of |products| (a magnitude
    for the rounding margin).  Returns (s32, mag32) float32 [rows]."""
    q = np.asarray(q, np.float32)
    p = np.asarray(Krows, np.float32) * q[None, :]
    rs = inv_sqrt_d_f32(q.shape[0])
    s = tree_sum_f32(p) * rs
    mag = tree_sum_f32(np.abs(p)) * rs
    return s.astype(np.float32), mag.astype(np.float32)


def cstar_lower_f32(q: np.ndarray, Krows: np.ndarray) -> np.float32:
    """cb = max over rows of fl(s32 - fl(mag32 * 2^-13)) <= exact max score."""
    s32, mag = score_f32(q, Krows)
    return F((s32 - mag * _CB_MARG).max())


def bound_levels_f32(ubar: np.ndarray, cb: np.float32, t: np.ndarray,
                     r: int) -> np.ndarray:
    """jbar_i (int64) from float32 ubar, cb and t (step 6)."""
    xb = ((ubar - F(cb)) * LOG2E_F32) + t
    y = (F(-r) * xb) - _LVL_SHIFT
    return np.maximum(np.ceil(y), 0).astype(np.int64)


def exact_levels(sp: np.ndarray, c_star: float, t: np.ndarray, r: int):
    """Exact inclusion and heavy levels (step 7), float64.

    x_i = (s_i - c*) log2 e + t_i;  j_i = max(0, ceil(-r x_i)) is the first
    level whose sample S(tau_j) contains i (ties included:
    s_i - c* + E_i >= log tau_j  <=>  -r x_i <= j);
    h_i = max(0, ceil(-r (s_i - c*) log2 e)) is the first level where
    w_i >= tau_j.  ``t`` may carry leading axes (several seeds).
    """
    sp = np.asarray(sp, np.float64)
    y = (sp - c_star) / math.log(2.0)
    x = y + np.asarray(t, np.float64)
    jl = np.maximum(np.ceil(-r * x), 0).astype(np.int64)
    hl = np.maximum(np.ceil(-r * y), 0).astype(np.int64)
    return jl, np.broadcast_to(hl, jl.shape)


def level_sums(jl, hl, w, Vp, D_R, N_R, nL):
    """Per-level sums over the pool for levels 0..nL-1 (step 8).

    Heavy B_j = {h_i <= j}: D_B, N_B, H_B (weights w_i).  Light sampled
    S cap A_j = {j_i <= j < h_i}: k (count), S1 = sum v, S2 = sum ||v||^2,
    Gs = sum ||v - c_j||^2 with the level's centre
    c_j = (N_R + N_B) / (D_R + D_B).  Returns a dict of arrays.
    """
    Vp = np.asarray(Vp, np.float64)
    d = Vp.shape[1]
    vn2 = (Vp * Vp).sum(axis=1)
    out = {key: np.zeros(nL) for key in ("k", "S2", "Gs", "D_B", "H_B",
                                          "n_sampled")}
    out["S1"] = np.zeros((nL, d))
    out["N_B"] = np.zeros((nL, d))
    for j in range(nL):
        heavy = hl <= j
        light = (jl <= j) & ~heavy
        out["D_B"][j] = w[heavy].sum()
        out["N_B"][j] = w[heavy] @ Vp[heavy]
        out["H_B"][j] = w[heavy] @ vn2[heavy]
        out["k"][j] = light.sum()
        out["S1"][j] = Vp[light].sum(axis=0)
        out["S2"][j] = vn2[light].sum()
        out["n_sampled"][j] = (jl <= j).sum()
        cj = (N_R + out["N_B"][j]) / (D_R + out["D_B"][j])
        out["Gs"][j] = ((Vp[light] - cj[None, :]) ** 2).sum()
    return out


@dataclasses.dataclass
class GroupResult:
    o: np.ndarray              # [G, d] float64
    beta: np.ndarray           # [G]
    level: np.ndarray          # [G] int
    keys_read: np.ndarray      # [G] int
    values_read: np.ndarray    # [G] int
    n_candidates: np.ndarray   # [G] int
    n_near: np.ndarray         # [G] int (near-threshold keys at the stop)
    J: int
    detail: list               # per-head dict (levels, bounds, sets ...)
    rows8: Optional[np.ndarray] = None   # [G] int: 8-bit rows read (refine8)


def oracle_decode_group(q: np.ndarray, K: np.ndarray, V: np.ndarray, n: int,
                        step_seed: int, g: int, p: Params,
                        quant: Optional[tuple] = None,
                        keep_detail: bool = True,
                        quant8: Optional[tuple] = None) -> GroupResult:
    """Decode step for query heads q [G, d] of one KV group.

    K, V float32 [>= n, d] (exact values of the cache).  ``quant`` may pass a
    precomputed (codes, packed, mins, deltas, vmax) from the oracle's own
    quantiser; otherwise it is computed here.  With ``p.refine8``, ``quant8``
    may pass the (codes8, mins, deltas8) of ``quantize_keys8`` likewise.
    """
    q = np.asarray(q, np.float32)
    Gh, d = q.shape
    K = np.asarray(K[:n], np.float32)
    V = np.asarray(V[:n], np.float32)
    pool = max(n - WINDOW, 0)
    if quant is None:
        codes, _, mins, deltas = quantize_keys(K, n)
        vmax = vmax_blocks(V, n)
    else:
        codes, _, mins, deltas, vmax = quant
    J = grid_J(pool, p.r) if p.J_override < 0 else int(p.J_override)
    out_o = np.zeros((Gh, d))
    out_beta = np.zeros(Gh)
    out_lvl = np.zeros(Gh, np.int64)
    out_kr = np.zeros(Gh, np.int64)
    out_vr = np.zeros(Gh, np.int64)
    out_nc = np.zeros(Gh, np.int64)
    out_near = np.zeros(Gh, np.int64)
    out_r8 = np.zeros(Gh, np.int64) if p.refine8 else None
    details = []
    Kd = K.astype(np.float64)
    Vd = V.astype(np.float64)
    vnorm2 = (Vd * Vd).sum(axis=1)
    if pool == 0:
        for h in range(Gh):
            o, _ = dense_attention(q[h], K, V)
            out_o[h] = o
            out_kr[h] = n
            out_vr[h] = n
            details.append({})
        return GroupResult(out_o, out_beta, out_lvl, out_kr, out_vr, out_nc,
                           out_near, J, details, out_r8)
    if p.refine8:
        codes8, mins8, deltas8 = (quant8 if quant8 is not None
                                  else quantize_keys8(K, n))
    delta_e = p.delta / (4.0 * (J + 1))
    nblk_pool = (pool + T_BLOCK - 1) // T_BLOCK
    Vmax = float(vmax[:nblk_pool].max())
    t_shared = None if p.per_head else perturb_t(step_seed, g, np.arange(pool))
    win = np.arange(pool, n)
    levels = np.arange(J + 1)
    tau = 2.0 ** (-levels / p.r)
    for h in range(Gh):
        # the perturbation: shared by the group, or the head's own draw
        t = (perturb_t(step_seed, head_stream(g, Gh, h), np.arange(pool))
             if p.per_head else t_shared)                  # float32 [pool]
        # step 2: bounds
        if p.two_digit:
            at, alpha, b_hi, b_lo = query_prep(q[h], mins, deltas,
                                               QM_TWO_DIGIT,
                                               closed_residual=True)
        else:
            at, alpha, b_hi, b_lo = query_prep(q[h], mins, deltas, p.QM)
        ubar, low, _ = key_bounds(codes, at, alpha, b_hi, b_lo, n)
        c_lo = F(low.max())
        # step 3: exact maximum over R and {ubar >= c*_lo}
        cset = np.nonzero(ubar[:pool] >= c_lo)[0]
        rows = np.concatenate([cset, win])
        s = Kd @ q[h].astype(np.float64) / math.sqrt(d)
        c_star = s[rows].max()
        cb = cstar_lower_f32(q[h], K[rows])
        # step 6: candidates
        jbar = bound_levels_f32(ubar[:pool], cb, t, p.r)
        # optional 8-bit refinement: the level from the tighter of the two
        # upper bounds (never below jbar, never above the exact level)
        if p.refine8:
            at8, al8, bh8, bl8 = query_prep(q[h], mins8, deltas8, p.QM8,
                                            levels=255)
            ubar8, _, _ = key_bounds(codes8, at8, al8, bh8, bl8, n)
            jref = bound_levels_f32(np.minimum(ubar[:pool], ubar8[:pool]), cb,
                                    t, p.r)
        else:
            ubar8, jref = None, jbar
        cand = jbar <= J
        # step 7: exact levels (all pool keys computed for the invariant
        # checks; only candidates enter the estimate)
        sp = s[:pool]
        jl, hl = exact_levels(sp, c_star, t, p.r)
        jl_c = np.where(cand, jl, J + 1)
        hl_c = np.where(cand, hl, J + 1)
        w = np.exp(s - c_star)
        wr = w[win]
        D_R = wr.sum()
        N_R = wr @ Vd[win]
        H_R = wr @ vnorm2[win]
        # step 8: per-level sums (only candidates can enter)
        nL = J + 1
        sums = level_sums(jl_c, hl_c, w[:pool], Vd[:pool], D_R, N_R, nL)
        k, S1, S2, Gs = sums["k"], sums["S1"], sums["S2"], sums["Gs"]
        D_B, N_B, H_B = sums["D_B"], sums["N_B"], sums["H_B"]
        cert = certificate_levels(tau, k, S1, Gs, S2, D_B, N_B, H_B, D_R, N_R,
                                  H_R, Vmax, delta_e, p.eps, p.measure,
                                  delta=p.delta)
        ok = np.nonzero(cert["certified"])[0]
        if len(ok):
            js = int(ok[0])
            out_o[h] = cert["o_hat"][js]
            out_beta[h] = cert["beta"][js]
            out_lvl[h] = js
            rset = np.union1d(cset, np.nonzero(jref <= js)[0])
            if p.refine8:
                out_r8[h] = len(np.setdiff1d(np.nonzero(jbar <= js)[0], cset))
            out_kr[h] = WINDOW + len(rset)
            out_vr[h] = WINDOW + int((jl_c <= js).sum())
            xs = (sp - c_star) + t.astype(np.float64) * math.log(2.0)
            thr = -(js / p.r) * math.log(2.0)
            near = (np.abs(xs - thr) < NEAR_BAND) | \
                   (np.abs((sp - c_star) - thr) < NEAR_BAND)
            out_near[h] = int((near & cand).sum())
        else:
            js = J + 1
            o, _ = dense_attention(q[h], K, V)
            out_o[h] = o
            out_beta[h] = 0.0
            out_lvl[h] = js
            out_kr[h] = n
            out_vr[h] = n
            if p.refine8:
                out_r8[h] = len(np.setdiff1d(np.nonzero(cand)[0], cset))
        out_nc[h] = int(cand.sum())
        if keep_detail:
            details.append({
                "ubar": ubar, "low": low, "c_lo": c_lo, "c_hi": F(ubar.max()),
                "cset": cset, "c_star": c_star, "cb": cb, "jbar": jbar,
                "cand": cand, "jl": jl, "hl": hl, "s": s, "w": w,
                "tau": tau, "cert": cert, "sums": sums, "jl_c": jl_c,
                "hl_c": hl_c, "k": k, "D_B": D_B, "S2": S2,
                "D_R": D_R, "N_R": N_R, "H_R": H_R, "Vmax": Vmax,
                "delta_e": delta_e, "t": t, "alpha": alpha, "b_hi": b_hi,
                "b_lo": b_lo, "at": at, "stop": js, "ubar8": ubar8,
                "jref": jref})
        else:
            details.append({"stop": js})
    return GroupResult(out_o, out_beta, out_lvl, out_kr, out_vr, out_nc,
                       out_near, J, details, out_r8)
