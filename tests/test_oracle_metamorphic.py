"""Metamorphic pins of the stop rule and the estimate (no worked example is
printed on the pages, so these relate runs of the oracle to each other by
properties the method must have; picx.dev summary, "Problem Setup" and
"Algorithm Components" 3):

* the certificate beta of every level does not involve eps, so a larger
  eps can only stop at the same level or earlier, under every measure;
* a larger delta loosens every confidence term (Chernoff, G, Z, H), so it
  can only stop at the same level or earlier;
* doubling every value doubles o_hat and beta and keeps the stop level (the
  value scale, the output norm and the value bound all scale with v);
* adding the same amount to every score (keys shifted along a direction the
  query sees as a constant) changes the 4-bit bounds and the candidates but
  not the weights w_i = exp(s_i - c*), hence not the result;
* with the group's shared draw, permuting a group's query heads permutes
  their results.
"""
import numpy as np
import pytest

import synth
from oracle.step import Params, oracle_decode_group


def _group(n=2000, G=4, seed_step=0):
    w = synth.workload("llama16k", B=1, n=n, Hq=2 * G, Hkv=2)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, 0)
    seed = int(synth.step_seeds(w, seed_step)[0])
    return w, K, V, q, seed


def _run(w, K, V, q, seed, g, **p):
    G = w.G
    base = dict(eps=w.eps, delta=w.delta, r=w.r)
    base.update(p)
    return oracle_decode_group(q[0, g * G:(g + 1) * G], K[0, g], V[0, g], w.n,
                               seed, g, Params(**base))


@pytest.mark.parametrize("measure", [0, 1, 2, 3])
def test_stop_level_monotone_in_eps(measure):
    w, K, V, q, seed = _group()
    for g in range(w.Hkv):
        prev, beta0 = None, None
        for eps in (0.02, 0.05, 0.1, 0.2):
            res = _run(w, K, V, q, seed, g, eps=eps, measure=measure)
            if prev is not None:
                assert np.all(res.level <= prev), (measure, g, eps)
            prev = res.level
            # the per-level beta is the same whatever eps
            b = np.stack([d["cert"]["beta"] for d in res.detail])
            if beta0 is None:
                beta0 = b
            assert np.array_equal(b, beta0)


@pytest.mark.parametrize("measure", [0, 1, 2])
def test_stop_level_monotone_in_delta(measure):
    w, K, V, q, seed = _group()
    for g in range(w.Hkv):
        prev, bprev = None, None
        for delta in (0.01, 0.05, 0.2):
            res = _run(w, K, V, q, seed, g, delta=delta, measure=measure)
            b = np.stack([d["cert"]["beta"] for d in res.detail])
            if prev is not None:
                assert np.all(res.level <= prev), (measure, g, delta)
                # every level's beta shrinks (or stays infinite)
                fin = np.isfinite(bprev)
                assert np.all(b[fin] <= bprev[fin])
            prev, bprev = res.level, b


def test_doubling_values_doubles_estimate_and_beta():
    w, K, V, q, seed = _group()
    for g in range(w.Hkv):
        a = _run(w, K, V, q, seed, g)
        b = _run(w, K, 2.0 * V, q, seed, g)
        assert np.array_equal(a.level, b.level)
        assert np.allclose(b.o, 2.0 * a.o, rtol=1e-12, atol=0)
        assert np.allclose(b.beta, 2.0 * a.beta, rtol=1e-12, atol=0)
        assert np.array_equal(a.keys_read, b.keys_read)


def test_common_score_shift_changes_no_result():
    # one query head per group (G = 1): keys shifted by an integer vector u
    # (exact in float32 for these bf16 keys) raise every score of the head
    # by the same q.u / sqrt(d)
    w, K, V, q, seed = _group(G=1)
    for g in range(w.Hkv):
        qq = q[0, g].astype(np.float64)
        u = np.rint(4.0 * qq / np.linalg.norm(qq)).astype(np.float32)
        assert abs(float(qq @ u)) > 1.0
        Ks = K.copy()
        Ks[0, g] = K[0, g] + u[None, :]
        assert np.array_equal(Ks[0, g] - u[None, :], K[0, g])   # exact
        a = _run(w, K, V, q, seed, g)
        b = _run(w, Ks, V, q, seed, g)
        assert np.array_equal(a.level, b.level)
        assert np.allclose(b.o, a.o, rtol=1e-9, atol=1e-12)
        assert np.allclose(b.beta, a.beta, rtol=1e-9, atol=1e-12)
        assert np.array_equal(a.values_read, b.values_read)


def test_permuting_query_heads_permutes_results():
    # with the group's shared draw, a head's result depends on its own query
    # only: reversing the heads of a group reverses the outputs exactly
    w, K, V, q, seed = _group()
    G = w.G
    for g in range(w.Hkv):
        a = _run(w, K, V, q, seed, g)
        qr = q.copy()
        qr[0, g * G:(g + 1) * G] = q[0, g * G:(g + 1) * G][::-1]
        b = _run(w, K, V, qr, seed, g)
        assert np.array_equal(a.o[::-1], b.o)
        assert np.array_equal(a.beta[::-1], b.beta)
        assert np.array_equal(a.level[::-1], b.level)
        assert np.array_equal(a.keys_read[::-1], b.keys_read)
