"""Pins for the optional 8-bit refinement of the oracle's decode step.

picx.dev summary, "Algorithm Components" 4: an 8-bit stage sits between the
4-bit scan and the exact 16-bit reads.  It tightens the candidates' upper
bounds, so it may only change which bf16 rows the step reads, never the
sample, the estimate, the certificate or the stop level: every key of the
sample at the stop level must still have its row read.
"""
import numpy as np

import synth
from oracle.step import Params, oracle_decode_group


def _group(n=3000, **over):
    w = synth.workload("llama16k", B=1, n=n, Hq=8, Hkv=2, **over)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, 0)
    seed = int(synth.step_seeds(w, 0)[0])
    return w, K, V, q, seed


def _both(w, K, V, q, seed, g, **pover):
    base = Params(w.eps, w.delta, w.r, **pover)
    ref = Params(w.eps, w.delta, w.r, refine8=True, **pover)
    G = w.G
    a = oracle_decode_group(q[0, g * G:(g + 1) * G], K[0, g], V[0, g], w.n,
                            seed, g, base)
    b = oracle_decode_group(q[0, g * G:(g + 1) * G], K[0, g], V[0, g], w.n,
                            seed, g, ref)
    return a, b


def test_refinement_changes_no_result():
    w, K, V, q, seed = _group()
    for g in range(w.Hkv):          # group 0 peaked, group 1 near-uniform
        a, b = _both(w, K, V, q, seed, g)
        assert np.array_equal(a.o, b.o) and np.array_equal(a.beta, b.beta)
        assert np.array_equal(a.level, b.level)
        assert np.array_equal(a.values_read, b.values_read)
        assert np.array_equal(a.n_candidates, b.n_candidates)
        assert a.rows8 is None and b.rows8 is not None
        assert np.all(b.keys_read <= a.keys_read)


def test_refined_rows_cover_the_sample_and_counts_agree():
    w, K, V, q, seed = _group()
    P = w.n - 64
    for g in range(w.Hkv):
        a, b = _both(w, K, V, q, seed, g)
        for h in range(w.G):
            det = b.detail[h]
            js = int(b.level[h])
            assert js <= b.J
            jbar, jref, jl = det["jbar"], det["jref"], det["jl_c"]
            cset = det["cset"]
            # jbar <= jref <= exact level for every candidate
            cand = det["cand"]
            assert np.all(jref >= jbar)
            assert np.all(jref[cand] <= det["jl"][cand])
            # every sampled pool key is read at bf16
            read = np.zeros(P, bool)
            read[cset] = True
            read[jref <= js] = True
            assert np.all(read[jl <= js])
            assert b.keys_read[h] == 64 + int(read.sum())
            assert b.keys_read[h] - 64 >= b.values_read[h] - 64
            # 8-bit rows: the 4-bit candidates up to the stop level outside
            # the exact-maximum set
            r8 = np.zeros(P, bool)
            r8[jbar <= js] = True
            r8[cset] = False
            assert b.rows8[h] == int(r8.sum())


def test_refinement_cuts_peaked_rows_per_head_draws_and_measures():
    """On the peaked group the refined bounds drop most of the 4-bit
    candidates' bf16 rows at the stop level; the invariance holds for
    per-query-head draws and the other measures too."""
    w, K, V, q, seed = _group()
    a, b = _both(w, K, V, q, seed, 0)
    assert b.keys_read.sum() - 64 * w.G < 0.6 * (a.keys_read.sum() - 64 * w.G)
    for pover in ({"per_head": True}, {"measure": 1}, {"measure": 2},
                  {"measure": 3}):
        a, b = _both(w, K, V, q, seed, 0, **pover)
        assert np.array_equal(a.o, b.o) and np.array_equal(a.level, b.level)
        assert np.all(b.keys_read <= a.keys_read)


def test_refinement_at_fallback_and_without_pool():
    w, K, V, q, seed = _group(eps=1e-7)
    a, b = _both(w, K, V, q, seed, 0)
    assert np.all(b.level == b.J + 1)
    assert np.array_equal(a.o, b.o) and np.all(b.keys_read == w.n)
    for h in range(w.G):
        det = b.detail[h]
        assert b.rows8[h] == len(np.setdiff1d(np.nonzero(det["cand"])[0],
                                              det["cset"]))
    w, K, V, q, seed = _group(n=50)
    a, b = _both(w, K, V, q, seed, 0)
    assert np.array_equal(a.o, b.o) and np.all(b.rows8 == 0)
