"""The synthetic input recipe: both back ends of ``synth`` draw the laws the
generator's header states (the stand-in for the Llama-3.1-8B KV caches the
pages measure on), and the draws are reproducible from their seeds."""
import math

import numpy as np
import pytest

import synth


def _small(**over):
    return synth.workload("llama16k", n=4096, Hq=8, Hkv=2, **over)


def _check_keys_values(K, V, mus, nus, needles, w):
    d = w.d
    oc = synth.outlier_channels(d)
    rest = [c for c in range(d) if c not in oc]
    for b in range(w.B):
        for g in range(w.Hkv):
            k = K[b, g].astype(np.float64)
            mask = np.ones(len(k), bool)
            mask[needles[b, g]] = False
            z = k[mask] - 4.0 * mus[g][None, :]
            # mean 4 mu_g, unit variance, outlier channels x8 (variance 64)
            sd = np.where(np.isin(np.arange(d), oc), 8.0, 1.0)
            assert np.all(np.abs(z.mean(axis=0)) < 5.0 * sd / math.sqrt(len(z)))
            var = z.var(axis=0)
            assert np.all(np.abs(var[rest] - 1.0) < 0.12)
            assert np.all(np.abs(var[oc] / 64.0 - 1.0) < 0.12)
            # needles sit 8 nu_g above the key law along nu_g
            proj_n = (k[~mask] - 4.0 * mus[g]) @ nus[g]
            assert abs(proj_n.mean() - 8.0) < 1.5
            # values: lambda * N(0, I), log lambda ~ N(0, 0.5^2): the
            # per-row norm is lambda * chi_d, so log ||v|| has mean
            # log sqrt(d) (to O(1/d)) and spread 0.5 (plus chi's)
            lv = np.log(np.linalg.norm(V[b, g].astype(np.float64), axis=1))
            assert abs(lv.mean() - 0.5 * math.log(d)) < 0.05
            assert abs(lv.std() - 0.5) < 0.05


def test_numpy_back_end_laws():
    w = _small()
    K, V, meta = synth.kv_numpy(w)
    assert K.shape == (w.B, w.Hkv, w.n, w.d) and K.dtype == np.float32
    # bf16 workloads hold bf16-representable values
    assert np.array_equal(synth.bf16_round_np(K), K)
    assert np.array_equal(synth.bf16_round_np(V), V)
    _check_keys_values(K, V, meta["mu"], meta["nu"], meta["needles"], w)
    # needles are distinct pool positions (never in the 64-token window)
    nd = meta["needles"]
    assert np.all(nd < w.n - synth.WINDOW)
    assert all(len(set(nd[b, g])) == w.n_needles for b in range(w.B)
               for g in range(w.Hkv))


def test_torch_back_end_laws():
    torch = pytest.importorskip("torch")
    w = _small()
    K, V, meta = synth.kv_torch(w)
    assert K.dtype == torch.bfloat16 and tuple(K.shape) == (w.B, w.Hkv, w.n, w.d)
    _check_keys_values(K.float().numpy(), V.float().numpy(),
                       meta["mu"].numpy(), meta["nu"].numpy(),
                       meta["needles"].numpy(), w)


def test_queries_peaked_and_near_uniform_groups():
    """Peaked groups: q = sqrt(d) nu_g + N(0, I), so a needle scores ~8
    above the other keys; odd groups are the same draw scaled by 0.1."""
    w = _small(B=1)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, step=0)
    torch = pytest.importorskip("torch")
    qt = synth.q_torch(w, {k: torch.from_numpy(np.asarray(v)) for k, v in
                           meta.items()}, step=0).float().numpy()
    for qq in (q, qt):
        for h in range(w.Hq):
            g = h // w.G
            along = qq[0, h] @ meta["nu"][g]
            scale = w.flat_scale if g % 2 == 1 else 1.0
            assert abs(along / (scale * math.sqrt(w.d)) - 1.0) < 0.4
    for g in range(0, w.Hkv, 2):
        s = K[0, g].astype(np.float64) @ q[0, g * w.G].astype(np.float64) \
            / math.sqrt(w.d)
        nd = meta["needles"][0, g]
        other = np.delete(s, nd)
        assert 6.0 < s[nd].mean() - other.mean() < 10.0


def test_tiny_case_planted_keys():
    w = synth.workload("tiny")
    K, V, meta = synth.kv_numpy(w)
    assert w.dtype == "f32" and w.d == 64 and w.n == 2048
    q = synth.q_numpy(w, meta, step=3, K=K)
    nd = meta["needles"][0, 0]
    assert len(nd) == 8
    target = 3.0 * q[0, 0] / np.linalg.norm(q[0, 0])
    assert np.allclose(K[0, 0, nd], target[None, :], rtol=0, atol=1e-6)


def test_stress_regimes():
    """flat: q scaled by 0.05; adversarial: the same keys as flat plus 6 nu_g
    on exactly ceil(eps^-2) pool keys; heavy: the same keys plus
    non-negative Pareto(1.5) - 1 boosts along nu_g (a heavy right tail)."""
    n = 2048
    flat = dataclass_small(synth.stress(n, 0.05, "flat"))
    K, V, meta = synth.kv_numpy(flat)
    q = synth.q_numpy(flat, meta)
    assert np.abs(q).max() < 0.05 * (math.sqrt(128) + 6)
    nu = meta["nu"][0].astype(np.float64)
    base = K[0, 0].astype(np.float64) @ nu
    adv = dataclass_small(synth.stress(n, 0.05, "adversarial"))
    Ka, _, _ = synth.kv_numpy(adv)
    diff = Ka[0, 0].astype(np.float64) @ nu - base
    m = math.ceil(0.05 ** -2)
    assert int((np.abs(diff - 6.0) < 0.5).sum()) == m
    assert int((np.abs(diff) < 0.5).sum()) == n - m
    heavy = dataclass_small(synth.stress(n, 0.05, "heavy"))
    Kh, _, _ = synth.kv_numpy(heavy)
    boost = Kh[0, 0].astype(np.float64) @ nu - base
    assert boost.min() > -0.5
    # Pareto(1.5) - 1 (Lomax): P(X > x) = (1 + x)^-1.5
    for x in (1.0, 3.0):
        frac = (boost > x).mean()
        p = (1.0 + x) ** -1.5
        assert abs(frac - p) < 4 * math.sqrt(p * (1 - p) / n) + 0.02


def dataclass_small(w):
    import dataclasses
    return dataclasses.replace(w, Hq=4, Hkv=1)


def test_seeds_reproducible_and_distinct():
    w = _small()
    K1, _, _ = synth.kv_numpy(w, layer=2)
    K2, _, _ = synth.kv_numpy(w, layer=2)
    K3, _, _ = synth.kv_numpy(w, layer=3)
    assert np.array_equal(K1, K2) and not np.array_equal(K1, K3)
    s0 = synth.step_seeds(w, 0)
    assert np.array_equal(s0, synth.step_seeds(w, 0))
    allseeds = np.concatenate([synth.step_seeds(w, s, layer=l)
                               for s in range(8) for l in range(4)])
    assert len(set(allseeds.tolist())) == len(allseeds)
