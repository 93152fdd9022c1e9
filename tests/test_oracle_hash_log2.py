"""Pins for the oracle's perturbation source (hash, uniform, own log2).

picx.dev summary, "Algorithm Components" 1: E_i = -ln u_i, with u_i a
uniform number built from 53 hashed bits.  The hash is SplitMix64; its published output vectors pin the
implementation, and distribution tests pin u ~ U(0,1], E ~ Exp(1).
"""
import numpy as np
import pytest
from scipy import stats

from oracle.fp32 import log2_m53_f32
from oracle.hashing import (GAMMA, PER_HEAD_STREAM, group_key, head_stream,
                            key_hashes, mix64, perturb_t)


def test_splitmix64_published_outputs():
    # First three outputs of the reference splitmix64.c (Vigna) seeded with
    # 0, as listed with that generator.
    with np.errstate(over="ignore"):
        z = np.arange(1, 4, dtype=np.uint64) * GAMMA
    out = [int(x) for x in mix64(z)]
    assert out == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                   0x06C45D188009454F]


def test_key_hash_is_generator_stream():
    # h_i is the (i+1)-th output of a splitmix64 generator seeded at the
    # group key: consecutive positions differ by exactly one gamma step.
    k = group_key(12345, 3)
    h = key_hashes(12345, 3, np.arange(5))
    with np.errstate(over="ignore"):
        manual = [int(mix64(np.uint64(k) + np.uint64(i + 1) * GAMMA))
                  for i in range(5)]
    assert [int(x) for x in h] == manual


def test_log2_exhaustive_mantissas():
    # every float32 mantissa at three exponents, against float64 log2
    for e in (0, 23, 52):
        if e < 23:
            m = np.arange(1 << e, 1 << (e + 1), dtype=np.uint64)
        else:
            m = (np.uint64(1) << np.uint64(e)) + (
                np.arange(1 << 23, dtype=np.uint64) << np.uint64(e - 23))
        ref = np.log2(m.astype(np.float64))
        got = log2_m53_f32(m).astype(np.float64)
        # half an ulp of the float32 result plus the truncation of m to
        # 24 bits (2^-23 / ln 2 = 1.7e-7)
        ulp = np.spacing(np.maximum(ref, 1.0).astype(np.float32)).astype(
            np.float64)
        assert np.all(np.abs(got - ref) <= 0.5 * ulp + 3.5e-7)


def test_log2_exact_powers_of_two():
    m = np.array([1 << k for k in range(54)], dtype=np.uint64)
    assert np.array_equal(log2_m53_f32(m), np.arange(54, dtype=np.float32))


def test_log2_random_53bit():
    rng = np.random.default_rng(1)
    m = rng.integers(1, 2 ** 53, size=200000, dtype=np.uint64)
    ref = np.log2(m.astype(np.float64))
    assert np.max(np.abs(log2_m53_f32(m) - ref)) < 2.5e-6


def test_uniform_and_exponential_laws():
    n = 400000
    t = perturb_t(987654321, 5, np.arange(n)).astype(np.float64)
    assert np.all(t >= 0.0) and np.all(np.isfinite(t))
    E = t * np.log(2.0)
    assert stats.kstest(E, "expon").pvalue > 1e-3
    u = 2.0 ** (-t)
    assert stats.kstest(u, "uniform").pvalue > 1e-3
    # mean of Exp(1) within 5 standard errors
    assert abs(E.mean() - 1.0) < 5.0 / np.sqrt(n)


def test_streams_uncorrelated_across_groups_and_steps():
    n = 200000
    a = perturb_t(1, 0, np.arange(n)).astype(np.float64)
    b = perturb_t(1, 1, np.arange(n)).astype(np.float64)
    c = perturb_t(2, 0, np.arange(n)).astype(np.float64)
    for x, y in ((a, b), (a, c), (b, c)):
        assert abs(np.corrcoef(x, y)[0, 1]) < 5.0 / np.sqrt(n)
    # lag-1 autocorrelation within a stream
    assert abs(np.corrcoef(a[:-1], a[1:])[0, 1]) < 5.0 / np.sqrt(n)


@pytest.mark.parametrize("seed", [0, 2 ** 64 - 1, 0x123456789ABCDEF])
def test_u_in_unit_interval(seed):
    h = key_hashes(seed, 0, np.arange(1000))
    m = (h >> np.uint64(11)) + np.uint64(1)
    assert m.min() >= 1 and m.max() <= 2 ** 53


def test_per_head_streams():
    # per-query-head draws: stream ids never meet the KV-group ids, each
    # head's draw is Exp(1) in nats and the heads' draws are uncorrelated
    # with each other and with the group's shared draw
    G, n = 4, 200000
    ids = [head_stream(g, G, h) for g in range(64) for h in range(G)]
    assert len(set(ids)) == len(ids) and min(ids) >= PER_HEAD_STREAM
    draws = [perturb_t(77, head_stream(3, G, h), np.arange(n)).astype(np.float64)
             for h in range(G)]
    shared = perturb_t(77, 3, np.arange(n)).astype(np.float64)
    for h in range(G):
        assert stats.kstest(draws[h] * np.log(2.0), "expon").pvalue > 1e-3
        assert abs(np.corrcoef(draws[h], shared)[0, 1]) < 5.0 / np.sqrt(n)
        for h2 in range(h + 1, G):
            assert abs(np.corrcoef(draws[h], draws[h2])[0, 1]) < 5.0 / np.sqrt(n)
