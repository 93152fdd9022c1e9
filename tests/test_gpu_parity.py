"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Bit-exact: the 4-bit codes, block bounds and value-norm bounds; every key's
upper bound ubar; c*_lo, c*_hi and cb; the candidate sets.  Set membership:
bit-exact except keys within 1e-5 nats of a threshold in perturbed
log-score (counted).  Outputs o and certificates beta: within 2e-3 relative
of the oracle evaluated with the device's memberships (which differ from the
oracle's only at the near-threshold keys).  Stop levels agree except where
the oracle's certificate sits within 0.2 % of its target.
"""
import math

import numpy as np
import pytest

import synth
from oracle.certificate import certificate_levels
from oracle.hashing import perturb_t
from oracle.quantize import quantize_keys, value_sq_norms_f32, vmax_blocks
from oracle.step import (Params, bound_levels_f32, dense_attention,
                         level_sums, oracle_decode_group)
from tests.gpu_common import GpuRun, ensure_built, gpu_levels, to_dev

pytestmark = pytest.mark.gpu

TOL = 2e-3
NEAR = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _case(name, n, step=0, B=1, **over):
    w = synth.workload(name, B=B, n=n, **over)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, step, K=K)
    return w, K, V, q


# ----------------------------------------------------------------- quantiser

@pytest.mark.parametrize("name,n,over", [
    ("tiny", 2048, {}), ("tiny", 1000, {}),
    ("llama16k", 1337, {"Hq": 8, "Hkv": 2}),
    ("llama16k", 130, {"Hq": 4, "Hkv": 4, "d": 64})])
def test_quantizer_bit_exact(name, n, over):
    import torch
    import certified_sparse_attention_gb300 as csa
    w, K, V, q = _case(name, n, **over)
    n_alloc = n + 75
    shape = csa.make_shape(w.B, w.Hq, w.Hkv, w.d, n_alloc, w.dtype)
    Kp = np.zeros((w.B, w.Hkv, n_alloc, w.d), np.float32)
    Vp = np.zeros_like(Kp)
    Kp[:, :, :n], Vp[:, :, :n] = K, V
    Kt, Vt = to_dev(Kp, w.dtype, "cuda"), to_dev(Vp, w.dtype, "cuda")
    K4, bounds, vmax, vnorm2 = csa.meta_buffers(shape, "cuda")
    csa.check(csa.csa_quantize_keys(shape, Kt, Vt, [n] * w.B, 0, K4, bounds,
                                    vmax, vnorm2))
    torch.cuda.synchronize()
    for g in range(w.Hkv):
        codes, packed, mins, deltas = quantize_keys(K[0, g], n)
        vm = vmax_blocks(V[0, g], n)
        nb = mins.shape[0]
        assert np.array_equal(K4[0, g, :nb * 64].cpu().numpy(), packed)
        assert np.array_equal(bounds[0, g, :nb, 0].cpu().numpy(), mins)
        assert np.array_equal(bounds[0, g, :nb, 1].cpu().numpy(), deltas)
        assert np.array_equal(vmax[0, g, :nb].cpu().numpy(), vm)
        vn = vnorm2[0, g].cpu().numpy()
        assert np.array_equal(vn[:n], value_sq_norms_f32(V[0, g], n))
        assert not vn[n:nb * 64].any()


def test_quantizer_append_one_block():
    # decode append: write token n, rebuild only its block
    import torch
    import certified_sparse_attention_gb300 as csa
    w, K, V, q = _case("llama16k", 1000, Hq=4, Hkv=1)
    n_alloc = 1100
    shape = csa.make_shape(1, 4, 1, 128, n_alloc, "bf16")
    Kp = np.zeros((1, 1, n_alloc, 128), np.float32)
    Vp = np.zeros_like(Kp)
    Kp[:, :, :1000], Vp[:, :, :1000] = K, V
    Kt, Vt = to_dev(Kp, "bf16", "cuda"), to_dev(Vp, "bf16", "cuda")
    K4, bounds, vmax, vnorm2 = csa.meta_buffers(shape, "cuda")
    csa.check(csa.csa_quantize_keys(shape, Kt, Vt, [1000], 0, K4, bounds, vmax,
                                    vnorm2))
    rng = np.random.default_rng(5)
    newk = synth.bf16_round_np(rng.standard_normal(128).astype(np.float32) * 3)
    newv = synth.bf16_round_np(rng.standard_normal(128).astype(np.float32))
    Kt[0, 0, 1000] = torch.from_numpy(newk).to(Kt)
    Vt[0, 0, 1000] = torch.from_numpy(newv).to(Vt)
    csa.check(csa.csa_quantize_keys(shape, Kt, Vt, [1001], 1000, K4, bounds,
                                    vmax, vnorm2))
    torch.cuda.synchronize()
    Kn = np.concatenate([K[0, 0], newk[None]], 0)
    Vn = np.concatenate([V[0, 0], newv[None]], 0)
    codes, packed, mins, deltas = quantize_keys(Kn, 1001)
    assert np.array_equal(K4[0, 0, :len(packed)].cpu().numpy(), packed)
    assert np.array_equal(bounds[0, 0, :len(mins), 0].cpu().numpy(), mins)
    assert np.array_equal(bounds[0, 0, :len(mins), 1].cpu().numpy(), deltas)
    assert np.array_equal(vmax[0, 0, :len(mins)].cpu().numpy(),
                          vmax_blocks(Vn, 1001))
    assert np.array_equal(vnorm2[0, 0, :1001].cpu().numpy(),
                          value_sq_norms_f32(Vn, 1001))


# ------------------------------------------------------------- decode step

def _compare_group(run, w, K, V, q, b, g, res, p, report):
    ub = run.ubar()
    cm = run.cmax()
    s32 = run.s32()
    o_g, beta_g, lvl_g, kr_g, stats = run.outputs()
    n = run.lens[b]
    P = n - 64
    J = res.J
    Vd = V[b, g, :n].astype(np.float64)
    t = perturb_t(run.seeds[b], g, np.arange(P))
    needK, needV = set(), set()
    for h in range(w.G):
        hq = g * w.G + h
        det = res.detail[h]
        # bit-exact bounds, maxima and candidates
        assert np.array_equal(ub[b, g, :n, h], det["ubar"]), (b, g, h)
        assert cm[b, hq, 0] == det["c_lo"] and cm[b, hq, 1] == det["c_hi"]
        assert cm[b, hq, 2] == det["cb"]
        cand_g = np.isfinite(s32[b, g, :P, h])
        assert np.array_equal(cand_g, det["cand"]), (b, g, h)
        assert stats[b, hq, 3] == res.n_candidates[h]
        # memberships: device float32 vs oracle float64
        c32 = cm[b, hq, 3]
        jg, hg = gpu_levels(s32[b, g, :P, h], c32, t, p.r, J)
        # levels beyond the grid are all "never" (J + 1)
        jo = np.minimum(det["jl_c"], J + 1)
        ho = np.minimum(det["hl_c"], J + 1)
        jg = np.where(cand_g, jg, J + 1)
        hg = np.where(cand_g, hg, J + 1)
        sp = det["s"][:P] - det["c_star"]
        xs = sp + t.astype(np.float64) * math.log(2.0)
        for gl, ol, val in ((jg, jo, xs), (hg, ho, sp)):
            bad = np.nonzero(gl != ol)[0]
            jm = np.minimum(gl[bad], ol[bad])
            thr = -(jm / p.r) * math.log(2.0)
            assert np.all(np.abs(val[bad] - thr) < NEAR), (b, g, h, bad)
            report["flips"] += len(bad)
        # oracle re-evaluated with the device's memberships
        jr = np.where(jg != jo, jg, jo)
        hr = np.where(hg != ho, hg, ho)
        sums = level_sums(jr, hr, det["w"][:P], Vd[:P], det["D_R"],
                          det["N_R"], J + 1)
        cert = certificate_levels(det["tau"], sums["k"], sums["S1"],
                                  sums["Gs"], sums["S2"], sums["D_B"],
                                  sums["N_B"], sums["H_B"], det["D_R"],
                                  det["N_R"], det["H_R"], det["Vmax"],
                                  det["delta_e"], p.eps, p.measure)
        ok = np.nonzero(cert["certified"])[0]
        ref_lvl = int(ok[0]) if len(ok) else J + 1
        gl = int(lvl_g[b, hq])
        if gl != ref_lvl:
            jm = min(gl, ref_lvl)
            assert jm <= J
            tgt = p.eps * cert["scale_lo"][jm]
            assert abs(cert["beta"][jm] - tgt) <= 2e-3 * tgt, (gl, ref_lvl)
            report["level_flips"] += 1
        if gl <= J:
            o_ref = cert["o_hat"][gl]
            b_ref = cert["beta"][gl]
            assert abs(beta_g[b, hq] - b_ref) <= TOL * b_ref
            kr = 64 + len(np.union1d(det["cset"],
                                     np.nonzero(det["jbar"] <= gl)[0]))
            assert kr_g[b, hq] == kr
            assert stats[b, hq, 2] == 64 + int((jr <= gl).sum())
        else:
            o_ref, _ = dense_attention(q[b, hq], K[b, g, :n], V[b, g, :n])
            assert beta_g[b, hq] == 0 and kr_g[b, hq] == n
        err = np.linalg.norm(o_g[b, hq] - o_ref)
        assert err <= TOL * np.linalg.norm(o_ref) + 1e-6, (b, g, h, err)
        report["heads"] += 1
        report["levels"].append(gl)
        # rows the head needs, for the group unions
        if gl <= J:
            needK.update(np.union1d(det["cset"],
                                    np.nonzero(det["jbar"] <= gl)[0]).tolist())
            needV.update(np.nonzero(jr <= gl)[0].tolist())
        else:
            needK.update(range(P))
            needV.update(range(P))
    for h in range(w.G):
        hq = g * w.G + h
        assert stats[b, hq, 7] == 64 + len(needK)
        assert stats[b, hq, 8] == 64 + len(needV)


def _run_and_compare(w, K, V, q, lens, seeds, n_alloc, **pover):
    run = GpuRun(w, K, V, q, lens, seeds, n_alloc, **pover)
    p = Params(run.params.eps, run.params.delta, run.params.r,
               measure=run.params.measure, J_override=run.params.J_override)
    report = {"flips": 0, "level_flips": 0, "heads": 0, "levels": []}
    for b in range(w.B):
        n = run.lens[b]
        if n <= 64:
            continue
        for g in range(w.Hkv):
            res = oracle_decode_group(q[b, g * w.G:(g + 1) * w.G], K[b, g],
                                      V[b, g], n, run.seeds[b], g, p)
            _compare_group(run, w, K, V, q, b, g, res, p, report)
    return run, report


@pytest.mark.parametrize("step", [0, 1, 2])
def test_decode_tiny_config(step):
    # one head, d=64, n=2048, fp32, planted keys, eps .05 delta .01 r 2
    w, K, V, q = _case("tiny", 2048, step=step)
    seeds = synth.step_seeds(w, step)
    run, rep = _run_and_compare(w, K, V, q, [2048], seeds, 2048)
    assert rep["heads"] == 1


@pytest.mark.parametrize("n", [1500, 4093])
def test_decode_llama_shape_ragged(n):
    # GQA 4, d=128, bf16, half the groups near-uniform; ragged lengths span
    # several 256-key tiles and a partial block
    w, K, V, q = _case("llama16k", n, Hq=16, Hkv=4)
    seeds = synth.step_seeds(w, 3)
    run, rep = _run_and_compare(w, K, V, q, [n], seeds, n + 29)
    assert rep["heads"] == 16


def test_decode_batch_mixed_lengths():
    # independent sequences with different lengths, one without a pool
    w, K, V, q = _case("llama16k", 1200, B=3, Hq=8, Hkv=2)
    lens = [1200, 777, 50]
    seeds = synth.step_seeds(w, 4)
    run, rep = _run_and_compare(w, K, V, q, lens, seeds, 1200)
    o_g, beta_g, lvl_g, kr_g, _ = run.outputs()
    for hq in range(8):
        g = hq // 4
        o_ref, _ = dense_attention(q[2, hq], K[2, g, :50], V[2, g, :50])
        assert np.linalg.norm(o_g[2, hq] - o_ref) <= 1e-5 * np.linalg.norm(
            o_ref) + 1e-6
        assert beta_g[2, hq] == 0 and lvl_g[2, hq] == 0 and kr_g[2, hq] == 50


@pytest.mark.parametrize("G,d", [(1, 128), (2, 64), (8, 128)])
def test_decode_group_sizes(G, d):
    w, K, V, q = _case("llama16k", 900, Hq=2 * G, Hkv=2, d=d)
    seeds = synth.step_seeds(w, 5)
    _run_and_compare(w, K, V, q, [900], seeds, 900)


@pytest.mark.parametrize("measure", [1, 2])
def test_decode_other_measures(measure):
    w, K, V, q = _case("llama16k", 1100, Hq=8, Hkv=2)
    seeds = synth.step_seeds(w, 6)
    _run_and_compare(w, K, V, q, [1100], seeds, 1100, measure=measure)


def test_decode_fallback_to_exact():
    # an unreachable target: no level certifies, every head falls back to
    # exact attention (level J+1, beta 0, keys_read n)
    w, K, V, q = _case("llama16k", 800, Hq=8, Hkv=2)
    seeds = synth.step_seeds(w, 7)
    run, rep = _run_and_compare(w, K, V, q, [800], seeds, 800, eps=1e-7)
    o_g, beta_g, lvl_g, kr_g, _ = run.outputs()
    J = int(np.ceil(2 * np.log2(800 - 64)))
    assert np.all(lvl_g == J + 1) and np.all(beta_g == 0)
    assert np.all(kr_g == 800)


def test_decode_extended_grid():
    # J beyond the default: the last levels hold every pool key as heavy
    w, K, V, q = _case("tiny", 700)
    seeds = synth.step_seeds(w, 8)
    _run_and_compare(w, K, V, q, [700], seeds, 700, J_override=60)


def test_dense_decode_matches_exact():
    import torch
    import certified_sparse_attention_gb300 as csa
    w, K, V, q = _case("llama16k", 3000, B=2, Hq=8, Hkv=2)
    shape = csa.make_shape(2, 8, 2, 128, 3000, "bf16")
    dd = csa.DenseDecode(shape, "cuda")
    o = dd(to_dev(q, "bf16", "cuda"), to_dev(K, "bf16", "cuda"),
           to_dev(V, "bf16", "cuda"), [3000, 1777]).cpu().numpy()
    for b, n in ((0, 3000), (1, 1777)):
        for hq in range(8):
            ref, _ = dense_attention(q[b, hq], K[b, hq // 4, :n],
                                     V[b, hq // 4, :n])
            assert np.linalg.norm(o[b, hq] - ref) <= 1e-5 * np.linalg.norm(
                ref) + 1e-6


def test_decode_llama16k_full_size():
    # the 16K single-layer workload at its full size: every head compared
    w, K, V, q = _case("llama16k", 16384)
    seeds = synth.step_seeds(w, 0)
    run, rep = _run_and_compare(w, K, V, q, [16384], seeds, 16384)
    assert rep["heads"] == 32
    print("near-threshold flips", rep["flips"], "level flips",
          rep["level_flips"], "levels", rep["levels"])
