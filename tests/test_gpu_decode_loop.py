"""Whole-token decode through csa_decode_step_device, one CUDA graph per token.

readsearch.ai "Abstract": the perturbations are drawn anew at every decode
step; picx.dev "CPU Speed": whole decode steps (all layers) are what the
pages time.  Here every token of a two-layer model appends one row per
layer (the K, V rows are already in the cache; the length grows over them),
and one captured graph runs both layers' steps with the lengths and seeds
read from device memory and the appended block re-quantised inside each
step's first kernel.  After every replay: the re-quantised metadata bit for
bit against the oracle's quantiser on the grown cache, and every head's
stop level, o, beta and keys_read against the oracle's decode step with the
same seeds.
"""
import numpy as np
import pytest

import synth
from oracle.quantize import quantize_keys, value_sq_norms_f32, vmax_blocks
from oracle.step import Params, oracle_decode_group
from tests.gpu_common import TOL, ensure_built, o_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _check_head(res, h, o, beta, lvl, kr, near, eps, where):
    """One head against the oracle: the same stop level unless the oracle's
    certificate sits within float rounding of its target there; o (element-
    wise), beta within 2e-3 and keys_read exactly at a common level (o is
    compared only when no key lies within 1e-5 nats of a threshold)."""
    cert = res.detail[h]["cert"]
    if lvl != res.level[h]:
        jm = int(min(lvl, res.level[h]))
        assert jm <= res.J, where
        tgt = eps * cert["scale_lo"][jm]
        assert abs(cert["beta"][jm] - tgt) <= 2e-3 * tgt, where
        return
    if near == 0:
        ok, worst = o_close(o, res.o[h])
        assert ok, (where, worst)
    if lvl <= res.J:
        assert abs(beta - res.beta[h]) <= TOL * res.beta[h], where
    assert kr == res.keys_read[h], where


def test_graph_per_token_against_oracle():
    import torch
    import certified_sparse_attention_gb300 as csa
    dev = torch.device("cuda:0")
    w = synth.workload("llama16k", B=2, Hq=8, Hkv=2, n=1600)
    L, T = 2, 3
    n0 = np.array([1500, 1333])          # lengths before the first append
    shape = csa.make_shape(w.B, w.Hq, w.Hkv, w.d, w.n, w.dtype)
    params = csa.make_params(w.eps, w.delta, w.r)
    p = Params(w.eps, w.delta, w.r)
    layers = []
    for lid in range(L):
        K, V, meta = synth.kv_numpy(w, layer=lid)
        qs = [synth.q_numpy(w, meta, t, layer=lid) for t in range(T)]
        seeds = [synth.step_seeds(w, t, layer=lid) for t in range(T)]
        Kt, Vt = to_dev(K, w.dtype, dev), to_dev(V, w.dtype, dev)
        mt = csa.meta_buffers(shape, dev)
        csa.check(csa.csa_quantize_keys(shape, Kt, Vt, [int(x) for x in n0],
                                        0, *mt))
        step = csa.DecodeStep(shape, params, dev, with_stats=True)
        q_dev = torch.empty((w.B, w.Hq, w.d), dtype=torch.bfloat16,
                            device=dev)
        seed_dev = torch.empty(w.B, dtype=torch.int64, device=dev)
        layers.append(dict(K=K, V=V, qs=qs, seeds=seeds, Kt=Kt, Vt=Vt, mt=mt,
                           step=step, q_dev=q_dev, seed_dev=seed_dev))
    lens_dev = torch.empty(w.B, dtype=torch.int64, device=dev)

    def load_token(t):
        lens_dev.copy_(torch.from_numpy(n0 + t + 1))
        for ly in layers:
            ly["q_dev"].copy_(to_dev(ly["qs"][t], w.dtype, dev))
            s = ly["seeds"][t].astype(np.uint64).view(np.int64)
            ly["seed_dev"].copy_(torch.from_numpy(s.copy()))

    def token():
        for ly in layers:
            ly["step"].device_step(ly["q_dev"], ly["Kt"], ly["Vt"], ly["mt"],
                                   lens_dev, ly["seed_dev"], True)

    side = torch.cuda.Stream(dev)
    load_token(0)
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        token()                           # eager warm-up of token 0
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        token()
    heads = 0
    for t in range(T):
        load_token(t)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        lens = n0 + t + 1
        for li, ly in enumerate(layers):
            csa.check(csa.csa_check(ly["step"].ws), "csa_check")
            # the appended token's block, re-quantised in the step
            K4, bounds, vmax, vnorm2 = [x.cpu().numpy() for x in ly["mt"]]
            for b in range(w.B):
                n = int(lens[b])
                for g in range(w.Hkv):
                    codes, packed, mins, deltas = quantize_keys(ly["K"][b, g], n)
                    nb = mins.shape[0]
                    assert np.array_equal(K4[b, g, :nb * 64], packed), (t, li, b, g)
                    assert np.array_equal(bounds[b, g, :nb, 0], mins)
                    assert np.array_equal(bounds[b, g, :nb, 1], deltas)
                    assert np.array_equal(vmax[b, g, :nb],
                                          vmax_blocks(ly["V"][b, g], n))
                    assert np.array_equal(vnorm2[b, g, :n],
                                          value_sq_norms_f32(ly["V"][b, g], n))
            st = ly["step"]
            o = st.o.cpu().numpy().astype(np.float64)
            beta = st.beta.cpu().numpy()
            lvl = st.level.cpu().numpy()
            kr = st.keys_read.cpu().numpy()
            stats = st.stats.cpu().numpy()
            for b in range(w.B):
                n = int(lens[b])
                seed = int(ly["seeds"][t][b])
                for g in range(w.Hkv):
                    G = w.G
                    res = oracle_decode_group(ly["qs"][t][b, g * G:(g + 1) * G],
                                              ly["K"][b, g], ly["V"][b, g], n,
                                              seed, g, p)
                    for h in range(G):
                        hq = g * G + h
                        _check_head(res, h, o[b, hq], beta[b, hq],
                                    int(lvl[b, hq]), int(kr[b, hq]),
                                    int(stats[b, hq, 4]), w.eps,
                                    (t, li, b, hq))
                        heads += 1
    assert heads == T * L * w.B * w.Hq
