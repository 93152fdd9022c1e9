"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Bit-exact: the 4-bit codes, block bounds and value-norm bounds; every key's
upper bound ubar; c*_lo, c*_hi and cb; the candidate sets.  Set membership:
bit-exact except keys within 1e-5 nats of a threshold in perturbed
log-score (counted).  Outputs o and certificates beta: within 2e-3 relative
of the oracle evaluated with the device's memberships (which differ from the
oracle's only at the near-threshold keys).  Stop levels agree except where
the oracle's certificate sits within 0.2 % of its target.
"""
import numpy as np
import pytest

import synth
from oracle.quantize import quantize_keys, value_sq_norms_f32, vmax_blocks
from oracle.step import dense_attention
from tests.gpu_common import DeviceRun, ensure_built, o_close, run_and_compare, to_dev

pytestmark = pytest.mark.gpu


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

@pytest.mark.parametrize("step", [0, 1, 2])
def test_decode_tiny_config(step):
    # one head, d=64, n=2048, fp32, planted keys, eps .05 delta .01 r 2
    w, K, V, q = _case("tiny", 2048, step=step)
    seeds = synth.step_seeds(w, step)
    run, rep = run_and_compare(w, K, V, q, [2048], seeds, 2048)
    assert rep["heads"] == 1


@pytest.mark.parametrize("n", [1500, 4093])
def test_decode_llama_shape_ragged(n):
    # GQA 4, d=128, bf16, half the groups near-uniform; ragged lengths span
    # several 256-key tiles and a partial block
    w, K, V, q = _case("llama16k", n, Hq=16, Hkv=4)
    seeds = synth.step_seeds(w, 3)
    run, rep = run_and_compare(w, K, V, q, [n], seeds, n + 29)
    assert rep["heads"] == 16


def test_decode_batch_mixed_lengths():
    # independent sequences with different lengths, one without a pool
    w, K, V, q = _case("llama16k", 1200, B=3, Hq=8, Hkv=2)
    lens = [1200, 777, 50]
    seeds = synth.step_seeds(w, 4)
    run, rep = run_and_compare(w, K, V, q, lens, seeds, 1200)
    o_g, beta_g, lvl_g, kr_g, _ = run.outputs()
    for hq in range(8):
        g = hq // 4
        o_ref, _ = dense_attention(q[2, hq], K[2, g, :50], V[2, g, :50])
        assert np.linalg.norm(o_g[2, hq] - o_ref) <= 1e-5 * np.linalg.norm(
            o_ref) + 1e-6
        assert beta_g[2, hq] == 0 and lvl_g[2, hq] == 0 and kr_g[2, hq] == 50


@pytest.mark.parametrize("sub,runs", [(1, 1), (3, 2), (4, 4)])
def test_decode_sub_batches(sub, runs):
    # the batch unsplit, asked for 3 sub-batches (two of two sequences) and
    # as 4 sub-batches on the library's streams: every group against the
    # oracle
    w, K, V, q = _case("llama16k", 1500, B=4, Hq=8, Hkv=2)
    lens = [1500, 1333, 901, 1500]
    seeds = synth.step_seeds(w, 8)
    run, rep = run_and_compare(w, K, V, q, lens, seeds, 1500, sub_batches=sub)
    assert run.map.sub_batches == runs
    assert rep["heads"] == 32


@pytest.mark.parametrize("G,n", [(4, 1100), (8, 900), (2, 1500)])
def test_decode_per_head_perturbations(G, n):
    # one perturbation draw per query head: candidates, memberships, o and
    # beta against the oracle with the same per-head draws, across
    # sub-batches
    w, K, V, q = _case("llama16k", n, B=2, Hq=2 * G, Hkv=2)
    seeds = synth.step_seeds(w, 9)
    run, rep = run_and_compare(w, K, V, q, [n, n - 77], seeds, n, perturb=1)
    assert rep["heads"] == 4 * G


@pytest.mark.parametrize("G,d,n", [(4, 128, 1500), (2, 64, 1100),
                                   (8, 128, 4093)])
def test_decode_two_digit_query_codes(G, d, n):
    # query codes of two s8 digits with the closed-form residual: the
    # bounds, maxima and candidate sets bit for bit against the oracle's
    # two-digit construction, results as always
    w, K, V, q = _case("llama16k", n, B=2, Hq=2 * G, Hkv=2, d=d)
    seeds = synth.step_seeds(w, 10)
    run, rep = run_and_compare(w, K, V, q, [n, n - 61], seeds, n, qcode=1)
    assert rep["heads"] == 4 * G


@pytest.mark.parametrize("G,d", [(1, 128), (2, 64), (8, 128)])
def test_decode_group_sizes(G, d):
    w, K, V, q = _case("llama16k", 900, Hq=2 * G, Hkv=2, d=d)
    seeds = synth.step_seeds(w, 5)
    run_and_compare(w, K, V, q, [900], seeds, 900)


@pytest.mark.parametrize("measure", [1, 2, 3])
def test_decode_other_measures(measure):
    w, K, V, q = _case("llama16k", 1100, Hq=8, Hkv=2)
    seeds = synth.step_seeds(w, 6)
    run_and_compare(w, K, V, q, [1100], seeds, 1100, measure=measure)


def test_decode_fallback_to_exact():
    # an unreachable target: no level certifies, every head falls back to
    # exact attention (level J+1, beta 0, keys_read n)
    w, K, V, q = _case("llama16k", 800, Hq=8, Hkv=2)
    seeds = synth.step_seeds(w, 7)
    run, rep = run_and_compare(w, K, V, q, [800], seeds, 800, eps=1e-7)
    o_g, beta_g, lvl_g, kr_g, _ = run.outputs()
    J = int(np.ceil(2 * np.log2(800 - 64)))
    assert np.all(lvl_g == J + 1) and np.all(beta_g == 0)
    assert np.all(kr_g == 800)


def test_decode_extended_grid():
    # J beyond the default: the last levels hold every pool key as heavy
    w, K, V, q = _case("tiny", 700)
    seeds = synth.step_seeds(w, 8)
    run_and_compare(w, K, V, q, [700], seeds, 700, J_override=60)


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
    run, rep = run_and_compare(w, K, V, q, [16384], seeds, 16384)
    assert rep["heads"] == 32
    print("near-threshold flips", rep["flips"], "level flips",
          rep["level_flips"], "levels", rep["levels"])


def test_decode_step_in_cuda_graph():
    # the step (two sub-batches of one sequence: fork and join by events) captured into a
    # CUDA graph and replayed gives what the eager call gives
    import torch
    import certified_sparse_attention_gb300 as csa
    w, K, V, q = _case("llama16k", 2000, B=2, Hq=8, Hkv=2)
    dev = torch.device("cuda:0")
    shape = csa.make_shape(w.B, w.Hq, w.Hkv, w.d, w.n, w.dtype)
    Kt = torch.from_numpy(K).to(dev).to(torch.bfloat16)
    Vt = torch.from_numpy(V).to(dev).to(torch.bfloat16)
    qt = torch.from_numpy(q).to(dev).to(torch.bfloat16)
    mt = csa.meta_buffers(shape, dev)
    csa.check(csa.csa_quantize_keys(shape, Kt, Vt, [w.n] * w.B, 0, *mt))
    seeds = [int(x) for x in synth.step_seeds(w, 11)]
    step = csa.DecodeStep(shape, csa.make_params(w.eps, w.delta, w.r), dev)
    side = torch.cuda.Stream(dev)
    with torch.cuda.stream(side):
        step(qt, Kt, Vt, mt, [w.n] * w.B, seeds)        # eager (warms up)
    torch.cuda.synchronize()
    o_ref = step.o.clone()
    lv_ref = step.level.clone()
    step.o.zero_()
    step.level.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        step(qt, Kt, Vt, mt, [w.n] * w.B, seeds)
    graph.replay()
    torch.cuda.synchronize()
    csa.check(csa.csa_check(step.ws), "csa_check")
    assert torch.equal(step.level, lv_ref)
    err = torch.linalg.norm(step.o - o_ref, dim=-1)
    assert torch.all(err <= 1e-4 * torch.linalg.norm(o_ref, dim=-1) + 1e-6)


def test_decode_largest_batch_ragged():
    # the largest batch the boundary takes (128 sequences), ragged lengths
    # from 1 to 400 tokens (many without a pool): every group against the
    # oracle, as two sub-batches of 64
    w, K, V, q = _case("llama16k", 400, B=128, Hq=4, Hkv=2)
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 401, size=w.B)]
    lens[0], lens[1] = 1, 400
    seeds = synth.step_seeds(w, 12)
    run, rep = run_and_compare(w, K, V, q, lens, seeds, 400)
    assert run.map.sub_batches == 2
    assert rep["heads"] == w.Hq * sum(1 for n in lens if n > 64)
    # sequences without a pool: exact attention, beta 0, level 0
    o_g, beta_g, lvl_g, kr_g, _ = run.outputs()
    for b, n in enumerate(lens):
        if n > 64:
            continue
        for hq in range(w.Hq):
            g = hq // w.G
            o_ref, _ = dense_attention(q[b, hq], K[b, g, :n], V[b, g, :n])
            assert np.linalg.norm(o_g[b, hq] - o_ref) <= 1e-5 * np.linalg.norm(o_ref) + 1e-6
            assert beta_g[b, hq] == 0 and lvl_g[b, hq] == 0 and kr_g[b, hq] == n


def test_decode_degenerate_inputs():
    # a zero query (every score 0: all keys weigh the same and are heavy at
    # level 0; the query code is all zeros) and a group whose cached keys
    # are all equal (every block constant: Delta = 1, codes 0): against the
    # oracle
    w, K, V, q = _case("llama16k", 1500, Hq=8, Hkv=2)
    seeds = synth.step_seeds(w, 13)
    q0 = q.copy()
    q0[0, :4] = 0.0
    run, rep = run_and_compare(w, K, V, q0, [1500], seeds, 1500)
    assert rep["heads"] == 8
    K1 = K.copy()
    K1[0, 1, :] = K[0, 1, :1]
    run, rep = run_and_compare(w, K1, V, q, [1500], seeds, 1500)
    assert rep["heads"] == 8


def test_decode_metamorphic_relations():
    # on the device: doubling every value doubles o and beta at the same
    # stop levels (every scaling is by a power of two, exact in float32; the
    # per-level sums are float atomics whose order varies from run to run,
    # so the two runs agree to float32 rounding, not bit for bit), and a
    # larger eps never stops a head later
    import torch
    w, K, V, q = _case("llama16k", 1500, B=2, Hq=8, Hkv=2)
    seeds = synth.step_seeds(w, 14)
    run = DeviceRun(w, K, V, q, [1500, 1400], seeds, 1500)
    o1, b1, l1, k1, _ = run.outputs()
    run2 = DeviceRun(w, K, 2.0 * V, q, [1500, 1400], seeds, 1500)
    o2, b2, l2, k2, _ = run2.outputs()
    assert np.array_equal(l1, l2) and np.array_equal(k1, k2)
    for b in range(2):
        for hq in range(8):
            assert o_close(o2[b, hq], 2.0 * o1[b, hq], tol=1e-5)[0], (b, hq)
    assert np.allclose(b2, 2.0 * b1, rtol=1e-5, atol=0)
    prev = None
    for eps in (0.02, 0.05, 0.2):
        r = DeviceRun(w, K, V, q, [1500, 1400], seeds, 1500, eps=eps)
        lv = r.outputs()[2]
        if prev is not None:
            assert np.all(lv <= prev)
        prev = lv
    torch.cuda.synchronize()


# ------------------------------------- the benchmarked grid (r = 4) and eps

@pytest.mark.parametrize("r,n", [(3, 4093), (4, 4093)])
def test_decode_finer_grids_small(r, n):
    # grids of r = 3 and 4 levels per octave: the level arithmetic -r x,
    # J = ceil(r log2 |P|) and the round-1 margin r - 1, on a peaked and a
    # near-uniform group, through two sub-batches
    w, K, V, q = _case("llama16k", n, B=2, Hq=8, Hkv=2, r=r)
    seeds = synth.step_seeds(w, 13)
    run, rep = run_and_compare(w, K, V, q, [n, n - 333], seeds, n)
    assert rep["heads"] == 16


def test_decode_128k_r4_groups():
    # the shape of the 128K benchmark (n = 131072, GQA 4, d = 128, bf16,
    # eps .05, delta .05, r = 4, J = 68): one peaked and one near-uniform
    # group, every key's bound and candidate, every head's o and beta
    w, K, V, q = _case("llama128k_b4", 131072, B=1, Hq=8, Hkv=2)
    assert w.r == 4
    seeds = synth.step_seeds(w, 1)
    run, rep = run_and_compare(w, K, V, q, [131072], seeds, 131072)
    assert rep["heads"] == 8
    print("128K r=4: levels", rep["levels"], "flips", rep["flips"],
          "level flips", rep["level_flips"], "worst o", rep["worst_o"])


@pytest.mark.parametrize("eps", [0.01, 0.1])
def test_decode_16k_eps_sweep(eps):
    # tighter and looser targets than the default on the full 16K length:
    # eps = 0.01 pushes the stop levels deep (most of the pool sampled)
    w, K, V, q = _case("llama16k", 16384, Hq=8, Hkv=2, eps=eps)
    seeds = synth.step_seeds(w, 2)
    run, rep = run_and_compare(w, K, V, q, [16384], seeds, 16384)
    assert rep["heads"] == 8
    print("eps", eps, "levels", rep["levels"], "worst o", rep["worst_o"])


# ------------------------------------------------- 8-bit refinement tier

@pytest.mark.parametrize("n,over", [(1337, {"Hq": 8, "Hkv": 2}),
                                    (130, {"Hq": 4, "Hkv": 4, "d": 64})])
def test_quantizer8_bit_exact(n, over):
    import torch
    import certified_sparse_attention_gb300 as csa
    from oracle.quantize import quantize_keys8
    w, K, V, q = _case("llama16k", n, **over)
    n_alloc = n + 75
    shape = csa.make_shape(w.B, w.Hq, w.Hkv, w.d, n_alloc, w.dtype)
    Kp = np.zeros((w.B, w.Hkv, n_alloc, w.d), np.float32)
    Kp[:, :, :n] = K
    Kt = to_dev(Kp, w.dtype, "cuda")
    K8, d8 = csa.meta8_buffers(shape, "cuda")
    csa.check(csa.csa_quantize_keys8(shape, Kt, [n] * w.B, 0, K8, d8))
    torch.cuda.synchronize()
    for g in range(w.Hkv):
        codes8, mins8, deltas8 = quantize_keys8(K[0, g], n)
        nb = mins8.shape[0]
        assert np.array_equal(K8[0, g, :nb * 64].cpu().numpy(), codes8)
        assert np.array_equal(d8[0, g, :nb].cpu().numpy(), deltas8)


@pytest.mark.parametrize("refine8,r,n", [(1, 2, 4093), (1, 4, 4093),
                                         (2, 4, 4093), (1, 2, 16384)])
def test_decode_refine8(refine8, r, n):
    # the 8-bit tier: every refined key's level bit for bit (through the
    # candidates scored, keys_read, the group unions and the 8-bit rows),
    # and the same memberships, o, beta and levels as without it
    w, K, V, q = _case("llama16k", n, B=2, Hq=8, Hkv=2, r=r)
    seeds = synth.step_seeds(w, 15)
    run, rep = run_and_compare(w, K, V, q, [n, n - 211], seeds, n,
                               refine8=refine8)
    assert rep["heads"] == 16


@pytest.mark.parametrize("G,n", [(4, 1500), (8, 4093)])
def test_decode_scan_dots_on_cuda_cores(G, n):
    # the scan's integer dot products by dp4a instead of tensor cores: the
    # same bounds bit for bit, hence the same everything
    w, K, V, q = _case("llama16k", n, B=2, Hq=2 * G, Hkv=2)
    seeds = synth.step_seeds(w, 16)
    run, rep = run_and_compare(w, K, V, q, [n, n - 99], seeds, n, dots=1)
    assert rep["heads"] == 4 * G
