"""Shared helpers of the GPU parity tests (run the CUDA path through the C
ABI, run the oracle on the same inputs, compare)."""
from __future__ import annotations

import math
import os

import numpy as np

import synth
from oracle.certificate import certificate_levels
from oracle.hashing import head_stream, perturb_t
from oracle.step import Params, dense_attention, level_sums, oracle_decode_group

F = np.float32
TOL = 2e-3      # o and beta, relative
NEAR = 1e-5     # nats: memberships this close to a threshold may differ


def o_close(o_dev, o_ref, tol=TOL):
    """Element-wise "within tol relative" for an output vector: every channel
    c satisfies |o_dev_c - o_ref_c| <= tol (|o_ref_c| + rms(o_ref)).  The rms
    floor keeps channels whose exact value is near zero (where any rounding
    is large relative to the channel) from failing on float32 rounding,
    while no single channel can hide an error behind the vector's norm."""
    o_dev = np.asarray(o_dev, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    rms = float(np.sqrt(np.mean(o_ref * o_ref)))
    err = np.abs(o_dev - o_ref)
    lim = tol * (np.abs(o_ref) + rms)
    return bool(np.all(err <= lim)), float(np.max(err / np.maximum(lim, 1e-300)))


def ensure_built():
    import certified_sparse_attention_gb300 as csa
    if not os.path.exists(csa.LIB_PATH):
        from certified_sparse_attention_gb300 import build
        build.build()
    return csa.load_library()


def to_dev(x, dtype, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x)).to(device)
    return t.to(torch.bfloat16 if dtype == "bf16" else torch.float32)


class DeviceRun:
    """One decode step of a workload on the GPU, with workspace views."""

    def __init__(self, w: synth.Workload, K, V, q, lens, seeds, n_alloc,
                 device="cuda:0", eps=None, delta=None, r=None,
                 measure=0, J_override=-1, sub_batches=0, perturb=0,
                 qcode=0, refine8=0, dots=0):
        import torch
        import certified_sparse_attention_gb300 as csa
        self.csa = csa
        self.w = w
        self.lens = [int(x) for x in lens]
        self.seeds = [int(x) for x in seeds]
        self.shape = csa.make_shape(w.B, w.Hq, w.Hkv, w.d, n_alloc, w.dtype)
        self.params = csa.make_params(w.eps if eps is None else eps,
                                      w.delta if delta is None else delta,
                                      w.r if r is None else r, measure,
                                      J_override, sub_batches, perturb,
                                      qcode, refine8, dots)
        Kp = np.zeros((w.B, w.Hkv, n_alloc, w.d), np.float32)
        Vp = np.zeros_like(Kp)
        Kp[:, :, :K.shape[2]] = K
        Vp[:, :, :V.shape[2]] = V
        self.K = to_dev(Kp, w.dtype, device)
        self.V = to_dev(Vp, w.dtype, device)
        self.q = to_dev(q, w.dtype, device)
        self.meta = csa.meta_buffers(self.shape, device)
        csa.check(csa.csa_quantize_keys(self.shape, self.K, self.V, self.lens,
                                        0, *self.meta),
                  "csa_quantize_keys")
        self.meta8 = None
        if refine8:
            self.meta8 = csa.meta8_buffers(self.shape, device)
            csa.check(csa.csa_quantize_keys8(self.shape, self.K, self.lens, 0,
                                             *self.meta8),
                      "csa_quantize_keys8")
        self.step = csa.DecodeStep(self.shape, self.params, device,
                                   with_stats=True)
        self.step(self.q, self.K, self.V, self.meta, self.lens, self.seeds,
                  meta8=self.meta8)
        torch.cuda.synchronize()
        csa.check(csa.csa_check(self.step.ws), "csa_check")
        self.map = csa.csa_workspace_layout(self.shape, self.params)

    def rerun(self, q, lens, seeds):
        """The same caches, a new step: fresh queries, lengths and seeds."""
        import torch
        self.lens = [int(x) for x in lens]
        self.seeds = [int(x) for x in seeds]
        self.q = to_dev(q, self.w.dtype, self.q.device)
        self.step(self.q, self.K, self.V, self.meta, self.lens, self.seeds,
                  meta8=self.meta8)
        torch.cuda.synchronize()
        self.csa.check(self.csa.csa_check(self.step.ws), "csa_check")

    def append(self, b, pos, k_row, v_row):
        """Write token `pos` of sequence b (all KV heads; [Hkv, d] rows) and
        re-quantise its block, as a decode step does after appending."""
        import torch
        dt = self.K.dtype
        self.K[b, :, pos] = torch.from_numpy(np.ascontiguousarray(k_row)).to(self.K.device).to(dt)
        self.V[b, :, pos] = torch.from_numpy(np.ascontiguousarray(v_row)).to(self.V.device).to(dt)
        lens = list(self.lens)
        lens[b] = max(lens[b], pos + 1)
        self.csa.check(self.csa.csa_quantize_keys(self.shape, self.K, self.V,
                                                  lens, pos, *self.meta),
                       "csa_quantize_keys")
        self.lens = lens

    def ws_view(self, off, per_seq, dtype):
        """A per-sequence array of the workspace ([B][per_seq] 4-byte
        words), gathered over the step's sub-batch regions."""
        import torch
        m = self.map
        parts = []
        for c in range(m.sub_batches):
            nb = min(m.sub_B, self.w.B - c * m.sub_B)
            if nb <= 0:
                break
            o = c * m.sub_stride + off
            t = self.step.ws[o:o + nb * per_seq * 4]
            parts.append(t.view(dtype).cpu().numpy())
        return np.concatenate(parts)

    def ubar(self):
        import torch
        w = self.w
        n = self.shape.n_max
        a = self.ws_view(self.map.ubar, w.Hkv * n * w.G, torch.float32)
        return a.reshape(w.B, w.Hkv, n, w.G)

    def cmax(self):
        import torch
        w = self.w
        a = self.ws_view(self.map.cmax, w.Hq * 4, torch.int32)
        return self.csa.decode_ordered(a.view(np.uint32)).reshape(w.B, w.Hq, 4)

    def s32(self):
        import torch
        w = self.w
        pcap = max(self.shape.n_max - 64, 1)
        a = self.ws_view(self.map.s32, w.Hkv * pcap * w.G, torch.float32)
        return a.reshape(w.B, w.Hkv, pcap, w.G)

    def outputs(self):
        st = self.step
        return (st.o.cpu().numpy().astype(np.float64), st.beta.cpu().numpy(),
                st.level.cpu().numpy(), st.keys_read.cpu().numpy(),
                st.stats.cpu().numpy())


def gpu_levels(s32, c32, t, r, J):
    """The device's float32 level arithmetic, replayed on the host from the
    device's own scores (to compare memberships key by key)."""
    s32 = np.asarray(s32, F)
    y = (s32 - F(c32)) * F(1.0 / math.log(2.0))
    x = y + np.asarray(t, F)

    def lvl(v):
        out = np.where(v <= F(J), np.maximum(np.ceil(v), 0), J + 1)
        return np.where(np.isnan(v), J + 1, out).astype(np.int64)
    return lvl(F(-r) * x), lvl(F(-r) * y)


# ------------------------------------------- comparison with the oracle

def compare_group(run, w, K, V, q, b, g, res, p, report):
    ub = run.ubar()
    cm = run.cmax()
    s32 = run.s32()
    o_g, beta_g, lvl_g, kr_g, stats = run.outputs()
    n = run.lens[b]
    P = n - 64
    J = res.J
    Vd = V[b, g, :n].astype(np.float64)
    needK, needV = set(), set()
    for h in range(w.G):
        hq = g * w.G + h
        det = res.detail[h]
        # bit-exact bounds, maxima and candidates
        assert np.array_equal(ub[b, g, :n, h], det["ubar"]), (b, g, h)
        assert cm[b, hq, 0] == det["c_lo"] and cm[b, hq, 1] == det["c_hi"]
        assert cm[b, hq, 2] == det["cb"]
        # candidates are rescored by bound-level range, round by round:
        # every candidate with jbar up to the stop level has its score, no
        # key outside the candidates has one, and a candidate left unscored
        # has its exact level beyond the stop (jl >= jbar)
        cand = det["cand"]
        lv = min(int(lvl_g[b, hq]), J)
        scored = np.isfinite(s32[b, g, :P, h])
        assert not np.any(scored & ~cand), (b, g, h)
        # (with the 8-bit tier a candidate is read from its refined level)
        jneed = det["jref"] if p.refine8 else det["jbar"]
        assert np.all(scored[cand & (jneed <= lv)]), (b, g, h)
        pend = cand & ~scored
        assert np.all(det["jl_c"][pend] > lv), (b, g, h)
        assert stats[b, hq, 3] == res.n_candidates[h]
        # memberships: device float32 vs oracle float64
        c32 = cm[b, hq, 3]
        # the head's perturbation, recomputed from the published hash (the
        # oracle's own draw for this head: shared or per head)
        t = perturb_t(run.seeds[b],
                      head_stream(g, w.G, h) if p.per_head else g, np.arange(P))
        assert np.array_equal(t, det["t"])
        jg, hg = gpu_levels(s32[b, g, :P, h], c32, t, p.r, J)
        # levels beyond the grid are all "never" (J + 1); so are the levels
        # of candidates not rescored (they lie beyond the stop level)
        jo = np.where(pend, J + 1, np.minimum(det["jl_c"], J + 1))
        ho = np.where(pend, J + 1, np.minimum(det["hl_c"], J + 1))
        jg = np.where(scored, jg, J + 1)
        hg = np.where(scored, hg, J + 1)
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
                                  det["delta_e"], p.eps, p.measure,
                                  delta=p.delta)
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
                                     np.nonzero(jneed <= gl)[0]))
            assert kr_g[b, hq] == kr
            if p.refine8:
                assert stats[b, hq, 9] == res.rows8[h], (b, g, h)
            assert stats[b, hq, 2] == 64 + int((jr <= gl).sum())
        else:
            o_ref, _ = dense_attention(q[b, hq], K[b, g, :n], V[b, g, :n])
            assert beta_g[b, hq] == 0 and kr_g[b, hq] == n
        ok_o, worst = o_close(o_g[b, hq], o_ref)
        assert ok_o, (b, g, h, worst)
        report["worst_o"] = max(report.get("worst_o", 0.0), worst)
        report["heads"] += 1
        report["levels"].append(gl)
        # rows the head needs, for the group unions
        if gl <= J:
            needK.update(np.union1d(det["cset"],
                                    np.nonzero(jneed <= gl)[0]).tolist())
            needV.update(np.nonzero(jr <= gl)[0].tolist())
        else:
            needK.update(range(P))
            needV.update(range(P))
    for h in range(w.G):
        hq = g * w.G + h
        assert stats[b, hq, 7] == 64 + len(needK)
        assert stats[b, hq, 8] == 64 + len(needV)


def run_and_compare(w, K, V, q, lens, seeds, n_alloc, **pover):
    run = DeviceRun(w, K, V, q, lens, seeds, n_alloc, **pover)
    p = Params(run.params.eps, run.params.delta, run.params.r,
               measure=run.params.measure, J_override=run.params.J_override,
               per_head=bool(run.params.perturb),
               two_digit=bool(run.params.qcode),
               refine8=bool(run.params.refine8))
    report = {"flips": 0, "level_flips": 0, "heads": 0, "levels": []}
    for b in range(w.B):
        n = run.lens[b]
        if n <= 64:
            continue
        for g in range(w.Hkv):
            res = oracle_decode_group(q[b, g * w.G:(g + 1) * w.G], K[b, g],
                                      V[b, g], n, run.seeds[b], g, p)
            compare_group(run, w, K, V, q, b, g, res, p, report)
    return run, report
