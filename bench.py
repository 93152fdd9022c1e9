#!/usr/bin/env python
"""Benchmark of certified sparse decode attention on GB300.

One step = the certified sparse decode-attention step of one layer for the
whole batch: B = 4 sequences at n = 131072 tokens, 32 query heads / 8 KV
heads, d = 128, bf16 KV cache, eps = 0.05, delta = 0.05, r = 4 (the 128K
headline workload).  Timed steps rotate over several independently seeded
layers resident in HBM, so the working set is far larger than L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  N > 1 runs under torch.distributed (one process per
GPU); every rank decodes its own batch (weak scaling, no collective on the
data path), the time is the maximum over ranks.
"""
from __future__ import annotations

import os

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import threading  # noqa: E402
import time  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "certified sparse decode-attn µs/step & HBM GB/s (% roofline) at 128K ctx"
WORKLOAD = "llama128k_b4"


# --------------------------------------------------------------- host logic

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return world, rank, local


def rank_layers(rank: int, world: int, layers: int):
    """Layer ids (generator seeds) decoded by a rank: disjoint per rank."""
    return [rank * 1000 + i for i in range(layers)]


def step_plan(rank: int, steps: int, layers: int):
    """(layer slot, step index) of every timed step of a rank."""
    return [(s % layers, s) for s in range(steps)]


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e nominal bandwidth (the measured copy peak is the roofline)


def workload_name(w) -> str:
    return (f"{w.name}: B={w.B} sequences x 1 layer per step, n={w.n}, "
            f"Hq={w.Hq}, Hkv={w.Hkv}, d={w.d}, bf16, eps={w.eps}, "
            f"delta={w.delta}, r={w.r}")


def algorithmic_bytes(stats, w, n):
    """Bytes the method must move per step (per (sequence, KV head)):
    scan |P| (d/2 + 8d/64 + 4/64) over the pool + the window's 64 scan rows,
    2d bytes per bf16 K row and per V row actually needed (unions over the
    GQA group, window included), and the per-level scratch (J+1)(2d+6)*4
    per query head."""
    d, G = w.d, w.G
    P = n - 64
    scan = n * (d / 2 + 8 * d / 64 + 4 / 64)
    st = stats.reshape(w.B, w.Hkv, G, -1)
    kr = st[:, :, 0, 7].astype(float)
    vr = st[:, :, 0, 8].astype(float)
    J = st[:, :, :, 5].astype(float)
    rows = 2 * d * (kr + vr)
    scratch = ((J + 1) * (2 * d + 6) * 4).sum(axis=2)
    per = {
        "scan": w.B * w.Hkv * scan,
        "rows_k": float((2 * d * kr).sum()),
        "rows_v": float((2 * d * vr).sum()),
        "scratch": float(scratch.sum()),
    }
    per["total"] = per["scan"] + float(rows.sum()) + per["scratch"]
    return per


class Coverage:
    """Certificate coverage: ||o_hat - o|| against beta and eps * M, with o
    and M = sqrt(sum_i a_i ||v_i||^2) from float64 exact attention."""

    def __init__(self, w):
        self.w = w
        self.n = self.beta_viol = self.eps_viol = self.fallback = 0
        self.ratio = []
        self.ratio_o = []

    def add(self, q, K, V, lens, step):
        import torch
        w = self.w
        G, d = w.G, w.d
        o_hat = step.o.double()
        beta = step.beta.double()
        level = step.level.long()
        J = int(math.ceil(w.r * math.log2(w.n - 64)))
        for b in range(w.B):
            n = int(lens[b])
            for g in range(w.Hkv):
                Kd = K[b, g, :n].double()
                Vd = V[b, g, :n].double()
                qd = q[b, g * G:(g + 1) * G].double()
                a = torch.softmax(qd @ Kd.T / math.sqrt(d), dim=1)
                o = a @ Vd
                M = torch.sqrt(a @ (Vd * Vd).sum(dim=1))
                hs = slice(g * G, (g + 1) * G)
                err = torch.linalg.norm(o_hat[b, hs] - o, dim=1)
                fb = level[b, hs] > J
                self.n += G
                self.fallback += int(fb.sum())
                self.beta_viol += int(((err > beta[b, hs] + 1e-7) & ~fb).sum())
                self.eps_viol += int((err > w.eps * M).sum())
                self.ratio.extend((err / (w.eps * M)).tolist())
                self.ratio_o.extend((err / (w.eps * torch.linalg.norm(o, dim=1))).tolist())

    def summary(self):
        import numpy as np
        r = np.asarray(self.ratio)
        return {"head_steps": self.n, "beta_violations": self.beta_viol,
                "eps_violations": self.eps_viol,
                "eps_violations_output_norm": int(np.sum(np.asarray(self.ratio_o) > 1.0)),
                "fallbacks": self.fallback,
                "delta": self.w.delta,
                "err_over_epsM": {"p50": round(float(np.percentile(r, 50)), 4),
                                  "p90": round(float(np.percentile(r, 90)), 4),
                                  "max": round(float(r.max()), 4)},
                "err_over_eps_norm_o": {
                    "p50": round(float(np.percentile(self.ratio_o, 50)), 4),
                    "p90": round(float(np.percentile(self.ratio_o, 90)), 4),
                    "max": round(float(np.max(self.ratio_o)), 4)},
                "reference": "float64 exact attention on the device"}


def run_mode(args, csa, w, shape, data, lens, seed_tab, nseed, plan, stream,
             device, measure, perturb=0):
    """The same steps under another stop measure (or with per-query-head
    perturbation draws): keys and values read per head, time per step, and
    the error against exact attention."""
    import torch
    params = csa.make_params(w.eps, w.delta, w.r, measure, perturb=perturb)
    step = csa.DecodeStep(shape, params, device, with_stats=False)
    diag = csa.DecodeStep(shape, params, device, with_stats=True)
    cov = Coverage(w)
    kr, vr = [], []
    for L in range(args.layers):
        d = data[L]
        diag(d["q"][L % 4], d["K"], d["V"], d["meta"], lens,
             seed_tab[L][L % nseed], stream)
        torch.cuda.synchronize()
        csa.check(csa.csa_check(diag.ws, stream), "csa_check (measure %d)" % measure)
        st = diag.stats.cpu().numpy()
        kr.append(st[..., 1].mean())
        vr.append(st[..., 2].mean())
        cov.add(d["q"][L % 4], d["K"], d["V"], lens, diag)
    for (L, s) in plan[:3]:
        d = data[L]
        step(d["q"][s % 4], d["K"], d["V"], d["meta"], lens,
             seed_tab[L][s % nseed], stream, meta8=d.get("meta8"))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for (L, s) in plan:
        d = data[L]
        step(d["q"][s % 4], d["K"], d["V"], d["meta"], lens,
             seed_tab[L][s % nseed], stream, meta8=d.get("meta8"))
    e1.record(stream)
    torch.cuda.synchronize()
    csa.check(csa.csa_check(step.ws, stream), "csa_check (measure %d, timed)" % measure)
    cs = cov.summary()
    return {"us_per_step": round(e0.elapsed_time(e1) / len(plan) * 1e3, 2),
            "keys_read_mean": round(float(sum(kr) / len(kr)), 1),
            "values_read_mean": round(float(sum(vr) / len(vr)), 1),
            "head_steps": cs["head_steps"],
            "beta_violations": cs["beta_violations"],
            "eps_violations_value_scale": cs["eps_violations"],
            "eps_violations_output_norm": cs["eps_violations_output_norm"],
            "err_over_epsM": cs["err_over_epsM"],
            "err_over_eps_norm_o": cs["err_over_eps_norm_o"]}


def clt_comparison(args, csa, w, shape, data, lens, seed_tab, nseed, plan,
                   stream, device, reads_cert):
    """The same steps under the uncertified CLT stop rule (picx.dev
    "Theoretical Contributions" compares the certificate with it)."""
    r = run_mode(args, csa, w, shape, data, lens, seed_tab, nseed, plan,
                 stream, device, csa.CSA_MEASURE_CLT)
    kc = float(sum(x[0] for x in reads_cert)) / len(reads_cert)
    vc = float(sum(x[1] for x in reads_cert)) / len(reads_cert)
    return {"us_per_step": r["us_per_step"],
            "keys_read_mean": r["keys_read_mean"],
            "values_read_mean": r["values_read_mean"],
            "certified_over_clt_keys": round(kc / r["keys_read_mean"], 3),
            "certified_over_clt_values": round(vc / r["values_read_mean"], 3),
            "eps_violations": r["eps_violations_value_scale"],
            "head_steps": r["head_steps"],
            "err_over_epsM": r["err_over_epsM"]}


def decode_loop(args, csa, w, device, stream):
    """Whole-model decode: every token appends one row per layer and runs
    that layer's step, over `args.decode_layers` layers of the workload's
    shape (readsearch.ai "Abstract": new perturbation draws for each
    decode step).  The lengths, the token index and every layer's seeds
    live in device memory, so the whole token (all layers) is captured once
    into a CUDA graph and replayed: per layer the graph picks the token's
    query and seeds, and runs csa_decode_step_device, whose first kernel
    re-quantises the appended token's block.  The K, V rows of the appended
    tokens are generated with the cache; the loop extends the length over
    them.  Also timed: the same token launched stream-ordered through
    csa_decode_step (host lengths and seeds, csa_quantize_keys on the
    appended block first)."""
    import torch
    import synth
    L, T = args.decode_layers, 8
    n0 = w.n - T
    shape = csa.make_shape(w.B, w.Hq, w.Hkv, w.d, w.n, w.dtype)
    params = csa.make_params(w.eps, w.delta, w.r)
    step = csa.DecodeStep(shape, params, device)
    layers = []
    q_all, seed_all = [], []
    for lid in range(L):
        K, V, meta = synth.kv_torch(w, layer=100 + lid, device=device)
        mt = csa.meta_buffers(shape, device)
        csa.check(csa.csa_quantize_keys(shape, K, V, [n0] * w.B, 0, *mt),
                  "csa_quantize_keys")
        q_all.append(torch.stack([synth.q_torch(w, meta, t, layer=100 + lid,
                                                device=device)
                                  for t in range(T)]))
        seed_all.append(torch.tensor(
            [[s - (1 << 64) if s >= (1 << 63) else s
              for s in seeds_for(w, 100 + lid, t)] for t in range(T)],
            dtype=torch.int64, device=device))
        layers.append((K, V, mt, lid))
    q_all = torch.stack(q_all, 1)            # [T, L, B, Hq, d]
    seed_all = torch.stack(seed_all, 1)      # [T, L, B]
    torch.cuda.synchronize()
    t_dev = torch.zeros(1, dtype=torch.int64, device=device)
    lens_dev = torch.zeros(w.B, dtype=torch.int64, device=device)
    q_cur = torch.empty_like(q_all[0, 0])
    seed_cur = torch.empty(w.B, dtype=torch.int64, device=device)

    def token_device():
        lens_dev.copy_((t_dev + (n0 + 1)).expand(w.B))
        qt = q_all.index_select(0, t_dev)[0]         # [L, B, Hq, d]
        st = seed_all.index_select(0, t_dev)[0]      # [L, B]
        for li, (K, V, mt, lid) in enumerate(layers):
            q_cur.copy_(qt[li])
            seed_cur.copy_(st[li])
            step.device_step(q_cur, K, V, mt, lens_dev, seed_cur, True)
        t_dev.add_(1)

    def token_host(t):
        pos = n0 + t
        lens = [pos + 1] * w.B
        for li, (K, V, mt, lid) in enumerate(layers):
            csa.check(csa.csa_quantize_keys(shape, K, V, lens, pos, *mt,
                                            stream=stream),
                      "csa_quantize_keys")
            step(q_all[t, li], K, V, mt, lens,
                 seeds_for(w, 100 + lid, t), stream)

    gs = torch.cuda.Stream(device)           # graphs are captured off the default stream
    with torch.cuda.stream(gs):
        token_device()                       # warm-up, eager (token 0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        token_device()
    t_dev.fill_(1)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(gs):
        e0.record(gs)
        for t in range(1, T):
            graph.replay()
        e1.record(gs)
    torch.cuda.synchronize()
    csa.check(csa.csa_check(step.ws, gs), "csa_check (decode loop)")
    us_graph = e0.elapsed_time(e1) / (T - 1) * 1e3
    e0.record(stream)
    for t in range(1, T):
        token_host(t)
    e1.record(stream)
    torch.cuda.synchronize()
    csa.check(csa.csa_check(step.ws, stream), "csa_check (decode loop)")
    us_host = e0.elapsed_time(e1) / (T - 1) * 1e3
    del layers, graph
    torch.cuda.empty_cache()
    return {"layers": L, "tokens_timed": T - 1, "context": f"{n0 + 1}..{w.n}",
            "us_per_token": round(us_graph, 1),
            "us_per_layer": round(us_graph / L, 1),
            "stream_ordered_us_per_token": round(us_host, 1),
            "stream_ordered_us_per_layer": round(us_host / L, 1),
            "note": "one CUDA graph per token over all layers: device "
                    "lengths and seeds, the appended block re-quantised "
                    "inside each step's first kernel; stream_ordered: host "
                    "lengths, csa_quantize_keys then csa_decode_step per "
                    "layer"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


# ------------------------------------------------------------ CPU baseline

def _oracle_task(job):
    """One (sequence, KV head) group of the workload on one host core: draw
    it with the seeded generator (numpy back end, the same law as the
    device inputs), then time the float64 oracle's certified step and the
    float64 dense step for its G query heads."""
    name, layer, step, g = job
    import synth
    from oracle.step import Params, dense_attention, oracle_decode_group
    full = synth.workload(name)
    one = synth.workload(name, B=1, Hq=2 * full.G, Hkv=2)   # a peaked and a flat group
    K, V, meta = synth.kv_numpy(one, layer=layer)
    q = synth.q_numpy(one, meta, step, layer=layer)
    seed = int(synth.step_seeds(one, step, layer=layer)[0])
    G = full.G
    p = Params(full.eps, full.delta, full.r)
    t0 = time.perf_counter()
    oracle_decode_group(q[0, g * G:(g + 1) * G], K[0, g], V[0, g], one.n,
                        seed, g, p, keep_detail=False)
    t1 = time.perf_counter()
    for h in range(G):
        dense_attention(q[0, g * G + h], K[0, g], V[0, g])
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def oracle_step_times(pool, cores, w, step, name=None):
    """Host time of the oracle for one step (all B x Hkv groups), from a
    bounded sample: `cores` groups (half peaked, half near-uniform), one
    per process, in parallel.  Returns (sparse, dense) seconds per whole
    step with the groups spread over the cores (mean core seconds per
    group x groups / cores), and the sparse core seconds per whole step."""
    groups = w.B * w.Hkv
    ns = min(cores, groups)
    jobs = [(name or WORKLOAD, 1000 + 97 * step + i, step, i % 2) for i in range(ns)]
    res = pool.map(_oracle_task, jobs, chunksize=1)
    sp = sum(r[0] for r in res) / ns * groups
    de = sum(r[1] for r in res) / ns * groups
    return sp / cores, de / cores, sp, de


def cpu_pool():
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")       # never fork a process that holds a GPU context
    return ctx.Pool(processes=cores), cores


# ------------------------------------------------------------------ arms

def setup_layers(w, layers, device, csa, refine8=0):
    import torch
    import synth
    shape = csa.make_shape(w.B, w.Hq, w.Hkv, w.d, w.n, w.dtype)
    data = []
    for lid in layers:
        K, V, meta = synth.kv_torch(w, layer=lid, device=device)
        mt = csa.meta_buffers(shape, device)
        csa.check(csa.csa_quantize_keys(shape, K, V, [w.n] * w.B, 0, *mt),
                  "csa_quantize_keys")
        qs = [synth.q_torch(w, meta, s, layer=lid, device=device)
              for s in range(4)]
        data.append({"K": K, "V": V, "meta": mt, "q": qs, "lid": lid})
        if refine8:
            m8 = csa.meta8_buffers(shape, device)
            csa.check(csa.csa_quantize_keys8(shape, K, [w.n] * w.B, 0, *m8),
                      "csa_quantize_keys8")
            data[-1]["meta8"] = m8
    torch.cuda.synchronize()
    return shape, data


def seeds_for(w, lid, s):
    import synth
    return [int(x) for x in synth.step_seeds(w, s, layer=lid)]


def run_ours(args, world, rank, local):
    import numpy as np
    import torch
    import synth
    import certified_sparse_attention_gb300 as csa
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    csa.load_library()
    w = synth.workload(WORKLOAD)
    if args.n or args.batch:
        # smaller captures for profilers; never used for the reported line
        import dataclasses
        w = dataclasses.replace(w, n=args.n or w.n, B=args.batch or w.B)
    layers = rank_layers(rank, world, args.layers)
    shape, data = setup_layers(w, layers, device, csa, args.refine8)
    # --sub-batches: profiler captures of the unsplit chain (a scheduling
    # choice only; the reported line uses the default)
    params = csa.make_params(w.eps, w.delta, w.r, sub_batches=args.sub_batches,
                             qcode=args.qcode, refine8=args.refine8,
                             dots=args.dots)
    step = csa.DecodeStep(shape, params, device, with_stats=False)
    step_diag = csa.DecodeStep(shape, params, device, with_stats=True)
    dense = csa.DenseDecode(shape, device)
    lens = [w.n] * w.B
    stream = torch.cuda.current_stream(device)

    nseed = max(args.steps, args.warmup, 64)
    seed_tab = [[seeds_for(w, d["lid"], s) for s in range(nseed)]
                for d in data]

    def one(s, L):
        d = data[L]
        step(d["q"][s % 4], d["K"], d["V"], d["meta"], lens,
             seed_tab[L][s % nseed], stream, meta8=d.get("meta8"))

    for s in range(args.warmup):
        one(s, s % args.layers)
        dense(data[s % args.layers]["q"][0], data[s % args.layers]["K"],
              data[s % args.layers]["V"], lens, stream)
    torch.cuda.synchronize()
    csa.csa_profile_read()                      # reset launch counter

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    plan = step_plan(rank, args.steps, args.layers)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for (L, s) in plan:
        one(s, L)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_sparse = e0.elapsed_time(e1) / args.steps
    launches = csa.csa_profile_read()["launches"]
    # the device status word of the last timed step (non-finite inputs, an
    # exhausted buffer): a failing run prints no number
    csa.check(csa.csa_check(step.ws, stream), "csa_check (timed steps)")
    # same-build dense comparator over the same rotation
    e0.record(stream)
    for (L, s) in plan:
        d = data[L]
        dense(d["q"][s % 4], d["K"], d["V"], lens, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    ms_dense = e0.elapsed_time(e1) / args.steps
    ms_sparse = max_over_ranks(ms_sparse, world, device)
    ms_dense = max_over_ranks(ms_dense, world, device)

    # per-step times (events around each step on the caller's stream, after
    # the join), for the median and 90th percentile
    ndist = min(len(plan), 100)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * ndist)]
    for i, (L, s) in enumerate(plan[:ndist]):
        evs[2 * i].record(stream)
        one(s, L)
        evs[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    per_step = sorted(evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(ndist))
    step_dist = {"steps": ndist,
                 "median_us": round(per_step[ndist // 2] * 1e3, 1),
                 "p90_us": round(per_step[min(ndist - 1, (9 * ndist) // 10)] * 1e3, 1)}

    # live per-phase times (CUDA events at phase boundaries on the stream)
    csa.csa_profile_enable(True)
    nprof = min(args.steps, 32)
    for (L, s) in plan[:nprof]:
        one(s, L)
    torch.cuda.synchronize()
    prof = csa.csa_profile_read()
    csa.csa_profile_enable(False)
    phase_ms = {k: v / max(prof["steps"], 1) for k, v in prof["ms"].items()}

    # algorithmic bytes: diagnostics of one step on every rotated layer;
    # the same steps against float64 exact attention (certificate coverage)
    abs_ = []
    reads = []
    cov = Coverage(w)
    for L in range(args.layers):
        d = data[L]
        step_diag(d["q"][L % 4], d["K"], d["V"], d["meta"], lens,
                  seed_tab[L][L % nseed], stream, meta8=d.get("meta8"))
        torch.cuda.synchronize()
        csa.check(csa.csa_check(step_diag.ws, stream), "csa_check")
        stats = step_diag.stats.cpu().numpy()
        abs_.append(algorithmic_bytes(stats, w, w.n))
        reads.append((stats[..., 1].mean(), stats[..., 2].mean()))
        cov.add(d["q"][L % 4], d["K"], d["V"], lens, step_diag)
    ab = {k: sum(x[k] for x in abs_) / len(abs_) for k in abs_[0]}
    clt, modes, loop = None, None, None
    if not args.no_modes and args.decode_layers > 0:
        loop = decode_loop(args, csa, w, device, stream)
    if not args.no_modes:
        clt = clt_comparison(args, csa, w, shape, data, lens, seed_tab, nseed,
                             plan, stream, device, reads)
        # the other error measures of the pages' problem setup as modes
        modes = {name: run_mode(args, csa, w, shape, data, lens, seed_tab,
                                nseed, plan, stream, device, m, pt)
                 for name, m, pt in (("output", csa.CSA_MEASURE_OUTPUT, 0),
                                     ("denom", csa.CSA_MEASURE_DENOM, 0),
                                     ("value_per_head_draws",
                                      csa.CSA_MEASURE_VALUE, 1))}
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    phase_bytes = {"scan": ab["scan"], "rescore": ab["rows_k"],
                   "vgather": ab["rows_v"]}
    phase_ms.setdefault("rescore", 0.0)
    dom = max(phase_bytes, key=lambda k: phase_ms.get(k, 0.0))
    dom_all = max(phase_ms, key=lambda k: phase_ms[k])
    achieved = phase_bytes[dom] / (phase_ms[dom] * 1e-3) / 1e9
    traffic, scan_issue = None, None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            with open(tpath) as f:
                tr = json.load(f)
            traffic = tr.get(dom)
            scan_issue = tr.get("scan_issue_active_pct")
        except (OSError, ValueError):
            traffic = None
    step_gbs = ab["total"] / (ms_sparse * 1e-3) / 1e9
    dense_bytes = w.B * w.Hkv * w.n * 4 * w.d
    dense_gbs = dense_bytes / (ms_dense * 1e-3) / 1e9

    # end to end through the C ABI with host buffers: H2D of the step's
    # queries, re-quantisation of the last token's block, the step, D2H of
    # the results
    qh = torch.empty_like(data[0]["q"][0], device="cpu").pin_memory()
    qh.copy_(data[0]["q"][0].cpu())
    qd = torch.empty_like(data[0]["q"][0])
    # o, beta, level and keys_read: one buffer, one copy back per step
    outh = torch.empty_like(step.outputs, device="cpu").pin_memory()
    ne2e = max(1, min(args.steps, 64))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for (L, s) in plan[:ne2e]:
        d = data[L]
        qd.copy_(qh, non_blocking=True)
        csa.check(csa.csa_quantize_keys(shape, d["K"], d["V"], lens,
                                        w.n - 1, *d["meta"], stream))
        step(qd, d["K"], d["V"], d["meta"], lens, seed_tab[L][s % nseed],
             stream, meta8=d.get("meta8"))
        outh.copy_(step.outputs, non_blocking=True)
        stream.synchronize()
    ms_e2e = (time.perf_counter() - t0) * 1e3 / ne2e
    ms_e2e = max_over_ranks(ms_e2e, world, device)
    h2d = qh.numel() * qh.element_size()
    d2h = outh.numel() * outh.element_size()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pool, cores = cpu_pool()
        try:
            sp, de, sp_core, de_core = oracle_step_times(pool, cores, w, 0)
            w16 = synth.workload("llama16k")
            sp16, de16, sp16_core, _ = oracle_step_times(pool, cores, w16, 0,
                                                         name="llama16k")
        finally:
            pool.close()
            pool.join()
        cpu = {"value": round(sp * 1e6, 1), "unit": "us/step",
               "cores": cores, "kind": "oracle",
               "sample": f"{min(cores, w.B * w.Hkv)} of the step's "
                         f"{w.B * w.Hkv} (sequence, KV head) groups (half "
                         "peaked, half near-uniform, drawn by the numpy back "
                         "end of the same generator), one per process in "
                         f"parallel on {cores} host cores; value = mean core "
                         "time per group x groups per step / cores",
               "single_core_us": round(sp_core * 1e6, 1),
               "dense_oracle_us": round(de * 1e6, 1),
               "llama16k": {"workload": workload_name(w16),
                            "value": round(sp16 * 1e6, 1),
                            "single_core_us": round(sp16_core * 1e6, 1),
                            "dense_oracle_us": round(de16 * 1e6, 1)}}

    levels = stats[..., 0]
    line = {
        "metric": METRIC,
        # whole job: N ranks each complete a step in ms_sparse (max over
        # ranks), so the job's time per step is ms_sparse / N
        "value": round(ms_sparse * 1e3 / world, 2),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_sparse, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded generator with Llama-3.1-8B-shaped "
                "heads (keys = norm-4 shared direction + N(0,1) with 4 "
                "outlier channels x8 and 32 needles per KV head; values "
                "N(0,1) x lognormal(0,0.5); half the groups near-uniform); "
                "stands in for the pages' real KV caches",
        "config": {"workload": workload_name(w),
                   "layers_rotated": args.layers,
                   "l2": f"inputs larger than L2: {args.layers} resident "
                         f"layers (~{args.layers * 2.3:.0f} GB) rotated "
                         "between steps",
                   "batch_per_gpu": w.B},
        "roofline": {"bound": "hbm", "kernel": dom,
                     "achieved": round(achieved, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "peak_source": peak_src, "traffic": traffic,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     # the scan's secondary bound: ncu issue-slot use
                     "scan_issue_active_pct": scan_issue},
        "step_roofline": {"algorithmic_bytes": round(ab["total"]),
                          "achieved_gbs": round(step_gbs, 1),
                          "frac": round(step_gbs / hbm_peak, 4),
                          "frac_of_nominal": round(step_gbs / NOMINAL_HBM_GBS, 4)},
        "phase_us": {k: round(v * 1e3, 1) for k, v in phase_ms.items()},
        "dominant_phase": dom_all,
        "step_us_distribution": step_dist,
        "dense_us_per_step": round(ms_dense * 1e3, 2),
        "dense_gbs": round(dense_gbs, 1),
        "sparse_over_dense_time": round(ms_sparse / ms_dense, 3),
        "levels_hist": [int(x) for x in np.bincount(levels.ravel())],
        "certificate": cov.summary(),
        "clt_comparison": clt,
        "measures": modes,
        "decode_loop": loop,
        "keys_read_mean": float(stats[..., 1].mean()),
        "values_read_mean": float(stats[..., 2].mean()),
        "clocks": clocks.summary(),
        "e2e": {"value": round(ms_e2e * 1e3 / world, 2), "unit": "us/step",
                "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(launches),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, world, rank, local):
    """The oracle, as it stands, on the host cores: each step is one whole
    step of the workload (all its (sequence, KV head) groups) spread over
    the host cores."""
    if rank != 0:
        return
    wfull = synth_workload(WORKLOAD)
    # each step costs seconds of host time: at most 3 warm-up and 6 timed
    # steps (the line reports the counts actually run)
    args.steps = max(1, min(args.steps, 6))
    args.warmup = min(args.warmup, 3)
    pool, cores = cpu_pool()
    times, core_times = [], []
    try:
        for s in range(args.warmup + args.steps):
            sp, _, sp_core, _ = oracle_step_times(pool, cores, wfull, s)
            if s >= args.warmup:
                times.append(sp)
                core_times.append(sp_core)
    finally:
        pool.close()
        pool.join()
    us = statistics.mean(times) * 1e6
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(us, 1), "unit": "us/step",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(us / 1e3, 3), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same generator and workload as the GPU arm)",
        "config": {"workload": workload_name(wfull)},
        "cpu_baseline": {"value": round(us, 1), "unit": "us/step",
                         "cores": cores, "kind": "oracle",
                         "sample": f"each step: {min(cores, wfull.B * wfull.Hkv)} of "
                                   f"its {wfull.B * wfull.Hkv} (sequence, KV head) "
                                   "groups, one per process in parallel on "
                                   f"{cores} host cores; value = mean core time "
                                   "per group x groups per step / cores",
                         "single_core_us": round(statistics.mean(core_times) * 1e6, 1)},
        "e2e": {"value": round(us, 1), "unit": "us/step",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def context_sweep(args):
    """Step time against context length: the certified sparse step and the
    same-build dense decode for the 16K single-layer shape, then 128K to 1M
    tokens (batch 1, and batch 4 up to 256K), two independently seeded
    layers rotated.  One JSON line per point; not part of the benchmark
    line."""
    import torch
    import synth
    import certified_sparse_attention_gb300 as csa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    csa.load_library()
    points = [("llama16k", 16384, 1)]
    points += [(WORKLOAD, n, B) for n in (131072, 262144, 524288, 1048576)
               for B in (1, 4) if not (B == 4 and n > 262144)]
    for name, n, B in points:
        w = synth.workload(name, n=n, B=B)
        shape, data = setup_layers(w, [0, 1], dev, csa)
        step = csa.DecodeStep(shape, csa.make_params(w.eps, w.delta, w.r), dev)
        dense = csa.DenseDecode(shape, dev)
        lens = [n] * B
        st = torch.cuda.current_stream(dev)

        def run_sparse(i):
            d = data[i % 2]
            step(d["q"][i % 4], d["K"], d["V"], d["meta"], lens,
                 seeds_for(w, d["lid"], i), st, meta8=d.get("meta8"))

        def run_dense(i):
            d = data[i % 2]
            dense(d["q"][i % 4], d["K"], d["V"], lens, st)

        res = {}
        for key, fn in (("sparse_us", run_sparse), ("dense_us", run_dense)):
            for i in range(4):
                fn(i)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for i in range(20):
                fn(i)
            e1.record(st)
            torch.cuda.synchronize()
            res[key] = round(e0.elapsed_time(e1) / 20 * 1e3, 1)
        csa.check(csa.csa_check(step.ws), "csa_check (context sweep)")
        print(json.dumps({"context_sweep": {"workload": name, "n": n, "B": B,
                                            "r": w.r, **res}}), flush=True)
        del data, step, dense
        torch.cuda.empty_cache()


def stress_sweep(args):
    """The stress sweep of the pages' setting: batch 1, 8 KV heads, GQA 4,
    d = 128, bf16, r = 2, n in {256K, 512K, 1M} tokens, eps in {0.01, 0.02,
    0.05, 0.1}, three attention regimes (flat: q x 0.05; heavy-tailed:
    Pareto(1.5) boosts along the needle direction; adversarial: ceil(eps^-2)
    keys sharing one boosted score over a flat background).  Per point: the
    certified step and the same-build dense decode (CUDA events, 10 steps
    after 3 warm-up steps), keys and values read per head, stop levels, and
    certificate coverage of 4 steps against float64 exact attention.  One
    JSON line per point; not part of the benchmark line."""
    import torch
    import synth
    import certified_sparse_attention_gb300 as csa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    csa.load_library()
    st = torch.cuda.current_stream(dev)
    for regime in ("flat", "heavy", "adversarial"):
        for n in (262144, 524288, 1048576):
            data = None
            for eps in (0.01, 0.02, 0.05, 0.1):
                w = synth.stress(n, eps, regime)
                if data is None or regime == "adversarial":
                    data = None
                    torch.cuda.empty_cache()
                    shape, data = setup_layers(w, [0], dev, csa)
                d = data[0]
                params = csa.make_params(w.eps, w.delta, w.r)
                step = csa.DecodeStep(shape, params, dev, with_stats=True)
                dense = csa.DenseDecode(shape, dev)
                lens = [n]
                seeds = [seeds_for(w, 0, i) for i in range(14)]

                def run_sparse(i):
                    step(d["q"][i % 4], d["K"], d["V"], d["meta"], lens,
                         seeds[i], st)

                def run_dense(i):
                    dense(d["q"][i % 4], d["K"], d["V"], lens, st)

                res = {}
                for key, fn in (("sparse_us", run_sparse),
                                ("dense_us", run_dense)):
                    for i in range(3):
                        fn(i)
                    torch.cuda.synchronize()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(st)
                    for i in range(3, 13):
                        fn(i)
                    e1.record(st)
                    torch.cuda.synchronize()
                    res[key] = round(e0.elapsed_time(e1) / 10 * 1e3, 1)
                cov = Coverage(w)
                kr, vr, lv = [], [], []
                for i in range(4):
                    run_sparse(i)
                    torch.cuda.synchronize()
                    csa.check(csa.csa_check(step.ws), "csa_check (stress)")
                    sts = step.stats.cpu()
                    kr.append(float(sts[..., 1].float().mean()))
                    vr.append(float(sts[..., 2].float().mean()))
                    lv.extend(sts[..., 0].flatten().tolist())
                    cov.add(d["q"][i % 4], d["K"], d["V"], lens, step)
                c = cov.summary()
                print(json.dumps({"stress_sweep": {
                    "regime": regime, "n": n, "eps": eps, "r": w.r, **res,
                    "sparse_over_dense": round(res["sparse_us"] / res["dense_us"], 3),
                    "keys_read_mean": round(sum(kr) / len(kr), 1),
                    "values_read_mean": round(sum(vr) / len(vr), 1),
                    "level_mean": round(sum(lv) / len(lv), 2),
                    "level_max": int(max(lv)),
                    "head_steps": c["head_steps"],
                    "beta_violations": c["beta_violations"],
                    "eps_violations": c["eps_violations"],
                    "fallbacks": c["fallbacks"],
                    "err_over_epsM_p90": c["err_over_epsM"]["p90"],
                    "err_over_epsM_max": c["err_over_epsM"]["max"]}}),
                    flush=True)
                del step, dense
            del data
            torch.cuda.empty_cache()


def dense_only(args):
    """The same-build dense decode alone on the benchmark workload (or the
    --n / --batch reduction), for profiler captures of that kernel: warm-up
    and timed calls on one resident layer; one JSON line with its time and
    bytes per second.  Not part of the benchmark line."""
    import dataclasses
    import torch
    import synth
    import certified_sparse_attention_gb300 as csa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    csa.load_library()
    w = synth.workload(WORKLOAD)
    if args.n or args.batch:
        w = dataclasses.replace(w, n=args.n or w.n, B=args.batch or w.B)
    shape, data = setup_layers(w, [0], dev, csa)
    d = data[0]
    dense = csa.DenseDecode(shape, dev)
    lens = [w.n] * w.B
    st = torch.cuda.current_stream(dev)
    for i in range(args.warmup):
        dense(d["q"][i % 4], d["K"], d["V"], lens, st)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(args.steps):
        dense(d["q"][i % 4], d["K"], d["V"], lens, st)
    e1.record(st)
    torch.cuda.synchronize()
    csa.check(csa.csa_check(dense.ws), "csa_check (dense)")
    us = e0.elapsed_time(e1) / args.steps * 1e3
    nbytes = 2 * w.B * w.Hkv * w.n * w.d * 2
    print(json.dumps({"dense_only": {"workload": w.name, "n": w.n, "B": w.B,
                                     "us": round(us, 1),
                                     "gbs": round(nbytes / us / 1e3, 1)}}))


def synth_workload(name):
    import synth
    return synth.workload(name)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--n", type=int, default=0,
                    help="override the context length (profiler captures)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch (profiler captures)")
    ap.add_argument("--dense-only", action="store_true",
                    help="time the same-build dense decode alone (profiler "
                         "captures of that kernel)")
    ap.add_argument("--stress-sweep", action="store_true",
                    help="the stress sweep (256K-1M tokens, eps 0.01-0.1, "
                         "flat / heavy-tailed / adversarial): one JSON line "
                         "per point instead of the benchmark line")
    ap.add_argument("--context-sweep", action="store_true",
                    help="print step times from 128K to 1M tokens and exit")
    ap.add_argument("--decode-layers", type=int, default=32,
                    help="layers of the whole-model decode loop (0: skip it)")
    ap.add_argument("--no-modes", action="store_true",
                    help="skip the CLT / other-measure comparisons (profiler captures)")
    ap.add_argument("--dots", type=int, default=0,
                    help="the scan's integer dots: 0 tensor cores, 1 dp4a")
    ap.add_argument("--refine8", type=int, default=0,
                    help="8-bit refinement tier: 0 off, 1 every group, 2 "
                         "groups whose first range reaches level r")
    ap.add_argument("--qcode", type=int, default=0,
                    help="query code of the 4-bit bounds: 0 int8, 1 two digits")
    ap.add_argument("--sub-batches", type=int, default=0,
                    help="sub-batches of the decode call (0: the library default)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank, local)
        return
    if args.dense_only:
        if rank == 0:
            dense_only(args)
        return
    if args.stress_sweep:
        if rank == 0:
            stress_sweep(args)
        return
    if args.context_sweep:
        if rank == 0:
            context_sweep(args)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
