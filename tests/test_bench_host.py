"""Host-side logic of the benchmark (no GPU): the algorithmic bytes it
divides by the kernels' times, the workload naming, the ranks' layer split,
the clock-record summary and the coverage count."""
import numpy as np

import bench
import synth


def test_algorithmic_bytes_per_unit():
    # per (sequence, KV head): the scan reads d/2 + 8d/64 + 4/64 bytes per
    # key (80.06 at d = 128, 16.4% of a dense K+V read); each K or V row
    # the group needs costs 2d bytes; each query head's per-level sums
    # (J + 1)(2d + 6) floats
    w = synth.workload("llama128k_b4")
    n = w.n
    stats = np.zeros((w.B, w.Hq, 10), np.int32)
    stats[..., 5] = 68                   # J
    stats[..., 7] = 1000                 # group keys read (same for the group)
    stats[..., 8] = 300                  # group values read
    ab = bench.algorithmic_bytes(stats, w, n)
    per_key = w.d / 2 + 8 * w.d / 64 + 4 / 64
    assert abs(per_key - 80.0625) < 1e-12
    assert abs(per_key / (4 * w.d) - 0.1564) < 1e-3
    groups = w.B * w.Hkv
    assert ab["scan"] == groups * n * per_key
    assert ab["rows_k"] == groups * 1000 * 2 * w.d
    assert ab["rows_v"] == groups * 300 * 2 * w.d
    assert ab["scratch"] == w.B * w.Hq * 69 * (2 * w.d + 6) * 4
    assert ab["total"] == ab["scan"] + ab["rows_k"] + ab["rows_v"] + ab["scratch"]


def test_workload_name_states_the_shape():
    w = synth.workload("llama128k_b4")
    name = bench.workload_name(w)
    for part in ("n=131072", "Hq=32", "Hkv=8", "d=128", "bf16", "r=4"):
        assert part in name


def test_ranks_take_disjoint_layers_and_cycle_them():
    world, layers, steps = 4, 3, 10
    seen = set()
    for rank in range(world):
        ids = bench.rank_layers(rank, world, layers)
        assert len(ids) == layers and not (seen & set(ids))
        seen |= set(ids)
        plan = bench.step_plan(rank, steps, layers)
        assert [s for _, s in plan] == list(range(steps))
        assert [slot for slot, _ in plan] == [s % layers for s in range(steps)]


def test_clock_summary_reads_reasons_and_median():
    cs = bench.ClockSampler(0)
    cs.rows = [["1980", "2070", "900.1", "Not Active", "Not Active",
                "Not Active", "Active"],
               ["2070", "2070", "950.0", "Not Active", "Not Active",
                "Not Active", "Not Active"],
               ["[N/A]", "2070", "955.0", "Not Active", "Active",
                "Not Active", "Not Active"]]
    s = cs.summary()
    assert s["sm_mhz"] == (1980 + 2070) / 2 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert s["samples"] == 3
    empty = bench.ClockSampler(0).summary()
    assert empty["sm_mhz"] is None and empty["reasons"] == []


def test_coverage_counts_violations_against_exact_attention():
    """The coverage check against float64 exact attention: an exact output
    has no violation; one moved by 2 eps M violates both its beta and the
    eps target; a fallback head (level past J) is not held to beta."""
    import math
    import types
    import torch
    w = types.SimpleNamespace(B=1, Hq=2, Hkv=1, G=2, d=8, n=200, r=2,
                              eps=0.05, delta=0.05)
    g = torch.Generator().manual_seed(3)
    K = torch.randn(1, 1, w.n, w.d, generator=g)
    V = torch.randn(1, 1, w.n, w.d, generator=g)
    q = torch.randn(1, 2, w.d, generator=g)
    a = torch.softmax(q[0].double() @ K[0, 0].double().T / math.sqrt(w.d), 1)
    o = a @ V[0, 0].double()
    M = torch.sqrt(a @ (V[0, 0].double() ** 2).sum(1))
    J = math.ceil(w.r * math.log2(w.n - 64))
    shift = torch.zeros(2, w.d, dtype=torch.float64)
    shift[1, 0] = 2 * w.eps * M[1]
    step = types.SimpleNamespace(o=(o + shift)[None].float(),
                                 beta=torch.full((1, 2), 1e-3),
                                 level=torch.tensor([[3, J + 1]]))
    cov = bench.Coverage(w)
    cov.add(q, K, V, [w.n], step)
    s = cov.summary()
    assert s["head_steps"] == 2 and s["fallbacks"] == 1
    assert s["eps_violations"] == 1
    assert s["beta_violations"] == 0          # head 1 fell back
    step.level = torch.tensor([[3, 5]])
    cov = bench.Coverage(w)
    cov.add(q, K, V, [w.n], step)
    assert cov.summary()["beta_violations"] == 1
