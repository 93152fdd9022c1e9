"""Host-side arithmetic of the benchmark (no GPU): the algorithmic bytes it
divides by the kernels' times, and the workload naming."""
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
