"""Write the oracle regression fixtures in this folder.

Calls only ``oracle/`` (and the seeded input generator ``synth``); no value
here comes from the CUDA library.  The pages print no worked example, so these
fixtures pin the oracle against its own earlier output (a regression guard),
not against the pages.

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import synth  # noqa: E402
from oracle.step import Params, oracle_decode_group  # noqa: E402

CASES = [
    # name, workload, overrides, n, step, seed[, oracle parameter overrides]
    ("tiny_n300", "tiny", {}, 300, 2, 77),
    ("llama_g2_n700", "llama16k", {"Hq": 8, "Hkv": 2}, 700, 0, 12345),
    # the uncertified CLT comparison rule and per-query-head draws
    ("llama_g2_n700_clt", "llama16k", {"Hq": 8, "Hkv": 2}, 700, 0, 12345,
     {"measure": 3}),
    ("llama_g2_n700_perhead", "llama16k", {"Hq": 8, "Hkv": 2}, 700, 0, 12345,
     {"per_head": True}),
    # the 8-bit refinement option (changes keys_read only)
    ("llama_g2_n700_refine8", "llama16k", {"Hq": 8, "Hkv": 2}, 700, 0, 12345,
     {"refine8": True}),
]


def _digest(a):
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()[:16]


def run_case(wname, over, n, step, seed, pover=None):
    w = synth.workload(wname, B=1, n=n, **over)
    K, V, meta = synth.kv_numpy(w)
    q = synth.q_numpy(w, meta, step, K=K)
    out = []
    for g in range(w.Hkv):
        res = oracle_decode_group(q[0, g * w.G:(g + 1) * w.G], K[0, g],
                                  V[0, g], n, seed, g,
                                  Params(w.eps, w.delta, w.r, **(pover or {})))
        for h, det in enumerate(res.detail):
            extra = ({"rows8": int(res.rows8[h]),
                      "jref_sha": _digest(det["jref"].astype(np.int64))}
                     if res.rows8 is not None else {})
            out.append({
                "g": g, "h": h, "J": res.J,
                "o": [float(x) for x in res.o[h]],
                "beta": float(res.beta[h]), "level": int(res.level[h]),
                "keys_read": int(res.keys_read[h]),
                "values_read": int(res.values_read[h]),
                "n_candidates": int(res.n_candidates[h]),
                "c_lo": float(det["c_lo"]), "c_hi": float(det["c_hi"]),
                "cb": float(det["cb"]),
                "jbar_sha": _digest(det["jbar"].astype(np.int64)),
                "ubar_sha": _digest(det["ubar"].astype(np.float32)),
                **extra,
            })
    return out


def main():
    for case in CASES:
        name, wname, over, n, step, seed = case[:6]
        pover = case[6] if len(case) > 6 else {}
        data = {"case": name, "workload": wname, "overrides": over, "n": n,
                "step": step, "seed": seed, "params": pover,
                "heads": run_case(wname, over, n, step, seed, pover)}
        with open(os.path.join(HERE, name + ".json"), "w") as f:
            json.dump(data, f, indent=1)
        print("wrote", name)


if __name__ == "__main__":
    main()
