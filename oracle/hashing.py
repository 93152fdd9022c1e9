"""Counter-hash perturbations E_i = -ln u_i.

picx.dev summary, "Algorithm Components" 1: each pool key's perturbation is
E_i = -ln u_i with u_i a uniform number made from 53 hashed bits;
readsearch.ai "Abstract": the draws are new at each decode step, and a GQA
group shares one scan.

The hash is SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; constants of Vigna's splitmix64.c): the
k-th output of a generator seeded with s is mix64(s + k * gamma).
  group key  K_{b,g} = mix64(step_seed_b + (g + 1) * gamma)
  key hash   h_i     = mix64(K_{b,g} + (i + 1) * gamma),  i = token position
  uniform    u_i     = ((h_i >> 11) + 1) * 2^-53  in (0, 1]
  log2 units t_i     = -log2 u_i = 53 - log2((h_i >> 11) + 1)  (float32)
so E_i = t_i * ln 2 >= 0 is finite.  The draw depends on (sequence, KV head,
position, step seed) only, so it is shared by the G query heads of a group.
Optional per-query-head draws (the alternative the sharing question leaves
open): query head h of group g uses stream PER_HEAD_STREAM + g G + h in
place of g, so every head has its own independent draw.
Test infrastructure only.
"""
from __future__ import annotations

import numpy as np

from .fp32 import log2_m53_f32

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)


def mix64(z):
    """SplitMix64 output function (wrapping 64-bit arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        z = z ^ (z >> np.uint64(31))
    return z


PER_HEAD_STREAM = 1 << 20    # stream ids of per-query-head draws start here


def head_stream(g: int, G: int, h: int) -> int:
    """Stream id of query head h of KV group g (per-query-head draws)."""
    return PER_HEAD_STREAM + g * G + h


def group_key(step_seed: int, g: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.uint64(step_seed) + np.uint64(g + 1) * GAMMA
    return mix64(s)[()]


def key_hashes(step_seed: int, g: int, idx: np.ndarray) -> np.ndarray:
    k = group_key(step_seed, g)
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = k + (idx + np.uint64(1)) * GAMMA
    return mix64(z)


def perturb_t(step_seed: int, g: int, idx: np.ndarray) -> np.ndarray:
    """t_i = -log2 u_i in float32 for positions ``idx`` of group g."""
    h = key_hashes(step_seed, g, idx)
    m = (h >> np.uint64(11)) + np.uint64(1)
    return np.float32(53.0) - log2_m53_f32(m)
