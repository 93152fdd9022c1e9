"""Seeded synthetic decode-attention inputs.

This module only draws random tensors with the shapes and value laws of the
decode workloads described in "Certified Sparse Attention via Perturbed
Retrieval" (picx.dev summary, Introduction / Background: Llama-3.1-8B-shaped
heads at 16K-128K tokens, 16-bit KV cache).  It contains none of the method's
arithmetic: no quantisation, no scores, no sampling.  Both the CPU oracle
(``oracle/``) and the CUDA path receive the tensors it returns.

Two back ends draw the same recipe:
  * ``numpy``  -- small cases for CPU tests (stable ``numpy.random`` streams);
  * ``torch``  -- any device; used for large, device-resident workloads.
The two back ends give different random streams; a test always hands the
*same* tensors to both sides.

Recipe (per layer ``l``, sequence ``b``, KV head ``g``):
  * keys    k_i = 4 * mu_g + z_i,  z_i ~ N(0, I_d), four fixed outlier
              channels of z multiplied by 8;  mu_g a random unit vector;
  * needles 32 pool positions per (b, g) get k_i += 8 * nu_g, where nu_g is
              the head group's needle direction (raises q.k/sqrt(d) by ~8);
  * values  v_i = lambda_i * N(0, I_d),  lambda_i ~ LogNormal(0, 0.5);
  * queries q = sqrt(d) * nu_g + N(0, I_d) per query head of group g; the
              odd groups are "near-uniform": q scaled by 0.1 (``flat_scale``);
  * 16-bit workloads round K, V and q to bfloat16 (round to nearest even).
The tiny case ("tiny"): fp32 K, V, q ~ N(0, 1), d = 64, one head, eight planted
pool keys reset to 3 q / ||q|| at every step.
Stress regimes: "flat" scales q by 0.05; "heavy" adds Pareto(1.5) - 1 boosts
along nu_g to every key; "adversarial" gives ceil(eps^-2) keys one shared
boosted score over a flat background.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

BASE_SEED = 20261202
WINDOW = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and law of one decode-attention workload."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    n: int
    dtype: str = "bf16"          # "bf16" or "f32"
    eps: float = 0.05
    delta: float = 0.05
    r: int = 2
    layers: int = 1
    steps: int = 1
    regime: str = "mixed"        # mixed | flat | heavy | adversarial | tiny
    n_needles: int = 32
    flat_scale: float = 0.1

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


def workload(name: str, **over) -> Workload:
    """Named workloads (the parity and benchmark cases)."""
    table = {
        # one head, d=64, n=2048 fp32, 8 planted keys, eps .05 delta .01 r 2
        "tiny": Workload("tiny", 1, 1, 1, 64, 2048, "f32", 0.05, 0.01, 2,
                         steps=16, regime="tiny", n_needles=8),
        # Llama-3.1-8B-shaped single layer at 16K
        "llama16k": Workload("llama16k", 1, 32, 8, 128, 16384, "bf16",
                             0.05, 0.05, 2),
        # batch 8 at 32K with appends
        "llama32k_b8": Workload("llama32k_b8", 8, 32, 8, 128, 32768, "bf16",
                                0.05, 0.05, 2, steps=64),
        # the 128K headline shape: batch 4, 32 layers, r = 4
        "llama128k_b4": Workload("llama128k_b4", 4, 32, 8, 128, 131072, "bf16",
                                 0.05, 0.05, 4, layers=32, steps=256),
    }
    w = table[name]
    return dataclasses.replace(w, **over) if over else w


def stress(n: int, eps: float, regime: str) -> Workload:
    """Stress sweep cases: batch 1, 8 KV heads, GQA 4, d=128, bf16, r=2."""
    return Workload(f"stress_{regime}_{n}_{eps}", 1, 32, 8, 128, n, "bf16",
                    eps, 0.05, 2, regime=regime)


def outlier_channels(d: int) -> list[int]:
    return [c * d // 128 for c in (5, 37, 70, 101)]


def bf16_round_np(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = (u + 0x7FFF + lsb) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _seed(*parts: int) -> np.random.SeedSequence:
    return np.random.SeedSequence([BASE_SEED, *[int(p) for p in parts]])


def _unit(rng: np.random.Generator, d: int) -> np.ndarray:
    u = rng.standard_normal(d)
    return (u / np.linalg.norm(u)).astype(np.float32)


# ----------------------------------------------------------------------------
# numpy back end
# ----------------------------------------------------------------------------

def kv_numpy(w: Workload, layer: int = 0, n: Optional[int] = None):
    """K, V as float32 arrays [B, Hkv, n, d] (bf16-representable for bf16).

    Returns (K, V, meta) where meta holds the per-group directions needed to
    draw matching queries and the needle positions.
    """
    n = w.n if n is None else n
    B, H, d = w.B, w.Hkv, w.d
    K = np.empty((B, H, n, d), np.float32)
    V = np.empty((B, H, n, d), np.float32)
    mus = np.empty((H, d), np.float32)
    nus = np.empty((H, d), np.float32)
    needles = np.zeros((B, H, max(w.n_needles, 0)), np.int64)
    for g in range(H):
        rg = np.random.default_rng(_seed(1, layer, g))
        mus[g] = _unit(rg, d)
        nus[g] = _unit(rg, d)
    oc = outlier_channels(d)
    pool = max(n - WINDOW, 0)
    for b in range(B):
        for g in range(H):
            rng = np.random.default_rng(_seed(2, layer, b, g))
            if w.regime == "tiny":
                K[b, g] = rng.standard_normal((n, d), dtype=np.float32)
                V[b, g] = rng.standard_normal((n, d), dtype=np.float32)
                if pool > 0 and w.n_needles > 0:
                    needles[b, g] = rng.choice(pool, size=w.n_needles,
                                               replace=False)
                continue
            z = rng.standard_normal((n, d), dtype=np.float32)
            z[:, oc] *= 8.0
            k = 4.0 * mus[g][None, :] + z
            lam = np.exp(0.5 * rng.standard_normal(n)).astype(np.float32)
            v = rng.standard_normal((n, d), dtype=np.float32) * lam[:, None]
            if pool > 0 and w.n_needles > 0:
                pos = rng.choice(pool, size=min(w.n_needles, pool),
                                 replace=False)
                needles[b, g, :len(pos)] = pos
                k[pos] += 8.0 * nus[g][None, :]
            if w.regime == "heavy":
                boost = rng.pareto(1.5, size=n).astype(np.float32)
                k += boost[:, None] * nus[g][None, :]
            elif w.regime == "adversarial":
                m = int(math.ceil(w.eps ** -2))
                pos = rng.choice(max(pool, 1), size=min(m, max(pool, 1)),
                                 replace=False)
                k[pos] += 6.0 * nus[g][None, :]
            K[b, g] = k
            V[b, g] = v
    if w.dtype == "bf16":
        K = bf16_round_np(K)
        V = bf16_round_np(V)
    return K, V, {"mu": mus, "nu": nus, "needles": needles}


def q_numpy(w: Workload, meta: dict, step: int = 0, layer: int = 0,
            K: Optional[np.ndarray] = None) -> np.ndarray:
    """Queries [B, Hq, d] float32 for one decode step.

    For the tiny case the planted keys of ``K`` (if given) are reset in place
    to 3 q / ||q|| so that the step's attention is peaked.
    """
    B, Hq, d, G = w.B, w.Hq, w.d, w.G
    q = np.empty((B, Hq, d), np.float32)
    for b in range(B):
        rng = np.random.default_rng(_seed(3, layer, b, step))
        for h in range(Hq):
            g = h // G
            e = rng.standard_normal(d, dtype=np.float32)
            if w.regime == "tiny":
                q[b, h] = e
                continue
            v = math.sqrt(d) * meta["nu"][g] + e
            if w.regime == "flat":
                v = v * 0.05
            elif w.regime == "mixed" and g % 2 == 1:
                v = v * w.flat_scale
            elif w.regime == "adversarial":
                v = v * 0.05
            q[b, h] = v
    if w.regime == "tiny" and K is not None:
        for b in range(B):
            for g in range(w.Hkv):
                qq = q[b, g * G]
                K[b, g, meta["needles"][b, g]] = 3.0 * qq / np.linalg.norm(qq)
    if w.dtype == "bf16":
        q = bf16_round_np(q)
    return q


def step_seeds(w: Workload, step: int, layer: int = 0) -> np.ndarray:
    """Per-sequence 64-bit step seeds (uint64 [B])."""
    ss = _seed(4, layer, step).generate_state(2 * w.B, np.uint32)
    ss = ss.astype(np.uint64)
    return (ss[0::2] << np.uint64(32)) | ss[1::2]


# ----------------------------------------------------------------------------
# torch back end (device-resident, large workloads)
# ----------------------------------------------------------------------------

def kv_torch(w: Workload, layer: int = 0, device="cpu", n: Optional[int] = None,
             n_alloc: Optional[int] = None):
    """K, V as torch tensors [B, Hkv, n_alloc, d] in the workload's dtype.

    Rows [n, n_alloc) are zero (room for appended tokens).
    """
    import torch
    n = w.n if n is None else n
    n_alloc = n if n_alloc is None else n_alloc
    B, H, d = w.B, w.Hkv, w.d
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    K = torch.zeros((B, H, n_alloc, d), dtype=dt, device=device)
    V = torch.zeros((B, H, n_alloc, d), dtype=dt, device=device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(_seed(5, layer).generate_state(1)[0]))
    mus = torch.randn((H, d), generator=gen, device=device)
    mus = mus / mus.norm(dim=1, keepdim=True)
    nus = torch.randn((H, d), generator=gen, device=device)
    nus = nus / nus.norm(dim=1, keepdim=True)
    oc = outlier_channels(d)
    pool = max(n - WINDOW, 0)
    needles = torch.zeros((B, H, max(w.n_needles, 0)), dtype=torch.int64,
                          device=device)
    scale = torch.ones(d, device=device)
    scale[oc] = 8.0
    for b in range(B):
        for g in range(H):
            z = torch.randn((n, d), generator=gen, device=device) * scale
            k = 4.0 * mus[g][None, :] + z
            lam = torch.exp(0.5 * torch.randn(n, generator=gen, device=device))
            v = torch.randn((n, d), generator=gen, device=device) * lam[:, None]
            if pool > 0 and w.n_needles > 0:
                pos = torch.randperm(pool, generator=gen, device=device)
                pos = pos[:min(w.n_needles, pool)]
                needles[b, g, :len(pos)] = pos
                k[pos] += 8.0 * nus[g][None, :]
            if w.regime == "heavy":
                u = torch.rand(n, generator=gen, device=device).clamp_min(1e-12)
                boost = u.pow(-1.0 / 1.5) - 1.0
                k += boost[:, None] * nus[g][None, :]
            elif w.regime == "adversarial":
                m = int(math.ceil(w.eps ** -2))
                pos = torch.randperm(max(pool, 1), generator=gen,
                                     device=device)[:m]
                k[pos] += 6.0 * nus[g][None, :]
            K[b, g, :n] = k.to(dt)
            V[b, g, :n] = v.to(dt)
    return K, V, {"mu": mus, "nu": nus, "needles": needles}


def q_torch(w: Workload, meta: dict, step: int = 0, layer: int = 0,
            device="cpu"):
    import torch
    B, Hq, d, G = w.B, w.Hq, w.d, w.G
    gen = torch.Generator(device=device)
    gen.manual_seed(int(_seed(6, layer, step).generate_state(1)[0]))
    e = torch.randn((B, Hq, d), generator=gen, device=device)
    grp = torch.arange(Hq, device=device) // G
    q = math.sqrt(d) * meta["nu"][grp][None, :, :] + e
    if w.regime in ("flat", "adversarial"):
        q = q * 0.05
    elif w.regime == "mixed":
        sc = torch.where(grp % 2 == 1, w.flat_scale, 1.0).to(q.dtype)
        q = q * sc[None, :, None]
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    return q.to(dt)
