"""Shared helpers of the GPU parity tests (run the CUDA path through the C
ABI, run the oracle on the same inputs, compare)."""
from __future__ import annotations

import math
import os

import numpy as np

import synth

F = np.float32


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


class GpuRun:
    """One decode step of a workload on the GPU, with workspace views."""

    def __init__(self, w: synth.Workload, K, V, q, lens, seeds, n_alloc,
                 device="cuda:0", eps=None, delta=None, r=None,
                 measure=0, J_override=-1):
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
                                      J_override)
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
        self.step = csa.DecodeStep(self.shape, self.params, device,
                                   with_stats=True)
        self.step(self.q, self.K, self.V, self.meta, self.lens, self.seeds)
        torch.cuda.synchronize()
        csa.check(csa.csa_check(self.step.ws), "csa_check")
        self.map = csa.csa_workspace_layout(self.shape, self.params)

    def ws_view(self, off, count, dtype):
        import torch
        nbytes = count * 4
        t = self.step.ws[off:off + nbytes]
        return t.view(dtype).cpu().numpy()

    def ubar(self):
        import torch
        w = self.w
        n = self.shape.n_max
        a = self.ws_view(self.map.ubar, w.B * w.Hkv * n * w.G, torch.float32)
        return a.reshape(w.B, w.Hkv, n, w.G)

    def cmax(self):
        import torch
        w = self.w
        a = self.ws_view(self.map.cmax, w.B * w.Hq * 4, torch.int32)
        return self.csa.decode_ordered(a.view(np.uint32)).reshape(w.B, w.Hq, 4)

    def s32(self):
        import torch
        w = self.w
        pcap = max(self.shape.n_max - 64, 1)
        a = self.ws_view(self.map.s32, w.B * w.Hkv * pcap * w.G, torch.float32)
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
