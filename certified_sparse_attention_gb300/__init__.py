"""Certified sparse decode attention on GB300 -- Python binding of libcsa.

Thin ctypes layer over the C ABI in ``include/csa.h``: the functions below
carry the same names as the C entry points and only marshal arguments (torch
tensors -> device pointers, Python ints -> host arrays).  Every step of the
decode path runs in the library's CUDA kernels; there is no Python or CPU
fallback, and a missing library raises ``CsaLibraryMissing``.

PyTorch supplies device memory and streams only.

Paper: "Certified Sparse Attention via Perturbed Retrieval" (arXiv
2610.24991), picx.dev summary "Methodology" and "Algorithm Components" 1-4.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libcsa.so")

CSA_OK = 0
CSA_BF16, CSA_F32 = 0, 1
CSA_MEASURE_VALUE, CSA_MEASURE_OUTPUT, CSA_MEASURE_DENOM, CSA_MEASURE_CLT = \
    0, 1, 2, 3
WINDOW = 64
BLOCK = 64

EXPORTED = ("csa_workspace_size", "csa_quantize_keys", "csa_decode_step",
            "csa_dense_workspace_size", "csa_dense_decode", "csa_check",
            "csa_status_string", "csa_workspace_layout",
            "csa_profile_enable", "csa_profile_read",
            "csa_dense_decode_static", "csa_decode_step_device",
            "csa_quantize_keys8", "csa_decode_step_refined")
# size of the fixed scratch array behind csa_dense_decode_static
DENSE_STATIC_SCRATCH_BYTES = 16 << 20
STATS_FIELDS = 10
STAT = {"level": 0, "keys_read": 1, "values_read": 2, "n_candidates": 3,
        "n_near_threshold": 4, "J": 5, "rounds": 6, "group_keys_read": 7,
        "group_values_read": 8, "rows8": 9}
PHASES = ("clear", "scan", "exact_max", "candidates", "rescore", "predict",
          "levels", "plan", "vgather", "certify", "fallback", "diagnostics",
          "refine8")


class CsaLibraryMissing(RuntimeError):
    pass


class CsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


class csa_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int),
                ("Hkv", ctypes.c_int), ("d", ctypes.c_int),
                ("n_max", ctypes.c_int64), ("dtype", ctypes.c_int)]


class csa_params(ctypes.Structure):
    _fields_ = [("eps", ctypes.c_float), ("delta", ctypes.c_float),
                ("r", ctypes.c_int), ("measure", ctypes.c_int),
                ("J_override", ctypes.c_int), ("sub_batches", ctypes.c_int),
                ("perturb", ctypes.c_int), ("qcode", ctypes.c_int),
                ("refine8", ctypes.c_int), ("dots", ctypes.c_int)]


class csa_head_stats(ctypes.Structure):
    _fields_ = [("level", ctypes.c_int32), ("keys_read", ctypes.c_int32),
                ("values_read", ctypes.c_int32),
                ("n_candidates", ctypes.c_int32),
                ("n_near_threshold", ctypes.c_int32), ("J", ctypes.c_int32),
                ("rounds", ctypes.c_int32),
                ("group_keys_read", ctypes.c_int32),
                ("group_values_read", ctypes.c_int32),
                ("rows8", ctypes.c_int32)]


class csa_workspace_map(ctypes.Structure):
    _fields_ = [("ubar", ctypes.c_size_t), ("cmax", ctypes.c_size_t),
                ("s32", ctypes.c_size_t), ("jr_hist", ctypes.c_size_t),
                ("bcnt", ctypes.c_size_t), ("total", ctypes.c_size_t),
                ("J1", ctypes.c_int32), ("sub_batches", ctypes.c_int32),
                ("sub_stride", ctypes.c_size_t), ("sub_B", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class csa_phase_times(ctypes.Structure):
    _fields_ = [("ms", ctypes.c_float * 13), ("steps", ctypes.c_int32),
                ("launches", ctypes.c_int64)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libcsa.so (once).  Raises CsaLibraryMissing if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise CsaLibraryMissing(
            f"{path} is missing: build it with "
            "`python -m certified_sparse_attention_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER
    lib.csa_workspace_size.argtypes = [P(csa_shape), P(csa_params)]
    lib.csa_workspace_size.restype = sz
    lib.csa_dense_workspace_size.argtypes = [P(csa_shape)]
    lib.csa_dense_workspace_size.restype = sz
    lib.csa_quantize_keys.argtypes = [P(csa_shape), vp, vp, P(ctypes.c_int64),
                                      ctypes.c_int64, vp, vp, vp, vp, vp]
    lib.csa_quantize_keys.restype = ctypes.c_int
    lib.csa_decode_step.argtypes = [P(csa_shape), P(csa_params), vp, vp, vp,
                                    vp, vp, vp, vp, P(ctypes.c_int64),
                                    P(ctypes.c_uint64), vp, vp, vp, vp, vp,
                                    vp, sz, vp]
    lib.csa_decode_step.restype = ctypes.c_int
    lib.csa_decode_step_device.argtypes = [P(csa_shape), P(csa_params), vp,
                                           vp, vp, vp, vp, vp, vp, vp, vp,
                                           ctypes.c_int, vp, vp, vp, vp, vp,
                                           vp, sz, vp]
    lib.csa_decode_step_device.restype = ctypes.c_int
    lib.csa_quantize_keys8.argtypes = [P(csa_shape), vp, P(ctypes.c_int64),
                                       ctypes.c_int64, vp, vp, vp]
    lib.csa_quantize_keys8.restype = ctypes.c_int
    lib.csa_decode_step_refined.argtypes = [P(csa_shape), P(csa_params), vp,
                                            vp, vp, vp, vp, vp, vp, vp, vp,
                                            P(ctypes.c_int64),
                                            P(ctypes.c_uint64), vp, vp, vp,
                                            vp, vp, vp, sz, vp]
    lib.csa_decode_step_refined.restype = ctypes.c_int
    lib.csa_dense_decode.argtypes = [P(csa_shape), vp, vp, vp,
                                     P(ctypes.c_int64), vp, vp, sz, vp]
    lib.csa_dense_decode.restype = ctypes.c_int
    lib.csa_dense_decode_static.argtypes = [P(csa_shape), vp, vp, vp,
                                            P(ctypes.c_int64), vp, vp]
    lib.csa_dense_decode_static.restype = ctypes.c_int
    lib.csa_check.argtypes = [vp, vp]
    lib.csa_check.restype = ctypes.c_int
    lib.csa_workspace_layout.argtypes = [P(csa_shape), P(csa_params),
                                         P(csa_workspace_map)]
    lib.csa_workspace_layout.restype = ctypes.c_int
    lib.csa_profile_enable.argtypes = [ctypes.c_int]
    lib.csa_profile_enable.restype = ctypes.c_int
    lib.csa_profile_read.argtypes = [P(csa_phase_times)]
    lib.csa_profile_read.restype = ctypes.c_int
    lib.csa_status_string.argtypes = [ctypes.c_int]
    lib.csa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(s: int) -> str:
    return load_library().csa_status_string(int(s)).decode()


# ------------------------------------------------------------ marshalling

def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _i64(xs: Sequence[int]):
    return (ctypes.c_int64 * len(xs))(*[int(x) for x in xs])


def _u64(xs: Sequence[int]):
    return (ctypes.c_uint64 * len(xs))(*[int(x) & 0xFFFFFFFFFFFFFFFF
                                         for x in xs])


def make_shape(B, Hq, Hkv, d, n_max, dtype) -> csa_shape:
    if not isinstance(dtype, int):
        dtype = CSA_F32 if str(dtype) in ("f32", "float32",
                                          "torch.float32") else CSA_BF16
    return csa_shape(int(B), int(Hq), int(Hkv), int(d), int(n_max), dtype)


def make_params(eps=0.05, delta=0.05, r=2, measure=CSA_MEASURE_VALUE,
                J_override=-1, sub_batches=0, perturb=0,
                qcode=0, refine8=0, dots=0) -> csa_params:
    return csa_params(float(eps), float(delta), int(r), int(measure),
                      int(J_override), int(sub_batches), int(perturb),
                      int(qcode), int(refine8), int(dots))


def csa_workspace_size(shape: csa_shape, params: csa_params) -> int:
    return int(load_library().csa_workspace_size(ctypes.byref(shape),
                                                 ctypes.byref(params)))


def csa_dense_workspace_size(shape: csa_shape) -> int:
    return int(load_library().csa_dense_workspace_size(ctypes.byref(shape)))


def csa_workspace_layout(shape: csa_shape, params: csa_params):
    m = csa_workspace_map()
    check(load_library().csa_workspace_layout(ctypes.byref(shape),
                                              ctypes.byref(params),
                                              ctypes.byref(m)),
          "csa_workspace_layout")
    return m


def decode_ordered(u):
    """Ordered-integer encoding of the maxima (csa_workspace_map.cmax) back
    to float32 values (numpy uint32 array in, float32 array out)."""
    import numpy as np
    u = np.asarray(u, dtype=np.uint32)
    bits = np.where(u >= np.uint32(0x80000000), u & np.uint32(0x7FFFFFFF),
                    ~u).astype(np.uint32)
    return bits.view(np.float32)


def csa_quantize_keys(shape, K, V, lens, from_token, K4, bounds, vmax,
                      vnorm2, stream=None) -> int:
    _check_batch(shape, lens)
    return load_library().csa_quantize_keys(
        ctypes.byref(shape), _ptr(K), _ptr(V), _i64(lens), int(from_token),
        _ptr(K4), _ptr(bounds), _ptr(vmax), _ptr(vnorm2), _stream(stream))


def csa_decode_step(shape, params, q, K, V, K4, bounds, vmax, vnorm2, lens,
                    seeds, o, beta, level, keys_read, stats, workspace,
                    workspace_bytes, stream=None) -> int:
    _check_batch(shape, lens, seeds)
    return load_library().csa_decode_step(
        ctypes.byref(shape), ctypes.byref(params), _ptr(q), _ptr(K), _ptr(V),
        _ptr(K4), _ptr(bounds), _ptr(vmax), _ptr(vnorm2), _i64(lens),
        _u64(seeds), _ptr(o),
        _ptr(beta), _ptr(level), _ptr(keys_read), _ptr(stats),
        _ptr(workspace), int(workspace_bytes), _stream(stream))


def csa_quantize_keys8(shape, K, lens, from_token, K8, delta8,
                       stream=None) -> int:
    _check_batch(shape, lens)
    return load_library().csa_quantize_keys8(
        ctypes.byref(shape), _ptr(K), _i64(lens), int(from_token), _ptr(K8),
        _ptr(delta8), _stream(stream))


def meta8_buffers(shape: csa_shape, device):
    """(K8, delta8) device tensors for csa_quantize_keys8 (the 8-bit tier)."""
    import torch
    nblk = (shape.n_max + BLOCK - 1) // BLOCK
    K8 = torch.zeros((shape.B, shape.Hkv, nblk * BLOCK, shape.d),
                     dtype=torch.uint8, device=device)
    d8 = torch.zeros((shape.B, shape.Hkv, nblk, shape.d), dtype=torch.float32,
                     device=device)
    return K8, d8


def csa_decode_step_refined(shape, params, q, K, V, K4, bounds, vmax, vnorm2,
                            K8, delta8, lens, seeds, o, beta, level,
                            keys_read, stats, workspace, workspace_bytes,
                            stream=None) -> int:
    _check_batch(shape, lens, seeds)
    return load_library().csa_decode_step_refined(
        ctypes.byref(shape), ctypes.byref(params), _ptr(q), _ptr(K), _ptr(V),
        _ptr(K4), _ptr(bounds), _ptr(vmax), _ptr(vnorm2), _ptr(K8),
        _ptr(delta8), _i64(lens), _u64(seeds), _ptr(o), _ptr(beta),
        _ptr(level), _ptr(keys_read), _ptr(stats), _ptr(workspace),
        int(workspace_bytes), _stream(stream))


def csa_decode_step_device(shape, params, q, K, V, K4, bounds, vmax, vnorm2,
                           lens_dev, seeds_dev, requantize_last, o, beta,
                           level, keys_read, stats, workspace,
                           workspace_bytes, stream=None) -> int:
    """lens_dev: device int64 [B]; seeds_dev: device uint64 (or int64) [B]."""
    return load_library().csa_decode_step_device(
        ctypes.byref(shape), ctypes.byref(params), _ptr(q), _ptr(K), _ptr(V),
        _ptr(K4), _ptr(bounds), _ptr(vmax), _ptr(vnorm2), _ptr(lens_dev),
        _ptr(seeds_dev), int(requantize_last), _ptr(o), _ptr(beta),
        _ptr(level), _ptr(keys_read), _ptr(stats), _ptr(workspace),
        int(workspace_bytes), _stream(stream))


def csa_dense_decode(shape, q, K, V, lens, o, workspace, workspace_bytes,
                     stream=None) -> int:
    _check_batch(shape, lens)
    return load_library().csa_dense_decode(
        ctypes.byref(shape), _ptr(q), _ptr(K), _ptr(V), _i64(lens), _ptr(o),
        _ptr(workspace), int(workspace_bytes), _stream(stream))


def csa_dense_decode_static(shape, q, K, V, lens, o, stream=None) -> int:
    _check_batch(shape, lens)
    return load_library().csa_dense_decode_static(
        ctypes.byref(shape), _ptr(q), _ptr(K), _ptr(V), _i64(lens), _ptr(o),
        _stream(stream))


def csa_profile_enable(on: bool) -> int:
    return load_library().csa_profile_enable(1 if on else 0)


def csa_profile_read() -> dict:
    """Accumulated ms per phase since the last read, steps, launches."""
    t = csa_phase_times()
    check(load_library().csa_profile_read(ctypes.byref(t)),
          "csa_profile_read")
    return {"ms": dict(zip(PHASES, list(t.ms))), "steps": int(t.steps),
            "launches": int(t.launches)}


def csa_check(workspace, stream=None) -> int:
    return load_library().csa_check(_ptr(workspace), _stream(stream))


def check(status: int, where: str = "csa") -> None:
    if status != CSA_OK:
        raise CsaError(status, where)


# ---------------------------------------------------- tensor conveniences

class KVMeta(NamedTuple):
    """Device metadata csa_quantize_keys writes and csa_decode_step reads."""
    K4: object
    bounds: object
    vmax: object
    vnorm2: object


def meta_buffers(shape: csa_shape, device) -> KVMeta:
    """Allocate K4, bounds, vmax, vnorm2 (torch, device) for a shape."""
    import torch
    nblk = (shape.n_max + BLOCK - 1) // BLOCK
    K4 = torch.zeros((shape.B, shape.Hkv, nblk * BLOCK, shape.d // 2),
                     dtype=torch.uint8, device=device)
    bounds = torch.zeros((shape.B, shape.Hkv, nblk, 2, shape.d),
                         dtype=torch.float32, device=device)
    vmax = torch.zeros((shape.B, shape.Hkv, nblk), dtype=torch.float32,
                       device=device)
    vnorm2 = torch.zeros((shape.B, shape.Hkv, shape.n_max),
                         dtype=torch.float32, device=device)
    return KVMeta(K4, bounds, vmax, vnorm2)


def _require(t, name: str, nbytes: int) -> None:
    """Refuse a tensor the kernels would read from host memory or past its
    end: it must be a contiguous CUDA tensor of at least ``nbytes``."""
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name}: a CUDA tensor is required")
    if not t.is_contiguous():
        raise ValueError(f"{name}: the tensor must be contiguous")
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name}: {have} bytes, the shape needs {nbytes}")


def _check_batch(shape: csa_shape, lens, seeds=None) -> None:
    if len(lens) != shape.B:
        raise ValueError(f"lens: {len(lens)} entries for B = {shape.B}")
    if seeds is not None and len(seeds) != shape.B:
        raise ValueError(f"seeds: {len(seeds)} entries for B = {shape.B}")


def check_step_inputs(shape: csa_shape, q, K, V, meta=None, lens=(),
                      seeds=None) -> None:
    """Host-side checks of the tensors and host arrays a decode step (or,
    without ``meta``, a dense decode) reads: the layouts of include/csa.h,
    on the device, contiguous and large enough.  Raises ValueError."""
    B, Hq, Hkv, d, n = shape.B, shape.Hq, shape.Hkv, shape.d, shape.n_max
    esz = 4 if shape.dtype == CSA_F32 else 2
    nblk = (n + BLOCK - 1) // BLOCK
    _check_batch(shape, lens, seeds)
    _require(q, "q", B * Hq * d * esz)
    _require(K, "K", B * Hkv * n * d * esz)
    _require(V, "V", B * Hkv * n * d * esz)
    if meta is not None:
        _require(meta.K4, "K4", B * Hkv * nblk * BLOCK * (d // 2))
        _require(meta.bounds, "bounds", B * Hkv * nblk * 2 * d * 4)
        _require(meta.vmax, "vmax", B * Hkv * nblk * 4)
        _require(meta.vnorm2, "vnorm2", B * Hkv * n * 4)


class DecodeStep:
    """Owns the workspace and output buffers of csa_decode_step for one
    shape and parameter set; ``__call__`` runs one step on the current
    stream (asynchronously)."""

    def __init__(self, shape: csa_shape, params: csa_params, device,
                 with_stats: bool = False):
        import torch
        self.shape, self.params = shape, params
        nbytes = csa_workspace_size(shape, params)
        if nbytes == 0:
            raise CsaError(1, "csa_workspace_size")
        self.ws_bytes = nbytes
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        B, Hq, d = shape.B, shape.Hq, shape.d
        # the four outputs are views of one buffer (``outputs``), so that a
        # caller reads a step's results back with a single copy
        nh = B * Hq
        self.outputs = torch.empty((nh * (d + 3),), dtype=torch.float32,
                                   device=device)
        self.o = self.outputs[:nh * d].view(B, Hq, d)
        self.beta = self.outputs[nh * d:nh * (d + 1)].view(B, Hq)
        self.level = self.outputs[nh * (d + 1):nh * (d + 2)].view(
            torch.int32).view(B, Hq)
        self.keys_read = self.outputs[nh * (d + 2):].view(
            torch.int32).view(B, Hq)
        self.stats = (torch.zeros((B, Hq, STATS_FIELDS), dtype=torch.int32,
                                  device=device) if with_stats else None)

    def __call__(self, q, K, V, meta: KVMeta, lens, seeds, stream=None,
                 meta8=None):
        """meta8: (K8, delta8) of the 8-bit tier, required when the
        parameters ask for it (csa_decode_step_refined)."""
        check_step_inputs(self.shape, q, K, V, meta, lens, seeds)
        if self.params.refine8:
            if meta8 is None:
                raise ValueError("refine8: the 8-bit codes (meta8) are needed")
            nblk = (self.shape.n_max + BLOCK - 1) // BLOCK
            n8 = self.shape.B * self.shape.Hkv * nblk
            _require(meta8[0], "K8", n8 * BLOCK * self.shape.d)
            _require(meta8[1], "delta8", n8 * self.shape.d * 4)
            st = csa_decode_step_refined(
                self.shape, self.params, q, K, V, meta.K4, meta.bounds,
                meta.vmax, meta.vnorm2, meta8[0], meta8[1], lens, seeds,
                self.o, self.beta, self.level, self.keys_read, self.stats,
                self.ws, self.ws_bytes, stream)
            check(st, "csa_decode_step_refined")
        else:
            st = csa_decode_step(self.shape, self.params, q, K, V, meta.K4,
                                 meta.bounds, meta.vmax, meta.vnorm2, lens,
                                 seeds, self.o, self.beta, self.level,
                                 self.keys_read, self.stats, self.ws,
                                 self.ws_bytes, stream)
            check(st, "csa_decode_step")
        return self.o, self.beta, self.level, self.keys_read

    def device_step(self, q, K, V, meta: KVMeta, lens_dev, seeds_dev,
                    requantize_last: bool = True, stream=None):
        """The step with lengths and seeds read from device tensors (int64
        [B] each), optionally re-quantising the block of the token just
        appended; capturable into a CUDA graph that is replayed with new
        lengths and seeds written into the same tensors."""
        check_step_inputs(self.shape, q, K, V, meta, [1] * self.shape.B)
        for t, name in ((lens_dev, "lens_dev"), (seeds_dev, "seeds_dev")):
            _require(t, name, 8 * self.shape.B)
        st = csa_decode_step_device(self.shape, self.params, q, K, V,
                                    meta.K4, meta.bounds, meta.vmax,
                                    meta.vnorm2, lens_dev, seeds_dev,
                                    1 if requantize_last else 0, self.o,
                                    self.beta, self.level, self.keys_read,
                                    self.stats, self.ws, self.ws_bytes,
                                    stream)
        check(st, "csa_decode_step_device")
        return self.o, self.beta, self.level, self.keys_read


class DenseDecode:
    """Owns the workspace of csa_dense_decode for one shape."""

    def __init__(self, shape: csa_shape, device):
        import torch
        self.shape = shape
        self.ws_bytes = csa_dense_workspace_size(shape)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8,
                              device=device)
        self.o = torch.empty((shape.B, shape.Hq, shape.d),
                             dtype=torch.float32, device=device)

    def __call__(self, q, K, V, lens, stream=None):
        check_step_inputs(self.shape, q, K, V, None, lens)
        check(csa_dense_decode(self.shape, q, K, V, lens, self.o, self.ws,
                               self.ws_bytes, stream), "csa_dense_decode")
        return self.o
