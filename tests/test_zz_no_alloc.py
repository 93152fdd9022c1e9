"""csa_dense_decode_static: dense decode with its split-K partials in the
library's fixed device array.  It must give exactly what csa_dense_decode
gives (the same kernels run), on consecutive calls that reuse the array with
different shapes and lengths, and must refuse shapes whose partials do not
fit.  The file name keeps it last in collection order, so it also runs after
every other GPU test in the same process."""
import numpy as np
import pytest

import certified_sparse_attention_gb300 as csa
from tests.gpu_common import ensure_built


@pytest.fixture(scope="module")
def lib():
    return ensure_built()


def test_oversize_shape_rejected(lib):
    # B=4, Hq=32, d=128 at n_max=262144: 256 splits x 128 heads x 130 floats
    # = 17,039,360 bytes > 16 MiB
    s = csa.make_shape(4, 32, 8, 128, 262144, "bf16")
    assert csa.csa_dense_workspace_size(s) > csa.DENSE_STATIC_SCRATCH_BYTES
    lens = [262144] * 4
    st = csa.csa_dense_decode_static(s, 1, 1, 1, lens, 1, stream=0)
    assert st == 6, csa.csa_status_string(st)          # CSA_ERR_WORKSPACE
    # the largest fitting length for this head count is accepted by the check
    s2 = csa.make_shape(4, 32, 8, 128, 258048, "bf16")
    assert csa.csa_dense_workspace_size(s2) <= csa.DENSE_STATIC_SCRATCH_BYTES


def test_invalid_arguments_rejected(lib):
    s = csa.make_shape(1, 8, 2, 128, 4096, "bf16")
    assert csa.csa_dense_decode_static(s, None, 1, 1, [4096], 1,
                                       stream=0) == 1
    assert csa.csa_dense_decode_static(s, 1, 1, 1, [0], 1, stream=0) == 1
    assert csa.csa_dense_decode_static(s, 1, 1, 1, [4097], 1, stream=0) == 1
    s3 = csa.make_shape(1, 8, 2, 96, 4096, "bf16")
    assert csa.csa_dense_decode_static(s3, 1, 1, 1, [4096], 1,
                                       stream=0) == 2


def _inputs(B, Hq, Hkv, d, n_max, dtype, seed, device):
    import torch
    g = torch.Generator().manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.randn(B, Hq, d, generator=g)
    K = torch.randn(B, Hkv, n_max, d, generator=g) + 0.5 * torch.randn(
        1, Hkv, 1, d, generator=g)
    V = torch.randn(B, Hkv, n_max, d, generator=g)
    return [x.to(tdt).to(device) for x in (q, K, V)]


@pytest.mark.gpu
def test_matches_workspace_entry_point_on_consecutive_calls(lib):
    import torch
    dev = torch.device("cuda:0")
    cases = [
        # longer first, so the second call finds stale partials of more
        # splits in the array than it writes itself
        dict(B=2, Hq=32, Hkv=8, d=128, n_max=5000, dtype="bf16",
             lens=[5000, 3100], seed=11),
        dict(B=3, Hq=8, Hkv=2, d=64, n_max=2100, dtype="f32",
             lens=[700, 2049, 1], seed=12),
    ]
    for c in cases:
        s = csa.make_shape(c["B"], c["Hq"], c["Hkv"], c["d"], c["n_max"],
                           c["dtype"])
        q, K, V = _inputs(c["B"], c["Hq"], c["Hkv"], c["d"], c["n_max"],
                          c["dtype"], c["seed"], dev)
        ref = csa.DenseDecode(s, dev)(q, K, V, c["lens"]).clone()
        o = torch.full((c["B"], c["Hq"], c["d"]), float("nan"),
                       dtype=torch.float32, device=dev)
        csa.check(csa.csa_dense_decode_static(s, q, K, V, c["lens"], o),
                  "csa_dense_decode_static")
        torch.cuda.synchronize()
        assert torch.isfinite(o).all()
        assert torch.equal(o, ref)
        # and against the definition, in float64 on the host
        qf = q.double().cpu().numpy()
        Kf = K.double().cpu().numpy()
        Vf = V.double().cpu().numpy()
        G = c["Hq"] // c["Hkv"]
        oh = o.cpu().numpy()
        for b, n in enumerate(c["lens"]):
            for h in range(c["Hq"]):
                s_ = Kf[b, h // G, :n] @ qf[b, h] / np.sqrt(c["d"])
                w = np.exp(s_ - s_.max())
                exact = w @ Vf[b, h // G, :n] / w.sum()
                np.testing.assert_allclose(oh[b, h], exact, rtol=0,
                                           atol=2e-5 * (1 + np.abs(exact).max()))


# A device reset ends the CUDA context, and with it the module that holds the
# scratch array; the array's device address in the next context may differ.
# The entry point caches the address per context, so a call after a reset
# must look it up again rather than write through the old address.  The
# check runs in a child process that holds device memory through the CUDA
# runtime alone (a reset would leave this process's torch allocations dead).
_RESET_CHILD = r'''
import ctypes, math, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import certified_sparse_attention_gb300 as csa
csa.load_library()
path = next(l.split()[-1] for l in open("/proc/self/maps")
            if "libcudart.so" in l)
rt = ctypes.CDLL(path)
rt.cudaMalloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t]
rt.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                          ctypes.c_int]
rt.cudaFree.argtypes = [ctypes.c_void_p]

def ok(e, what):
    if e != 0:
        raise SystemExit(f"{what}: cuda error {e}")

def bf16_bits(x):
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

def upload(a):
    p = ctypes.c_void_p()
    ok(rt.cudaMalloc(ctypes.byref(p), a.nbytes), "cudaMalloc")
    ok(rt.cudaMemcpy(p, a.ctypes.data, a.nbytes, 1), "H2D")
    return p.value

def download(p, shape):
    a = np.empty(shape, np.float32)
    ok(rt.cudaMemcpy(a.ctypes.data, p, a.nbytes, 2), "D2H")
    return a

B, Hq, Hkv, d, n = 2, 8, 2, 128, 3000
lens = [3000, 1777]
rng = np.random.default_rng(5)
qb = bf16_bits(rng.normal(0, 1, (B, Hq, d)))
Kb = bf16_bits(rng.normal(0, 1, (B, Hkv, n, d)) + 0.5)
Vb = bf16_bits(rng.normal(0, 1, (B, Hkv, n, d)))
shape = csa.make_shape(B, Hq, Hkv, d, n, "bf16")

def run_static():
    q, K, V = upload(qb), upload(Kb), upload(Vb)
    o = upload(np.full((B, Hq, d), np.nan, np.float32))
    csa.check(csa.csa_dense_decode_static(shape, q, K, V, lens, o, stream=0),
              "static")
    ok(rt.cudaDeviceSynchronize(), "sync")
    out = download(o, (B, Hq, d))
    for p in (q, K, V, o):
        ok(rt.cudaFree(p), "cudaFree")
    return out

def run_workspace():
    q, K, V = upload(qb), upload(Kb), upload(Vb)
    o = upload(np.zeros((B, Hq, d), np.float32))
    nb = csa.csa_dense_workspace_size(shape)
    ws = upload(np.zeros(nb, np.uint8))
    csa.check(csa.csa_dense_decode(shape, q, K, V, lens, o, ws, nb, stream=0),
              "workspace")
    ok(rt.cudaDeviceSynchronize(), "sync")
    out = download(o, (B, Hq, d))
    for p in (q, K, V, o, ws):
        ok(rt.cudaFree(p), "cudaFree")
    return out

before = run_static()
ref = run_workspace()
assert np.array_equal(before, ref)
ok(rt.cudaDeviceReset(), "cudaDeviceReset")
after1 = run_static()
after2 = run_static()
assert np.array_equal(after1, ref) and np.array_equal(after2, ref)
f = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
q64, K64, V64 = f(qb), f(Kb), f(Vb)
G = Hq // Hkv
for b in range(B):
    for h in range(Hq):
        s = K64[b, h // G, :lens[b]] @ q64[b, h] / math.sqrt(d)
        w = np.exp(s - s.max())
        exact = w @ V64[b, h // G, :lens[b]] / w.sum()
        assert np.allclose(after1[b, h], exact, rtol=0, atol=2e-5 * (1 + np.abs(exact).max()))
print("reset ok")
'''


@pytest.mark.gpu
def test_lookup_again_after_device_reset(lib):
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _RESET_CHILD, root],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "reset ok" in r.stdout
