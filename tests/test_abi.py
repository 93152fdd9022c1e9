"""The C-ABI library builds, loads and exports every entry point that
include/csa.h declares; host-side argument checks (no GPU work)."""
import ctypes
import os
import re

import numpy as np
import pytest

import certified_sparse_attention_gb300 as csa
from tests.gpu_common import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "csa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return ensure_built()


def test_every_declared_symbol_exported(lib):
    names = _declared()
    assert "csa_decode_step" in names and "csa_quantize_keys" in names
    for nm in names:
        assert hasattr(lib, nm), nm
    assert set(csa.EXPORTED) == set(names)


def test_workspace_sizes(lib):
    s = csa.make_shape(4, 32, 8, 128, 131072, "bf16")
    p = csa.make_params(0.05, 0.05, 4)
    ws = csa.csa_workspace_size(s, p)
    m = csa.csa_workspace_layout(s, p)
    assert ws == m.total and ws > 0
    assert m.J1 == 69                   # J = ceil(4 log2 131008) = 68
    assert m.ubar % 256 == 0 and m.s32 % 256 == 0
    assert csa.csa_dense_workspace_size(s) > 0
    # two sub-batches of two sequences by default; the regions do not
    # overlap and the unsplit layout fits too
    assert m.sub_batches == 2 and m.sub_B == 2 and m.sub_stride % 256 == 0
    one = csa.make_params(0.05, 0.05, 4, sub_batches=1)
    m1 = csa.csa_workspace_layout(s, one)
    assert m1.sub_batches == 1 and m1.sub_B == 4
    assert m.total >= max(2 * m.sub_stride, m1.total)
    assert m.sub_stride < m1.total
    # one sequence: nothing to split; an uneven split rounds up
    s1 = csa.make_shape(1, 32, 8, 128, 4096, "bf16")
    assert csa.csa_workspace_layout(s1, p).sub_batches == 1
    s3 = csa.make_shape(3, 32, 8, 128, 4096, "bf16")
    m3 = csa.csa_workspace_layout(s3, csa.make_params(sub_batches=3))
    assert m3.sub_batches == 3 and m3.sub_B == 1


@pytest.mark.parametrize("bad", [
    dict(d=96), dict(Hq=12, Hkv=8), dict(Hq=48, Hkv=3), dict(B=129)])
def test_unsupported_shapes(lib, bad):
    kw = dict(B=1, Hq=32, Hkv=8, d=128, n_max=4096, dtype="bf16")
    kw.update(bad)
    s = csa.make_shape(**kw)
    assert csa.csa_workspace_size(s, csa.make_params()) == 0


@pytest.mark.parametrize("pk", [dict(eps=0.0), dict(delta=1.0),
                                dict(delta=0.0), dict(r=0), dict(r=5),
                                dict(measure=4), dict(J_override=300),
                                dict(sub_batches=5), dict(sub_batches=-1),
                                dict(perturb=2), dict(qcode=2)])
def test_invalid_params(lib, pk):
    s = csa.make_shape(1, 8, 2, 128, 4096, "bf16")
    kw = dict(eps=0.05, delta=0.05, r=2)
    kw.update(pk)
    assert csa.csa_workspace_size(s, csa.make_params(**kw)) == 0


def test_decode_rejects_bad_arguments_before_launch(lib):
    s = csa.make_shape(1, 8, 2, 128, 4096, "bf16")
    p = csa.make_params()
    # null inputs, bad lengths, missing workspace: rejected on the host,
    # nothing is launched (these calls run without a GPU)
    st = lib.csa_decode_step(ctypes.byref(s), ctypes.byref(p), None, None,
                             None, None, None, None, None,
                             (ctypes.c_int64 * 1)(100),
                             (ctypes.c_uint64 * 1)(1), None, None, None,
                             None, None, None, 0, None)
    assert st == 1
    fake = 256
    st = lib.csa_decode_step(ctypes.byref(s), ctypes.byref(p), fake, fake,
                             fake, fake, fake, fake, fake,
                             (ctypes.c_int64 * 1)(5000),
                             (ctypes.c_uint64 * 1)(1), fake, fake, fake,
                             fake, None, fake, 1 << 30, None)
    assert st == 1                       # len > n_max
    st = lib.csa_decode_step(ctypes.byref(s), ctypes.byref(p), fake, fake,
                             fake, fake, fake, fake, fake,
                             (ctypes.c_int64 * 1)(100),
                             (ctypes.c_uint64 * 1)(1), fake, fake, fake,
                             fake, None, fake, 16, None)
    assert st == 6                       # workspace too small
    assert csa.status_string(6).startswith("workspace")


def test_device_length_step_rejects_bad_arguments_before_launch(lib):
    # the device-length variant: the same host checks (its lengths are on
    # the device and checked there), plus the re-quantisation flag
    s = csa.make_shape(1, 8, 2, 128, 4096, "bf16")
    p = csa.make_params()
    fake = 256
    f = lib.csa_decode_step_device
    assert f(ctypes.byref(s), ctypes.byref(p), fake, fake, fake, fake, fake,
             fake, fake, None, fake, 1, fake, fake, fake, fake, None, fake,
             1 << 30, None) == 1                     # no length array
    assert f(ctypes.byref(s), ctypes.byref(p), fake, fake, fake, fake, fake,
             fake, fake, fake, fake, 2, fake, fake, fake, fake, None, fake,
             1 << 30, None) == 1                     # flag not 0 or 1
    assert f(ctypes.byref(s), ctypes.byref(p), fake, fake, fake, fake, fake,
             fake, fake, fake, fake, 1, fake, fake, fake, fake, None, fake,
             16, None) == 6                          # workspace too small


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(csa.CsaLibraryMissing):
        csa._lib_save = csa._lib
        csa._lib = None
        try:
            csa.load_library(str(tmp_path / "nope.so"))
        finally:
            csa._lib = csa._lib_save


def test_plain_c_caller_builds(lib, tmp_path):
    # the boundary needs no PyTorch: a plain C program (CUDA runtime for
    # device memory only) compiles and links against libcsa.so; it runs a
    # quantise + decode step on a GPU
    import shutil
    import subprocess
    cc = shutil.which("cc") or shutil.which("gcc")
    cuda = "/usr/local/cuda"
    if not cc or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime_api.h")):
        pytest.skip("no C compiler or CUDA headers")
    libdir = os.path.dirname(csa.LIB_PATH)
    cudalib = next((os.path.join(cuda, p) for p in ("lib64", "lib", "targets/sbsa-linux/lib")
                    if os.path.exists(os.path.join(cuda, p, "libcudart.so"))), None)
    if cudalib is None:
        pytest.skip("no libcudart.so")
    out = tmp_path / "decode_example"
    cmd = [cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c", "decode_example.c"),
           "-L", libdir, "-lcsa", "-L", cudalib, "-lcudart", "-lm", "-o", str(out)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    assert out.exists()


def test_binding_structs_match_the_header(tmp_path):
    # the ctypes mirrors of the header's structs have the C compiler's size
    # and field offsets (a plain C program built against include/csa.h
    # prints them; a field the binding lacks would change the size or an
    # offset), and the phase names match CSA_NPHASE
    import shutil
    import subprocess
    cc = shutil.which("cc") or shutil.which("gcc")
    if not cc:
        pytest.skip("no C compiler")
    structs = (csa.csa_shape, csa.csa_params, csa.csa_head_stats,
               csa.csa_workspace_map, csa.csa_phase_times)
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "csa.h"',
             "int main(void) {"]
    for st in structs:
        nm = st.__name__
        lines.append(f'  printf("{nm} sizeof %zu\\n", sizeof({nm}));')
        for f, _ in st._fields_:
            lines.append(f'  printf("{nm} {f} %zu\\n", offsetof({nm}, {f}));')
    lines += ['  printf("CSA_NPHASE value %d\\n", CSA_NPHASE);', "  return 0;",
              "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = {}
    for ln in subprocess.run([str(exe)], capture_output=True, text=True,
                             check=True).stdout.split("\n"):
        if ln:
            a, b, c = ln.split()
            got[(a, b)] = int(c)
    for st in structs:
        nm = st.__name__
        assert got[(nm, "sizeof")] == ctypes.sizeof(st), nm
        for f, _ in st._fields_:
            assert got[(nm, f)] == getattr(st, f).offset, (nm, f)
    assert len(csa.PHASES) == got[("CSA_NPHASE", "value")]
    assert ctypes.sizeof(csa.csa_phase_times._fields_[0][1]) == \
        4 * len(csa.PHASES)


def test_workspace_layout_properties(lib):
    # over many shapes and parameters: the documented arrays lie inside
    # their sub-batch region, 256-byte aligned and disjoint; the regions
    # fit in the reported size; the sub-batches cover the batch; J1 is the
    # grid of the longest sequence
    from oracle.step import grid_J
    rng = np.random.default_rng(11)
    for _ in range(300):
        G = int(rng.choice([1, 2, 4, 8]))
        Hkv = int(rng.integers(1, 9))
        d = int(rng.choice([64, 128]))
        B = int(rng.choice([1, 2, 3, 4, 7, 32, 128]))
        n = int(rng.choice([1, 63, 64, 65, 100, 1000, 4096, 131072, 1 << 20]))
        r = int(rng.integers(1, 5))
        p = csa.make_params(0.05, 0.05, r, int(rng.integers(0, 4)), -1,
                            int(rng.integers(0, 5)), int(rng.integers(0, 2)))
        s = csa.make_shape(B, G * Hkv, Hkv, d, n, "bf16")
        m = csa.csa_workspace_layout(s, p)
        assert csa.csa_workspace_size(s, p) == m.total > 0
        assert 1 <= m.sub_batches <= 4 and m.sub_B >= 1
        assert m.sub_B * m.sub_batches >= B > (m.sub_batches - 1) * m.sub_B
        region = m.sub_stride if m.sub_batches > 1 else m.total
        assert m.sub_batches * m.sub_stride <= m.total or m.sub_batches == 1
        assert m.J1 == grid_J(max(n - 64, 0), r) + 1
        Bs, Hq = m.sub_B, G * Hkv
        pcap = max(n - 64, 1)
        arrays = [(m.ubar, Bs * Hkv * n * G * 4), (m.cmax, Bs * Hq * 16),
                  (m.s32, Bs * Hkv * pcap * G * 4),
                  (m.jr_hist, Bs * Hq * (m.J1 + 1) * 4),
                  (m.bcnt, Bs * Hkv * m.J1 * 4)]
        for off, size in arrays:
            assert off % 256 == 0 and off + size <= region, (off, size, region)
        arrays.sort()
        for (o1, s1), (o2, _) in zip(arrays, arrays[1:]):
            assert o1 + s1 <= o2


class _FakeDev:
    """Stands in for a CUDA tensor in host-only checks."""

    def __init__(self, nbytes, esz=2, contiguous=True, cuda=True):
        self.n, self.esz = nbytes // esz, esz
        self.contig, self.is_cuda = contiguous, cuda

    def numel(self):
        return self.n

    def element_size(self):
        return self.esz

    def is_contiguous(self):
        return self.contig


def test_step_inputs_checked_before_the_call():
    # the tensor wrappers refuse what the kernels would read past its end or
    # from host memory, and host arrays of the wrong length, before calling
    # the library
    B, Hq, Hkv, d, n = 2, 8, 2, 128, 1000
    s = csa.make_shape(B, Hq, Hkv, d, n, "bf16")
    nblk = (n + 63) // 64
    ok = dict(q=_FakeDev(B * Hq * d * 2), K=_FakeDev(B * Hkv * n * d * 2),
              V=_FakeDev(B * Hkv * n * d * 2))
    meta = csa.KVMeta(_FakeDev(B * Hkv * nblk * 64 * d // 2, 1),
                      _FakeDev(B * Hkv * nblk * 2 * d * 4, 4),
                      _FakeDev(B * Hkv * nblk * 4, 4),
                      _FakeDev(B * Hkv * n * 4, 4))
    csa.check_step_inputs(s, ok["q"], ok["K"], ok["V"], meta, [n, n], [1, 2])
    csa.check_step_inputs(s, ok["q"], ok["K"], ok["V"], None, [n, n])
    bad = [
        dict(lens=[n]),                                   # one length short
        dict(seeds=[1, 2, 3]),
        dict(K=_FakeDev(B * Hkv * n * d * 2 - 2)),        # one element short
        dict(q=_FakeDev(B * Hq * d * 2, contiguous=False)),
        dict(V=_FakeDev(B * Hkv * n * d * 2, cuda=False)),
        dict(meta=meta._replace(vnorm2=_FakeDev(B * Hkv * n * 2, 4))),
    ]
    for over in bad:
        args = dict(q=ok["q"], K=ok["K"], V=ok["V"], meta=meta, lens=[n, n],
                    seeds=[1, 2])
        args.update(over)
        with pytest.raises(ValueError):
            csa.check_step_inputs(s, **args)
    # an f32 shape needs four bytes per element: bf16-sized tensors fail
    s32 = csa.make_shape(B, Hq, Hkv, d, n, "f32")
    with pytest.raises(ValueError):
        csa.check_step_inputs(s32, ok["q"], ok["K"], ok["V"], None, [n, n])
    # a host tensor is refused
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        csa.check_step_inputs(s, torch.zeros(B, Hq, d, dtype=torch.bfloat16),
                              ok["K"], ok["V"], None, [n, n])


def test_host_arrays_checked_in_the_low_level_wrappers(lib):
    # lens / seeds with other than B entries would make the library read
    # past a host array: the wrappers refuse them before the call
    s = csa.make_shape(2, 8, 2, 128, 4096, "bf16")
    p = csa.make_params()
    with pytest.raises(ValueError):
        csa.csa_quantize_keys(s, 1, 1, [100], 0, 1, 1, 1, 1, stream=0)
    with pytest.raises(ValueError):
        csa.csa_decode_step(s, p, 1, 1, 1, 1, 1, 1, 1, [100, 100], [1],
                            1, 1, 1, 1, None, 1, 1 << 20, stream=0)
    with pytest.raises(ValueError):
        csa.csa_dense_decode(s, 1, 1, 1, [1, 2, 3], 1, 1, 1 << 20, stream=0)
    with pytest.raises(ValueError):
        csa.csa_dense_decode_static(s, 1, 1, 1, [1], 1, stream=0)
