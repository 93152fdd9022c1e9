"""The boundary from plain C on a GPU: `tests/c/decode_example.c` (no
PyTorch, the CUDA runtime for device memory only) is compiled against
include/csa.h and libcsa.so and run.  It quantises 4096 random bf16 keys and
values, runs one certified decode step through `csa_decode_step`, checks the
device status word and reads o, beta, the stop level and keys_read back; it
exits 0 when every output is finite and in range and prints one line per
query head.
"""
import os
import re
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu


def test_plain_c_caller_runs(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests.gpu_common import ensure_built
    import certified_sparse_attention_gb300 as csa
    ensure_built()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cc = shutil.which("cc") or shutil.which("gcc")
    cuda = "/usr/local/cuda"
    if not cc or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime_api.h")):
        pytest.skip("no C compiler or CUDA headers")
    cudalib = next((os.path.join(cuda, p) for p in ("lib64", "lib", "targets/sbsa-linux/lib",
                                                     "targets/x86_64-linux/lib")
                    if os.path.exists(os.path.join(cuda, p, "libcudart.so"))), None)
    if cudalib is None:
        pytest.skip("no libcudart.so")
    libdir = os.path.dirname(csa.LIB_PATH)
    exe = tmp_path / "decode_example"
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                        "-I", os.path.join(cuda, "include"),
                        os.path.join(root, "tests", "c", "decode_example.c"),
                        "-L", libdir, "-lcsa", "-L", cudalib, "-lcudart", "-lm", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = os.pathsep.join([libdir, cudalib, env.get("LD_LIBRARY_PATH", "")])
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    lines = [l for l in r.stdout.splitlines() if l.startswith("head ")]
    assert len(lines) == 4, r.stdout
    for h, l in enumerate(lines):
        m = re.match(r"head (\d+): level (\d+) beta (\S+) keys_read (\d+)", l)
        assert m and int(m.group(1)) == h, l
        assert 64 <= int(m.group(4)) <= 4096
