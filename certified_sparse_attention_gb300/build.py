"""Build the C-ABI shared library libcsa.so for sm_103a, in tree.

    python -m certified_sparse_attention_gb300.build

Each .cu file under csrc/ is compiled by nvcc in parallel (one -gencode:
compute_103a / sm_103a), then linked into certified_sparse_attention_gb300/
_lib/libcsa.so.  No CMake; about a minute on a few cores.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT, "libcsa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"),
                 "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(nvcc, src, obj, extra):
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler",
           "-fPIC", "-I", os.path.join(ROOT, "include"), "-c",
           os.path.join(CSRC, src), "-o", obj, *extra]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(verbose: bool = False, extra=None) -> str:
    nvcc = nvcc_path()
    os.makedirs(OUT, exist_ok=True)
    objs_dir = os.path.join(OUT, "obj")
    os.makedirs(objs_dir, exist_ok=True)
    srcs = sources()
    objs = [os.path.join(objs_dir, s[:-3] + ".o") for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs),
                                                      os.cpu_count() or 1))) as ex:
        futs = [ex.submit(_compile, nvcc, s, o, list(extra or []))
                for s, o in zip(srcs, objs)]
        for f in futs:
            log = f.result()
            if verbose and log:
                print(log, file=sys.stderr)
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv,
                extra=["-Xptxas", "-v"] if "-v" in sys.argv else None))
