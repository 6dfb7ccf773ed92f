"""Build libhswa.so in-tree for GB300 (sm_103a) with nvcc.

Each translation unit is compiled in parallel; the shared library links
the CUDA runtime dynamically. The result goes to ``_build/libhswa.so`` next
to this file and is rebuilt only when a source, header or flag changes.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libhswa.so")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")

SOURCES = ["runtime.cu", "decode.cu", "prefill.cu", "copy.cu", "pool.cpp", "tree.cpp"]
HEADERS = ["common.cuh", "internal.h", "kernels.h", "tc.cuh"]

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
    "--expt-relaxed-constexpr",
    "-I" + INCLUDE, "-I" + CSRC,
]


def _stamp(extra):
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(INCLUDE, "hswa.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(FLAGS + extra).encode())
    return h.hexdigest()


def _compile(src, extra):
    obj = os.path.join(OUT_DIR, os.path.basename(src) + ".o")
    cmd = [NVCC] + FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
    return obj, r.stderr


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link libhswa.so; returns its path."""
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    os.makedirs(OUT_DIR, exist_ok=True)
    stamp_file = os.path.join(OUT_DIR, "stamp")
    stamp = _stamp(extra)
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return LIB
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    if verbose or ptxas_info:
        for (obj, log) in results:
            if log.strip():
                sys.stderr.write(log)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [NVCC, "-shared", "-cudart", "shared", "-gencode", "arch=compute_103a,code=sm_103a",
           "-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64"),
           "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
