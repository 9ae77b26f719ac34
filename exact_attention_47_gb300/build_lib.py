"""Build the in-tree CUDA library ``lib/libattn47_sm103.so`` with nvcc.

Every translation unit is compiled for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``), in parallel, then linked into
one shared object with the CUDA runtime linked statically, so that the
library loads on a machine without a GPU (e.g. to check its exported
symbols) and needs only the driver at run time.

Usage: ``python -m exact_attention_47_gb300.build_lib`` or ``build()``.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_NAME = "libattn47_sm103.so"
LIB_PATH = os.path.join(LIB_DIR, LIB_NAME)

SOURCES = ["api.cu", "fwd_sm103.cu", "bwd_sm103.cu", "decode_sm103.cu", "kv_append_sm103.cu", "fusion_sm103.cu", "gemm_sm103.cu", "ssd_sm103.cu"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = GENCODE + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                    "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    exe = shutil.which("nvcc")
    if exe is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return exe


def _run(cmd):
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if proc.returncode != 0:
        raise RuntimeError("command failed (%d): %s\n%s" % (proc.returncode, " ".join(cmd), proc.stdout))
    return proc.stdout


def _stale(obj, src):
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(INCLUDE, "attn47.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose=False, ptxas_info=False):
    """Compile (only what changed) and link; returns the library path."""
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        if ptxas_info or _stale(o, s):
            cmd = [nvcc] + CFLAGS + (["-Xptxas", "-v"] if ptxas_info else []) + ["-c", s, "-o", o]
            jobs.append(cmd)
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        outs = list(ex.map(_run, jobs))
    if verbose or ptxas_info:
        for out in outs:
            sys.stdout.write(out)
    objs = [os.path.join(BUILD_DIR, s.replace(".cu", ".o")) for s in SOURCES]
    if jobs or not os.path.exists(LIB_PATH):
        tmp = LIB_PATH + ".tmp"
        _run([nvcc] + GENCODE + ["-shared", "-cudart", "static", "-o", tmp] + objs)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))
