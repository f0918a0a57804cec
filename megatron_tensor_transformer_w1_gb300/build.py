"""Build libtpffn.so (the C-ABI CUDA library) in-tree, for sm_103a only.

Each translation unit is compiled by its own nvcc process, in parallel, then
linked into ``megatron_tensor_transformer_w1_gb300/libtpffn.so`` with the CUDA
runtime linked statically.  Object files go to ``_build/`` at the repository
root.  Rebuilds only what changed (by modification time).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", platform.machine()  # objects never cross architectures
                     + ("-" + "-".join(x.strip("-").replace("=", "_") for x in os.environ.get("TPFFN_NVCC_EXTRA", "").split())
                        if os.environ.get("TPFFN_NVCC_EXTRA") else ""))
LIB = os.path.join(PKG, "libtpffn.so")
SOURCES = ["tp_gemm_tc.cu", "tp_attention.cu", "tp_kernels.cu", "tp_api.cu", "tp_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]
# extra nvcc flags (e.g. -DTPFFN_INSTRUMENT for per-CTA wait counters); part of the build stamp
EXTRA = os.environ.get("TPFFN_NVCC_EXTRA", "").split()


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _deps_mtime():
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return max(os.path.getmtime(p) for p in paths)


def _compile(src, verbose):
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= _deps_mtime():
        return obj
    cmd = [_nvcc(), *ARCH, *FLAGS, *EXTRA, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    if force:
        for f in os.listdir(BUILD):
            if f.endswith(".o"):
                os.remove(os.path.join(BUILD, f))
    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    stamp = os.path.join(BUILD, "libtpffn.stamp")
    fresh = (os.path.exists(LIB) and os.path.exists(stamp)
             and open(stamp).read() == f"{platform.machine()} {os.path.getmtime(LIB)}"
             and os.path.getmtime(LIB) >= max(os.path.getmtime(o) for o in objs))
    if not fresh:
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, LIB)
        with open(stamp, "w") as fh:
            fh.write(f"{platform.machine()} {os.path.getmtime(LIB)}")
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="--force" in sys.argv))
