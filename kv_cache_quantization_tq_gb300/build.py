"""Build libtq.so in place (nvcc for sm_103a + the host C++ glue).

Usage: python -m kv_cache_quantization_tq_gb300.build   (or build() from Python)

Each translation unit is compiled in its own process, in parallel, then
linked with nvcc into ``kv_cache_quantization_tq_gb300/libtq.so``.  Object
files go to ``kv_cache_quantization_tq_gb300/_build/``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtq.so")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")

CU = ["encode.cu", "decode.cu", "decode_tc.cu", "decode_hy.cu", "decode_alt.cu", "decode_static.cu", "dequant.cu", "pack.cu"]
CPP = ["host.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources_newer(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "tq.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps)


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if needed) and return the path of libtq.so."""
    if not force and not _sources_newer(LIB):
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC]
    jobs = []
    for f in CU:
        obj = os.path.join(BUILD, f + ".o")
        jobs.append([nvcc, *ARCH, "-lineinfo", *common, "-Xcompiler", "-fPIC", "-Xptxas", "-v" if verbose else "-O3",
                     "-c", os.path.join(CSRC, f), "-o", obj])
    for f in CPP:
        obj = os.path.join(BUILD, f + ".o")
        jobs.append([nvcc, *common, "-Xcompiler", "-fPIC", "-c", os.path.join(CSRC, f), "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        outs = list(ex.map(_run, jobs))
    if verbose:
        for o in outs:
            sys.stdout.write(o)
    objs = [os.path.join(BUILD, f + ".o") for f in CU + CPP]
    tmp = LIB + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
