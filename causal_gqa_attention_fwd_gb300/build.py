"""Build libgqa_attn.so in-tree with nvcc for sm_103a.

Each .cu translation unit is compiled in parallel into _build/, then linked
into causal_gqa_attention_fwd_gb300/libgqa_attn.so with the CUDA runtime
linked statically (the library does not need libcuda at load time; the
driver's tensor-map encoder is fetched at run time).
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgqa_attn.so")
DEBUG_LIB = os.path.join(PKG, "libgqa_attn_debug.so")

SOURCES = ["api.cu", "attn_fwd.cu", "attn_bwd.cu", "attn_bwd_split.cu", "attn_decode.cu"]
HEADERS = ["sm103.cuh", "kernels.h", "tmap.h", "rope.h", "bwd_common.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I" + INCLUDE, "-I" + CSRC,
]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Build the library (debug=True: the -DGQA_DEBUG variant with bounds checks in the kernels,
    libgqa_attn_debug.so, objects in _build/debug)."""
    build_dir = os.path.join(BUILD, "debug") if debug else BUILD
    lib_path = DEBUG_LIB if debug else LIB
    if debug:
        extra_flags = (*extra_flags, "-DGQA_DEBUG")
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "gqa_attn.h")]
    objs, procs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stdout.write(out.decode())
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    if force or procs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp%d" % os.getpid()
        cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "static",
               "-Xcompiler", "-fPIC", *objs, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv)
