"""Builds libasp.so in-tree for sm_103a with nvcc (no CMake, no torch extension).

Each .cu translation unit compiles in parallel; the objects link into
``adaptive_sparse_paged_gb300/libasp.so`` against the shared CUDA runtime,
so a process that already loaded torch's libcudart.so.13 reuses it.

    python -m adaptive_sparse_paged_gb300.build [--verbose]
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG_DIR, "libasp.so")
SOURCES = ["abi.cu", "summarize.cu", "select.cu", "select_cluster.cu", "decode.cu",
           "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libasp.so")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def compile_flags() -> list:
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                   "-I", CSRC, "--expt-relaxed-constexpr"]


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile every kernel source and link libasp.so; returns its path."""
    nvcc = _nvcc()
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, "asp_internal.cuh"), os.path.join(CSRC, "score_common.cuh"),
                   os.path.join(INCLUDE, "asp.h"), os.path.abspath(__file__)]
    if not force and os.path.exists(LIB_PATH):
        built = os.path.getmtime(LIB_PATH)
        if all(os.path.getmtime(d) <= built for d in deps):
            return LIB_PATH
    tmp = tempfile.mkdtemp(prefix="asp_build_")
    try:
        procs = []
        objs = []
        for src in srcs:
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            objs.append(obj)
            cmd = [nvcc, "-c", src, "-o", obj] + compile_flags()
            if verbose:
                cmd.append("-Xptxas=-v")
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
        failed = []
        for src, pr in procs:
            out, _ = pr.communicate()
            if verbose or pr.returncode:
                sys.stdout.write(out)
            if pr.returncode:
                failed.append(src)
        if failed:
            raise RuntimeError("nvcc failed on: " + ", ".join(failed))
        out_tmp = os.path.join(tmp, "libasp.so")
        link = [nvcc, "-shared", "-o", out_tmp] + objs + ARCH + [
            "-cudart", "shared", "-ldl", "-Xlinker", "-rpath," + _cuda_lib_dir(nvcc)]
        if verbose:
            print(" ".join(link), flush=True)
        r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode:
            sys.stdout.write(r.stdout)
            raise RuntimeError("linking libasp.so failed")
        os.replace(out_tmp, LIB_PATH)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv, force="--force" in sys.argv))
