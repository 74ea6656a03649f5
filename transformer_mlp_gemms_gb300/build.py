"""Build the in-tree shared library ``_build/libkt_mlp.so`` with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked with ``nvcc -shared``.
The CUDA runtime is linked statically; the driver's tensor-map encoder is looked
up at run time, so the library has no link-time dependency on libcuda.

    python -m transformer_mlp_gemms_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libkt_mlp.so")

SOURCES = ["kt_gemm_act.cu", "kt_gemm_geglu.cu", "kt_gemm_down.cu", "kt_mlp_two_act_f16.cu", "kt_mlp_two_act_bf16.cu",
           "kt_mlp_two_geglu.cu", "kt_fused.cu", "kt_mlp_kernels.cu", "kt_mlp_abi.cpp", "kt_planner.cpp"]
HEADERS = [os.path.join(CSRC, "kt_internal.h"), os.path.join(CSRC, "kt_gemm.cuh"), os.path.join(INCLUDE, "kt_mlp.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def _flags(src: str):
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if src.endswith(".cu"):
        return ARCH + ["-lineinfo", "--expt-relaxed-constexpr"] + common
    return common


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    objs, procs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + HEADERS):
            cmd = [cc, "-c", path, "-o", obj] + _flags(src)
            if ptxas_info and src.endswith(".cu"):
                cmd += ["-Xptxas", "-v"]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0 or verbose or ptxas_info:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {', '.join(failed)}")
    if force or procs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [cc, "-shared", "-o", tmp] + ARCH + objs + ["-lrt", "-lpthread", "-ldl"]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print -Xptxas -v register / smem usage")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info))


if __name__ == "__main__":
    main()
