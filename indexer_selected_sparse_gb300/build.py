"""Build libqsa.so in-tree: one nvcc per translation unit, in parallel, for
sm_103a only, then a shared-library link against the CUDA runtime."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libqsa.so")
SOURCES = ["qsa_api.cu", "qsa_append.cu", "qsa_score.cu", "qsa_select.cu", "qsa_attn.cu",
           "qsa_static.cu", "qsa_score_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqsa")


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if p.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + p.stdout)
    return p.stdout


def build_library(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    flags = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
             "-I", os.path.join(ROOT, "include")] + ARCH
    if ptxas_info:
        flags += ["-Xptxas", "-v"]
    objs = []
    jobs = []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        jobs.append([cc, "-c", os.path.join(CSRC, src), "-o", obj] + flags)
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(_run, jobs))
    if verbose or ptxas_info:
        for log in logs:
            sys.stdout.write(log)
    _run([cc, "-shared", "-o", LIB] + objs + ARCH + ["-lcudart"])
    return LIB


if __name__ == "__main__":
    print(build_library(verbose=True, ptxas_info="-v" in sys.argv))
