"""Build the in-tree CUDA libraries for sm_103a (B300).

    python -m sub_bit_weight_binary_b300.build [--force] [--verbose-ptxas]

libbonsai.so        the C ABI of include/bonsai.h (kernels + host checks)
libbonsai_synth.so  the device twin of the seeded input generator
Both land next to this file; nvcc cross-compiles without a GPU.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                  "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]

LIBS = {
    "libbonsai.so": ["api.cu", "pack.cu", "gemv.cu", "gemv_lut.cu", "gemm.cu", "xnor.cu", "xnor_tc.cu", "splitk.cu", "rotate.cu", "stage.cu", "selftest.cu"],
    "libbonsai_synth.so": ["synth.cu"],
}
HEADERS = ["common.cuh", "tcgen05.cuh"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, verbose_ptxas: bool) -> str:
    cmd = [nvcc()] + NVFLAGS + (["-Xptxas", "-v"] if verbose_ptxas else []) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return r.stderr


def build(force: bool = False, verbose_ptxas: bool = False) -> list[str]:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [
        os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    jobs = []
    for lib, srcs in LIBS.items():
        for s in srcs:
            src = os.path.join(CSRC, s)
            obj = os.path.join(BUILD, s.replace(".cu", ".o"))
            if force or _stale(obj, [src] + headers):
                jobs.append((src, obj))
    logs = []
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
            for log in ex.map(lambda j: _compile(j[0], j[1], verbose_ptxas), jobs):
                logs.append(log)
    out = []
    for lib, srcs in LIBS.items():
        target = os.path.join(HERE, lib)
        objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in srcs]
        if force or _stale(target, objs):
            tmp = target + ".tmp%d" % os.getpid()
            cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("link failed for %s:\n%s\n%s" % (lib, r.stdout, r.stderr))
            os.replace(tmp, target)
        out.append(target)
    if verbose_ptxas:
        for log in logs:
            sys.stderr.write(log)
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args()
    for p in build(a.force, a.verbose_ptxas):
        print(p)
