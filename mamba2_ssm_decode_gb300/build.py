"""Build the CUDA library libssu_gb300.so in-tree (sm_103a only).

Each translation unit under csrc/ is compiled by nvcc in parallel into
_build/, then linked into mamba2_ssm_decode_gb300/libssu_gb300.so.  No cmake,
no torch extension machinery: the library is plain C ABI (include/ssu.h).

    python -m mamba2_ssm_decode_gb300.build [--force] [--ptxas-info]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libssu_gb300.so")
HEADER = os.path.join(ROOT, "include", "ssu.h")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xcompiler", "-Wall", "-Xcompiler", "-fvisibility=hidden"]
# export only the C ABI: hide the statically linked CUDA runtime's symbols
LINK_FLAGS = ["-Xlinker", "--exclude-libs,ALL"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libssu_gb300.so")
    return path


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)
            if f.endswith((".cuh", ".h"))] + [HEADER, os.path.abspath(__file__)]


def _stale(target, inputs):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(i) > t for i in inputs)


def _compile(src, ptxas_info):
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    if ptxas_info:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, ptxas_info: bool = False, verbose: bool = False) -> str:
    """Compile (if anything changed) and return the path of libssu_gb300.so."""
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    deps = _deps()
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    todo = [s for s, o in zip(srcs, objs) if force or ptxas_info or _stale(o, [s, *deps])]
    if todo:
        with cf.ThreadPoolExecutor(max_workers=min(len(todo), os.cpu_count() or 4)) as ex:
            for obj, log in ex.map(lambda s: _compile(s, ptxas_info), todo):
                if verbose or ptxas_info:
                    print(f"== {os.path.basename(obj)}\n{log}", file=sys.stderr)
    if force or todo or _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *LINK_FLAGS, "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, ptxas_info=args.ptxas_info, verbose=True))
