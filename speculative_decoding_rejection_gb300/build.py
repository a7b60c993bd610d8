"""Builds libspecverify.so (sm_103a) in-tree with nvcc.

Each .cu file is compiled in parallel into _build/, then linked into a shared
library next to this file. No cmake, one -gencode.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = ROOT / "_build"
LIB = PKG / "libspecverify.so"
SOURCES = ["rowpass.cu", "linear.cu", "stream.cu", "resident.cu", "small.cu", "topk.cu", "tree.cu",
           "rheo.cu", "api.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(verbose: bool = False, extra_flags=()) -> Path:
    BUILD.mkdir(exist_ok=True)
    cc = nvcc()
    objs = []
    cmds = []
    for src in SOURCES:
        obj = BUILD / (Path(src).stem + ".o")
        objs.append(obj)
        cmds.append([cc, *ARCH, *FLAGS, *extra_flags, "-c", str(CSRC / src), "-o", str(obj)])
    with ThreadPoolExecutor(max_workers=min(len(cmds), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(_run, cmds))
    tmp = LIB.with_suffix(".so.tmp")
    logs.append(_run([cc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]))
    os.replace(tmp, LIB)
    if verbose:
        print("\n".join(l for l in logs if l.strip()))
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
