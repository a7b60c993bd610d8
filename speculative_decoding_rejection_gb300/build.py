"""Builds libspecverify.so (sm_103a) in-tree with nvcc, and the same sources
with SPEC_CHECKED as libspecverify_checked.so (every global access of the
kernels bounds-checked against the call's buffers; a test build).

Each .cu file is compiled in parallel into _build/ (_build/checked/), then
linked into a shared library next to this file. No cmake, one -gencode.
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
CHECKED_LIB = PKG / "libspecverify_checked.so"
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


def build(verbose: bool = False, extra_flags=(), checked: bool = True) -> Path:
    """Compiles and links the library (and, with `checked`, its bounds-checked
    build); returns the product library's path."""
    cc = nvcc()
    variants = [(BUILD, LIB, [])]
    if checked:
        variants.append((BUILD / "checked", CHECKED_LIB, ["-DSPEC_CHECKED"]))
    cmds, links = [], []
    for out_dir, lib_path, defs in variants:
        out_dir.mkdir(parents=True, exist_ok=True)
        objs = []
        for src in SOURCES:
            obj = out_dir / (Path(src).stem + ".o")
            objs.append(obj)
            cmds.append([cc, *ARCH, *FLAGS, *defs, *extra_flags, "-c", str(CSRC / src), "-o",
                         str(obj)])
        links.append((objs, lib_path))
    with ThreadPoolExecutor(max_workers=min(len(cmds), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(_run, cmds))
    for objs, lib_path in links:
        tmp = lib_path.with_suffix(".so.tmp")
        logs.append(_run([cc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]))
        os.replace(tmp, lib_path)
    if verbose:
        print("\n".join(l for l in logs if l.strip()))
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
