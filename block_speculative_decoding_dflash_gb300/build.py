"""Builds libdflash.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel into ``_build/`` and the
objects are linked into ``block_speculative_decoding_dflash_gb300/libdflash.so``.
No cmake; a rebuild only recompiles sources newer than their object.
"""

from __future__ import annotations

import os
import platform
import struct
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build", platform.machine())
LIB = os.path.join(PKG, "libdflash.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps_mtime() -> float:
    heads = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    heads.append(os.path.join(ROOT, "include", "dflash.h"))
    return max(os.path.getmtime(h) for h in heads)


def _compile(src: str, force: bool) -> str:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    path = os.path.join(CSRC, src)
    if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(
            os.path.getmtime(path), _deps_mtime()):
        return obj
    cmd = [nvcc()] + ARCH + FLAGS + ["-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


_ELF_MACHINE = {"x86_64": 62, "aarch64": 183}


def _lib_matches_host() -> bool:
    """False if an existing libdflash.so was linked for another CPU."""
    try:
        with open(LIB, "rb") as f:
            head = f.read(20)
        return struct.unpack("<H", head[18:20])[0] == _ELF_MACHINE.get(platform.machine(), -1)
    except (OSError, struct.error):
        return False


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    if not _lib_matches_host():
        force_link = True
    else:
        force_link = False
    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, force), srcs))
    if force or force_link or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-o", LIB] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(f"built {LIB}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
