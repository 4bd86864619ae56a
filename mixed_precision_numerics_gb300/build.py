"""Build libmpnum.so in-tree: nvcc for sm_103a, one object per .cu, compiled in parallel."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmpnum.so")
HEADER = os.path.join(ROOT, "include", "mpnum.h")

SOURCES = ["mp_common.cu", "mp_adamw.cu", "mp_fp8.cu", "mp_nvfp4.cu", "mp_mx.cu"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = GENCODE + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                        "-I", os.path.join(ROOT, "include")]


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [HEADER, __file__]


def _stale(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in _deps())


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    cmd = ["nvcc", *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{p.stderr}")
    if verbose and p.stderr:
        sys.stderr.write(p.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu and link libmpnum.so next to this file; returns its path."""
    if not force and not _stale(LIB):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    p = subprocess.run(["nvcc", *GENCODE, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
