"""Builds libsmla.so (the C-ABI library) in-tree with nvcc for sm_103a, and its debug
twin libsmla_debug.so (the same sources with SMLA_DEBUG: device-side bounds checks
of every computed shared-memory address and gathered row, reported as
SMLA_ERR_INTERNAL; no trap).

Each .cu file is compiled in parallel, then linked into a shared library next to
this file.  Usage: ``python -m sparse_mla_decode_03_gb300.build [-v]``."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsmla.so")
LIB_DEBUG = os.path.join(HERE, "libsmla_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I", os.path.join(ROOT, "include")]
SOURCES = ["smla_decode.cu", "smla_combine.cu", "smla_api.cu", "smla_noalloc.cu", "smla_simt.cu",
           "smla_paged.cu"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _compile(job: tuple) -> tuple:
    src, debug = job
    obj = os.path.join(OBJ, ("debug_" if debug else "") + os.path.splitext(src)[0] + ".o")
    extra = ["-DSMLA_DEBUG"] if debug else []
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, p.returncode, p.stdout + p.stderr, debug


def _link(objs, path: str) -> None:
    tmp = path + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        sys.stderr.write(p.stdout + p.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, path)


def build(verbose: bool = False) -> str:
    os.makedirs(OBJ, exist_ok=True)
    jobs = [(src, debug) for debug in (False, True) for src in SOURCES]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(_compile, jobs))
    for src, _, rc, log, debug in results:
        if (verbose and not debug) or rc != 0:
            sys.stderr.write(f"--- {src}{' (SMLA_DEBUG)' if debug else ''}\n{log}")
        if rc != 0:
            raise RuntimeError(f"nvcc failed on {src}")
    _link([r[1] for r in results if not r[4]], LIB)
    _link([r[1] for r in results if r[4]], LIB_DEBUG)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
