"""Build the CUDA library ``liboasis.so`` in-tree for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel with nvcc
(``-gencode arch=compute_103a,code=sm_103a``) and the objects are linked into
a shared library next to this file.  No torch headers are involved: the
library exposes a plain C ABI (``include/oasis.h``).
"""
from __future__ import annotations

import concurrent.futures
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "liboasis.so")
SOURCES = ["api.cu", "attn.cu", "score_topk.cu", "admit_gather.cu", "noalloc.cu"]
INCLUDE_DIRS = [CSRC, os.path.join(ROOT, "include")]
_INCLUDE_RE = re.compile(r'^\s*#\s*include\s*"([^"]+)"', re.M)


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; set NVCC or install the CUDA toolkit")
    return cand


def _flags(extra=()) -> list:
    return [
        "-gencode", "arch=compute_103a,code=sm_103a",
        "-O3", "-lineinfo", "-std=c++17",
        "-Xcompiler", "-fPIC,-fvisibility=hidden",
        "-I", os.path.join(ROOT, "include"),
        *extra,
    ]


def deps(src: str) -> list:
    """``src`` and every header it reaches through ``#include "..."``,
    followed recursively through ``csrc/`` and ``include/`` (system headers,
    in angle brackets, are not followed)."""
    seen, todo = [], [src]
    while todo:
        f = todo.pop()
        if f in seen:
            continue
        seen.append(f)
        base = os.path.dirname(f)
        with open(f) as fh:
            names = _INCLUDE_RE.findall(fh.read())
        for name in names:
            for d in [base] + INCLUDE_DIRS:
                cand = os.path.normpath(os.path.join(d, name))
                if os.path.exists(cand):
                    todo.append(cand)
                    break
    return seen


def _stale(target: str, deps: list) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile (only what changed unless ``force``) and return the .so path."""
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, deps(s)):
            jobs.append([nvcc, *_flags(extra_flags), "-c", s, "-o", o])

    def run(cmd):
        p = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, p

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, p in ex.map(run, jobs):
            if verbose or p.returncode != 0:
                sys.stderr.write(p.stdout + p.stderr)
            if p.returncode != 0:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
               "-cudart", "shared", "-o", tmp, *objs]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            sys.stderr.write(p.stdout + p.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
