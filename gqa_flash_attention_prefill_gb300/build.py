"""Builds libgqa_prefill.so in-tree for sm_103a (nvcc, no cmake).

Each csrc/*.cu translation unit is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a``, then linked into a shared object
next to this file.  Run ``python -m gqa_flash_attention_prefill_gb300.build``
or call :func:`build`.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgqa_prefill.so")
SOURCES = ["host.cu", "inst_d64.cu", "inst_d64_pair.cu", "inst_d128.cu", "inst_d256.cu",
           "inst_split.cu", "inst_paged.cu", "inst_mask.cu", "inst_balanced.cu", "merge.cu",
           "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _flags():
    # Hidden by default: the library exports only the C ABI (GQA_API).
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-Xcompiler", "-fvisibility=hidden", "-I", CSRC, "-I", INCLUDE]


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "gqa_prefill.h"))
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + _flags()
    if verbose:
        cmd += ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    if verbose:
        sys.stderr.write(res.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libgqa_prefill.so."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= _deps_mtime()):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB + ".tmp"
    # The driver's tensor-map encoder is fetched at run time through the
    # runtime's entry-point query, so nothing links against libcuda.
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
