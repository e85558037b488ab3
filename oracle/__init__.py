"""CPU oracle for fused GQA flash-attention prefill (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and it
shares no code with the CUDA library; see ``gqa_oracle.c`` for the definition
it computes and the page passages each step follows.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, library cross-checks, brute force, the tile counts printed on
the SGLang "gfx950 SWA prefix trim" page) and by the planted-mistake suite
``tests/test_oracle_mutations.py``.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libgqa_oracle.so")
_lib = None


def _compile(src: str, out: str) -> None:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", out + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        # OpenMP is optional: the oracle is correct single-threaded.
        subprocess.run(base, check=True, capture_output=True)
    os.replace(out + ".tmp", out)


def build(force: bool = False) -> str:
    """Compile the oracle to ``oracle/_build/libgqa_oracle.so`` if stale."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        _compile(_SRC, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    i32p = ctypes.POINTER(ctypes.c_int32)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.gqa_oracle_prefill.restype = ctypes.c_int
    lib.gqa_oracle_prefill.argtypes = [
        dp, dp, dp, i32p, i32p, i32p, ctypes.c_int, ctypes.c_long,
        ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_int, dp, ctypes.c_int,
        ctypes.POINTER(ctypes.c_uint8), dp, dp]
    lib.gqa_oracle_prefill_masked.restype = ctypes.c_int
    lib.gqa_oracle_prefill_masked.argtypes = lib.gqa_oracle_prefill.argtypes + [
        ctypes.POINTER(ctypes.c_uint32), i32p]
    lib.gqa_oracle_tile_census.restype = ctypes.c_long
    lib.gqa_oracle_tile_census.argtypes = [
        i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, i32p, ctypes.c_long]
    lib.gqa_oracle_num_threads.restype = ctypes.c_int
    lib.gqa_oracle_num_threads.argtypes = []
    return lib


def load(path: str | None = None):
    """Load the compiled oracle (building it first when ``path`` is None)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def compile_variant(src_text: str) -> str:
    """Compile an edited copy of the oracle source into a temp dir (used by
    the planted-mistake tests) and return the path of the shared object."""
    d = tempfile.mkdtemp(prefix="gqa_oracle_variant_")
    src = os.path.join(d, "variant.c")
    with open(src, "w") as f:
        f.write(src_text)
    out = os.path.join(d, "libvariant.so")
    _compile(src, out)
    return out


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def remove_variant(path: str) -> None:
    shutil.rmtree(os.path.dirname(path), ignore_errors=True)


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as_f64(x):
    """Exact widening of a torch tensor / numpy array to contiguous float64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().cpu().to(torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _as_i32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _as_u32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x).astype(np.uint32, copy=False))


def num_threads() -> int:
    return int(load().gqa_oracle_num_threads())


def prefill(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale, window=0,
            sinks=None, smooth_softmax=False, rows=None, lib=None, out=None, lse=None,
            custom_mask=None, mask_indptr=None):
    """Run the oracle.  q [total_q,Hq,d]; k,v [total_kv,Hkv,d]; metadata as
    int arrays.  ``rows`` optionally lists the token rows to compute (the
    others come back as NaN, or untouched when ``out``/``lse`` are given:
    caller-owned contiguous float64 buffers of the result shapes, reused
    across calls).  ``custom_mask`` (uint32 words) and ``mask_indptr``
    (int32 [B+1]) add the custom-mask condition (see gqa_oracle.c).
    Returns (out float64 [total_q,Hq,d], lse float64 [total_q,Hq])."""
    lib = lib or load()
    q64, k64, v64 = _as_f64(q), _as_f64(k), _as_f64(v)
    cu, pre, kvi = _as_i32(cu_seqlens_q), _as_i32(prefix_lens), _as_i32(kv_indptr)
    total_q, hq, d = q64.shape
    total_kv, hkv, dk = k64.shape
    assert dk == d and v64.shape == k64.shape
    num_seqs = len(pre)
    if out is None:
        out = np.full((total_q, hq, d), np.nan)
    if lse is None:
        lse = np.full((total_q, hq), np.nan)
    assert out.dtype == np.float64 and out.shape == (total_q, hq, d) and out.flags.c_contiguous
    assert lse.dtype == np.float64 and lse.shape == (total_q, hq) and lse.flags.c_contiguous
    sel = None
    if rows is not None:
        sel = np.zeros(total_q, dtype=np.uint8)
        sel[np.asarray(rows, dtype=np.int64)] = 1
    s64 = None if sinks is None else _as_f64(sinks).reshape(hq)
    args = [
        _ptr(q64, ctypes.c_double), _ptr(k64, ctypes.c_double),
        _ptr(v64, ctypes.c_double), _ptr(cu, ctypes.c_int32),
        _ptr(pre, ctypes.c_int32), _ptr(kvi, ctypes.c_int32), num_seqs,
        total_q, total_kv, hq, hkv, d, float(scale), int(window),
        None if s64 is None else _ptr(s64, ctypes.c_double),
        1 if smooth_softmax else 0,
        None if sel is None else _ptr(sel, ctypes.c_uint8),
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double)]
    if custom_mask is None:
        rc = lib.gqa_oracle_prefill(*args)
    else:
        words = _as_u32(custom_mask)
        mip = _as_i32(mask_indptr)
        rc = lib.gqa_oracle_prefill_masked(*args, _ptr(words, ctypes.c_uint32),
                                           _ptr(mip, ctypes.c_int32))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out, lse


def tile_census(cu_seqlens_q, prefix_lens, hkv, rows, block_n, window, lib=None):
    """Per-unit tile bookkeeping derived from the mask predicate.  Returns an
    int32 array [n_units, 6] of (b, g, q0, kv_lo, n_tiles, n_masked) in
    (b, g, q-tile) order."""
    lib = lib or load()
    cu, pre = _as_i32(cu_seqlens_q), _as_i32(prefix_lens)
    num_seqs = len(pre)
    e = np.diff(cu.astype(np.int64))
    max_units = int(hkv * np.sum((e + rows - 1) // rows)) if num_seqs else 0
    rec = np.zeros((max(max_units, 1), 6), dtype=np.int32)
    n = lib.gqa_oracle_tile_census(
        _ptr(cu, ctypes.c_int32), _ptr(pre, ctypes.c_int32), num_seqs, hkv,
        rows, block_n, int(window), _ptr(rec, ctypes.c_int32), max(max_units, 1))
    if n < 0:
        raise ValueError("oracle census rejected the arguments")
    return rec[:n].copy()
