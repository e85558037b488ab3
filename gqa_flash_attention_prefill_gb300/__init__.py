"""Fused GQA flash-attention prefill for GB300 (sm_103a).

Thin ctypes binding over ``libgqa_prefill.so`` (the C ABI declared in
``include/gqa_prefill.h``): the functions here only marshal torch tensors into
pointers and sizes.  Every step of the computation runs in the CUDA kernels;
there is no CPU or PyTorch fallback, and calling in without the built library
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = ["load", "gqa_flash_prefill", "gqa_flash_prefill_debug", "prefill", "prepare",
           "PreparedCall",
           "plan", "force_block_n", "force_q_tiles", "get_device_status", "get_stream_status", "set_tuning",
           "gqa_flash_prefill_splitkv", "splitkv_workspace", "prefill_splitkv",
           "gqa_flash_prefill_splitkv_noalloc", "prefill_splitkv_noalloc",
           "gqa_flash_prefill_masked", "prefill_masked",
           "NOALLOC_SCRATCH_BYTES", "gqa_flash_prefill_paged", "prefill_paged",
           "clear_config_cache", "config_block_n", "selftest_timeout", "GQAError",
           "GQA_F16", "GQA_BF16", "GQA_DEV_TIMEOUT", "GQA_DEV_BAD_METADATA", "SPLITS_BALANCED",
           "FLAG_METADATA_READY", "set_call_flags", "get_call_flags",
           "EXPORTED_SYMBOLS"]

GQA_F16, GQA_BF16 = 0, 1
GQA_OK, GQA_ERR_INVALID, GQA_ERR_UNSUPPORTED, GQA_ERR_CUDA = 0, -1, -2, -3
GQA_DEV_TIMEOUT, GQA_DEV_BAD_METADATA = 1, 2
SPLITS_BALANCED = -1  # num_splits of the balanced split (GQA_SPLITS_BALANCED)
FLAG_METADATA_READY = 1  # GQA_FLAG_METADATA_READY (gqa_prefill_set_call_flags)

EXPORTED_SYMBOLS = [
    "gqa_flash_prefill", "gqa_flash_prefill_debug", "gqa_prefill_plan",
    "gqa_prefill_force_block_n", "gqa_prefill_get_device_status",
    "gqa_prefill_status_string", "gqa_prefill_version", "gqa_prefill_set_tuning",
    "gqa_prefill_clear_config_cache", "gqa_prefill_config_block_n",
    "gqa_prefill_selftest_timeout", "gqa_prefill_force_q_tiles",
    "gqa_flash_prefill_splitkv", "gqa_prefill_splitkv_workspace",
    "gqa_flash_prefill_splitkv_noalloc", "gqa_flash_prefill_paged",
    "gqa_prefill_get_stream_status", "gqa_flash_prefill_masked",
    "gqa_prefill_set_call_flags", "gqa_prefill_get_call_flags",
]
NOALLOC_SCRATCH_BYTES = 32 << 20  # the library's file-scope split-KV scratch (gqa_prefill.h)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgqa_prefill.so")
_lib = None


class GQAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {code} ({_status_string(code)})")


class _Plan(ctypes.Structure):
    _fields_ = [("rows_per_unit", ctypes.c_int), ("block_n", ctypes.c_int),
                ("kv_stages", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("grid", ctypes.c_int), ("max_units", ctypes.c_int),
                ("q_tiles", ctypes.c_int)]


def load(path: Optional[str] = None):
    """Load libgqa_prefill.so (built by ``__graft_entry__.build()`` or
    ``python -m gqa_flash_attention_prefill_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    # GQA_PREFILL_LIB names another build of the same library (used to time
    # two builds against each other on one machine).
    p = path or os.environ.get("GQA_PREFILL_LIB") or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library {p} is missing: build it with "
            "`python -m gqa_flash_attention_prefill_gb300.build`")
    lib = ctypes.CDLL(p)
    vp, i32p, fp = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    core = [vp, vp, vp, i32p, i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_float, ctypes.c_int, fp, ctypes.c_int, vp, fp, vp]
    lib.gqa_flash_prefill.argtypes = core
    lib.gqa_flash_prefill.restype = ctypes.c_int
    lib.gqa_flash_prefill_debug.argtypes = core + [vp]
    lib.gqa_flash_prefill_debug.restype = ctypes.c_int
    lib.gqa_flash_prefill_splitkv.argtypes = core[:-1] + [ctypes.c_int, vp, ctypes.c_size_t, vp]
    lib.gqa_flash_prefill_splitkv.restype = ctypes.c_int
    lib.gqa_flash_prefill_masked.argtypes = core[:18] + [vp, vp, ctypes.c_longlong, vp, fp, vp]
    lib.gqa_flash_prefill_masked.restype = ctypes.c_int
    lib.gqa_flash_prefill_paged.argtypes = [vp] * 7 + [ctypes.c_int] * 10 + [
        ctypes.c_float, ctypes.c_int, vp, ctypes.c_int, vp, vp, vp]
    lib.gqa_flash_prefill_paged.restype = ctypes.c_int
    lib.gqa_flash_prefill_splitkv_noalloc.argtypes = core[:-1] + [ctypes.c_int, vp]
    lib.gqa_flash_prefill_splitkv_noalloc.restype = ctypes.c_int
    lib.gqa_prefill_splitkv_workspace.argtypes = [ctypes.c_int] * 9 + [
        ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_size_t)]
    lib.gqa_prefill_splitkv_workspace.restype = ctypes.c_int
    lib.gqa_prefill_plan.argtypes = [ctypes.c_int] * 8 + [ctypes.POINTER(_Plan)]
    lib.gqa_prefill_plan.restype = ctypes.c_int
    lib.gqa_prefill_force_block_n.argtypes = [ctypes.c_int]
    lib.gqa_prefill_force_block_n.restype = ctypes.c_int
    lib.gqa_prefill_force_q_tiles.argtypes = [ctypes.c_int]
    lib.gqa_prefill_force_q_tiles.restype = ctypes.c_int
    lib.gqa_prefill_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.gqa_prefill_get_device_status.restype = ctypes.c_int
    lib.gqa_prefill_get_stream_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]
    lib.gqa_prefill_get_stream_status.restype = ctypes.c_int
    lib.gqa_prefill_status_string.argtypes = [ctypes.c_int]
    lib.gqa_prefill_status_string.restype = ctypes.c_char_p
    lib.gqa_prefill_version.argtypes = []
    lib.gqa_prefill_version.restype = ctypes.c_char_p
    lib.gqa_prefill_set_tuning.argtypes = [ctypes.c_int]
    lib.gqa_prefill_set_tuning.restype = ctypes.c_int
    lib.gqa_prefill_clear_config_cache.argtypes = []
    lib.gqa_prefill_clear_config_cache.restype = ctypes.c_int
    lib.gqa_prefill_config_block_n.argtypes = [ctypes.c_int] * 7 + [
        ctypes.POINTER(ctypes.c_int)] * 3
    lib.gqa_prefill_config_block_n.restype = ctypes.c_int
    lib.gqa_prefill_selftest_timeout.argtypes = [ctypes.c_int, ctypes.c_void_p,
                                                 ctypes.POINTER(ctypes.c_int)]
    lib.gqa_prefill_selftest_timeout.restype = ctypes.c_int
    lib.gqa_prefill_set_call_flags.argtypes = [ctypes.c_uint]
    lib.gqa_prefill_set_call_flags.restype = ctypes.c_int
    lib.gqa_prefill_get_call_flags.argtypes = []
    lib.gqa_prefill_get_call_flags.restype = ctypes.c_uint
    if path is None:
        _lib = lib
    return lib


def _status_string(code: int) -> str:
    try:
        return load().gqa_prefill_status_string(code).decode()
    except Exception:  # pragma: no cover - library missing
        return "?"


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return GQA_BF16
    if t.dtype == torch.float16:
        return GQA_F16
    raise TypeError(f"q/k/v must be float16 or bfloat16, got {t.dtype}")


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _args(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale, window, sinks,
          smooth_softmax, out, lse, stream, max_seqlen_q):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [rows, heads, d] tensor")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("prefix_lens", prefix_lens),
                    ("kv_indptr", kv_indptr)):
        if str(t.dtype) != "torch.int32" or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 tensor")
    total_q, hq, d = q.shape
    total_kv, hkv, _ = k.shape
    return (_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q), _ptr(prefix_lens),
            _ptr(kv_indptr), int(prefix_lens.numel()), int(total_q), int(total_kv),
            int(max_seqlen_q), int(hq), int(hkv), int(d), _dtype_code(q), float(scale),
            int(window), _ptr(sinks), 1 if smooth_softmax else 0, _ptr(out), _ptr(lse),
            _stream_handle(stream))


def gqa_flash_prefill(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale,
                      window=0, sinks=None, smooth_softmax=False, out=None,
                      lse=None, stream=None, max_seqlen_q=0):
    """Marshal torch CUDA tensors into the C ABI call (see gqa_prefill.h).
    ``out`` [total_q, Hq, d] and ``lse`` (fp32 [total_q, Hq] or None) are
    written in place; returns ``out``."""
    rc = load().gqa_flash_prefill(*_args(q, k, v, cu_seqlens_q, prefix_lens,
                                         kv_indptr, scale, window, sinks,
                                         smooth_softmax, out, lse, stream,
                                         max_seqlen_q))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_flash_prefill")
    return out


def gqa_flash_prefill_masked(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale,
                             custom_mask, mask_indptr, window=0, sinks=None,
                             smooth_softmax=False, out=None, lse=None, stream=None,
                             max_seqlen_q=0):
    """gqa_flash_prefill with a custom mask (see gqa_prefill.h): custom_mask
    is a device tensor of 32-bit words (int32 or uint32), mask_indptr a
    device int32 [B+1] of word offsets."""
    for name, t in (("custom_mask", custom_mask), ("mask_indptr", mask_indptr)):
        if t.element_size() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous tensor of 32-bit words")
    a = _args(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale, window, sinks,
              smooth_softmax, out, lse, stream, max_seqlen_q)
    rc = load().gqa_flash_prefill_masked(*a[:18], _ptr(custom_mask), _ptr(mask_indptr),
                                         int(custom_mask.numel()), *a[18:])
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_flash_prefill_masked")
    return out


def prefill_masked(batch, custom_mask, mask_indptr, out=None, lse=None, with_lse=True,
                   stream=None):
    """gqa_flash_prefill_masked on one ``workloads.Batch`` already on the GPU
    (custom_mask / mask_indptr from ``workloads.pack_custom_mask``, on the
    GPU); allocates out/lse with torch when not given.  Returns (out, lse)."""
    import torch
    if out is None:
        out = torch.empty_like(batch.q)
    if lse is None and with_lse:
        lse = torch.empty(batch.q.shape[:2], dtype=torch.float32, device=batch.q.device)
    gqa_flash_prefill_masked(batch.q, batch.k, batch.v, batch.cu_seqlens_q, batch.prefix_lens,
                             batch.kv_indptr, batch.scale, custom_mask, mask_indptr,
                             window=batch.window, sinks=batch.sinks, smooth_softmax=batch.smooth,
                             out=out, lse=lse, stream=stream, max_seqlen_q=batch.max_seqlen_q)
    return out, lse


def gqa_flash_prefill_debug(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale,
                            unit_log, window=0, sinks=None, smooth_softmax=False,
                            out=None, lse=None, stream=None, max_seqlen_q=0):
    """Same as gqa_flash_prefill, and writes one 8-int record per work unit
    into ``unit_log`` (device int32 [max_units, 8])."""
    rc = load().gqa_flash_prefill_debug(*_args(q, k, v, cu_seqlens_q, prefix_lens,
                                               kv_indptr, scale, window, sinks,
                                               smooth_softmax, out, lse, stream,
                                               max_seqlen_q), _ptr(unit_log))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_flash_prefill_debug")
    return out


def gqa_flash_prefill_splitkv(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale,
                              workspace, num_splits=0, window=0, sinks=None,
                              smooth_softmax=False, out=None, lse=None, stream=None,
                              max_seqlen_q=0):
    """Split-KV form of gqa_flash_prefill (see gqa_prefill.h); ``workspace``
    is a device tensor (any dtype) at least ``splitkv_workspace(...)`` bytes,
    or None when the call does not split."""
    a = _args(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale, window, sinks,
              smooth_softmax, out, lse, stream, max_seqlen_q)
    ws = _ptr(workspace)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = load().gqa_flash_prefill_splitkv(*a[:-1], int(num_splits), ws, nbytes, a[-1])
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_flash_prefill_splitkv")
    return out


def splitkv_workspace(num_seqs, total_q, max_seqlen_q, hq, hkv, d, dtype, window,
                      num_splits=0):
    """(splits used, workspace bytes) for a split-KV call with these shapes."""
    used, nbytes = ctypes.c_int(0), ctypes.c_size_t(0)
    code = dtype if isinstance(dtype, int) else (GQA_BF16 if "bf16" in str(dtype) else GQA_F16)
    rc = load().gqa_prefill_splitkv_workspace(int(num_seqs), int(total_q), int(max_seqlen_q),
                                              int(hq), int(hkv), int(d), code, int(window),
                                              int(num_splits), ctypes.byref(used),
                                              ctypes.byref(nbytes))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_splitkv_workspace")
    return used.value, nbytes.value


def gqa_flash_prefill_splitkv_noalloc(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale,
                                      num_splits=0, window=0, sinks=None, smooth_softmax=False,
                                      out=None, lse=None, stream=None, max_seqlen_q=0):
    """Split-KV with the library's file-scope scratch (see gqa_prefill.h): no
    workspace, nothing allocated; overlapping calls race on the scratch."""
    a = _args(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, scale, window, sinks,
              smooth_softmax, out, lse, stream, max_seqlen_q)
    rc = load().gqa_flash_prefill_splitkv_noalloc(*a[:-1], int(num_splits), a[-1])
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_flash_prefill_splitkv_noalloc")
    return out


def prefill_splitkv_noalloc(batch, num_splits=0, out=None, lse=None, stream=None):
    """gqa_flash_prefill_splitkv_noalloc on one ``workloads.Batch`` already on
    the GPU, into caller buffers (out is required: the call allocates nothing)."""
    gqa_flash_prefill_splitkv_noalloc(batch.q, batch.k, batch.v, batch.cu_seqlens_q,
                                      batch.prefix_lens, batch.kv_indptr, batch.scale,
                                      num_splits=num_splits, window=batch.window,
                                      sinks=batch.sinks, smooth_softmax=batch.smooth, out=out,
                                      lse=lse, stream=stream, max_seqlen_q=batch.max_seqlen_q)
    return out, lse


def prefill_splitkv(batch, num_splits=0, workspace=None, out=None, lse=None, with_lse=True,
                    stream=None):
    """Split-KV run of one ``workloads.Batch`` already on the GPU; allocates the
    workspace (and out/lse) with torch when not given.  Returns (out, lse)."""
    import torch
    if out is None:
        out = torch.empty_like(batch.q)
    if lse is None and with_lse:
        lse = torch.empty(batch.q.shape[:2], dtype=torch.float32, device=batch.q.device)
    used, nbytes = splitkv_workspace(batch.num_seqs, batch.total_q, batch.max_seqlen_q,
                                     batch.hq, batch.hkv, batch.d, batch.dtype_name,
                                     batch.window, num_splits)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=batch.q.device)
    gqa_flash_prefill_splitkv(batch.q, batch.k, batch.v, batch.cu_seqlens_q,
                              batch.prefix_lens, batch.kv_indptr, batch.scale, workspace,
                              num_splits=num_splits, window=batch.window, sinks=batch.sinks,
                              smooth_softmax=batch.smooth, out=out, lse=lse, stream=stream,
                              max_seqlen_q=batch.max_seqlen_q)
    return out, lse


def gqa_flash_prefill_paged(q, k_pages, v_pages, cu_seqlens_q, prefix_lens, kv_page_indptr,
                            kv_page_indices, scale, window=0, sinks=None, smooth_softmax=False,
                            out=None, lse=None, stream=None, max_seqlen_q=0):
    """Marshal a paged-KV call (see gqa_prefill.h): k_pages / v_pages are
    [num_pages, page_size, Hkv, d]; returns ``out``."""
    for name, t in (("q", q), ("out", out)):
        if t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [rows, heads, d] tensor")
    for name, t in (("k_pages", k_pages), ("v_pages", v_pages)):
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [pages, page_size, heads, d] tensor")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("prefix_lens", prefix_lens),
                    ("kv_page_indptr", kv_page_indptr), ("kv_page_indices", kv_page_indices)):
        if str(t.dtype) != "torch.int32" or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 tensor")
    total_q, hq, d = q.shape
    num_pages, page_size, hkv, _ = k_pages.shape
    rc = load().gqa_flash_prefill_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(cu_seqlens_q), _ptr(prefix_lens),
        _ptr(kv_page_indptr), _ptr(kv_page_indices), int(kv_page_indices.numel()),
        int(page_size), int(num_pages), int(prefix_lens.numel()), int(total_q),
        int(max_seqlen_q), int(hq), int(hkv), int(d), _dtype_code(q), float(scale), int(window),
        _ptr(sinks), 1 if smooth_softmax else 0, _ptr(out), _ptr(lse), _stream_handle(stream))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_flash_prefill_paged")
    return out


def prefill_paged(paged, out=None, lse=None, with_lse=True, stream=None):
    """Run one ``workloads.PagedBatch`` already on the GPU.  Returns (out, lse)."""
    import torch
    b = paged.batch
    if out is None:
        out = torch.empty_like(b.q)
    if lse is None and with_lse:
        lse = torch.empty(b.q.shape[:2], dtype=torch.float32, device=b.q.device)
    gqa_flash_prefill_paged(b.q, paged.k_pages, paged.v_pages, b.cu_seqlens_q, b.prefix_lens,
                            paged.page_indptr, paged.page_indices, b.scale, window=b.window,
                            sinks=b.sinks, smooth_softmax=b.smooth, out=out, lse=lse,
                            stream=stream, max_seqlen_q=b.max_seqlen_q)
    return out, lse


def prefill(batch, out=None, lse=None, with_lse=True, stream=None):
    """Run one ``workloads.Batch`` already on the GPU; allocates out/lse with
    torch when not given.  Returns (out, lse)."""
    import torch
    if out is None:
        out = torch.empty_like(batch.q)
    if lse is None and with_lse:
        lse = torch.empty(batch.q.shape[:2], dtype=torch.float32, device=batch.q.device)
    gqa_flash_prefill(batch.q, batch.k, batch.v, batch.cu_seqlens_q,
                      batch.prefix_lens, batch.kv_indptr, batch.scale,
                      window=batch.window, sinks=batch.sinks,
                      smooth_softmax=batch.smooth, out=out, lse=lse,
                      stream=stream, max_seqlen_q=batch.max_seqlen_q)
    return out, lse


class PreparedCall:
    """gqa_flash_prefill (or, with ``num_splits``, gqa_flash_prefill_splitkv
    on ``workspace``) with its arguments marshalled once: calling the object
    re-issues the same C ABI call (same buffers, same stream), which keeps
    the host cost of a call to the ctypes round trip.  For callers that
    replay a fixed sequence of calls over resident buffers, such as the
    layers of a prefill."""

    __slots__ = ("_fn", "_args", "_name", "out", "lse", "workspace")

    def __init__(self, batch, out, lse=None, stream=None, num_splits=None, workspace=None):
        a = _args(batch.q, batch.k, batch.v, batch.cu_seqlens_q, batch.prefix_lens,
                  batch.kv_indptr, batch.scale, batch.window, batch.sinks, batch.smooth, out, lse,
                  stream, batch.max_seqlen_q)
        if num_splits is None:
            self._fn, self._name, self._args = load().gqa_flash_prefill, "gqa_flash_prefill", a
        else:
            nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
            self._fn, self._name = load().gqa_flash_prefill_splitkv, "gqa_flash_prefill_splitkv"
            self._args = a[:-1] + (int(num_splits), _ptr(workspace), nbytes, a[-1])
        self.out, self.lse, self.workspace = out, lse, workspace

    def __call__(self):
        rc = self._fn(*self._args)
        if rc != GQA_OK:
            raise GQAError(rc, self._name)


def prepare(batch, out, lse=None, stream=None, num_splits=None, workspace=None) -> PreparedCall:
    """A PreparedCall of one ``workloads.Batch`` already on the GPU, writing
    ``out`` (and ``lse`` when given) on ``stream``; with ``num_splits`` (for
    example SPLITS_BALANCED) the split-KV entry point on ``workspace``."""
    return PreparedCall(batch, out, lse, stream, num_splits, workspace)


def set_call_flags(flags: int) -> None:
    """Flags for the calling thread's later calls (gqa_prefill_set_call_flags):
    FLAG_METADATA_READY, or 0."""
    rc = load().gqa_prefill_set_call_flags(int(flags))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_set_call_flags")


def get_call_flags() -> int:
    return int(load().gqa_prefill_get_call_flags())


def plan(num_seqs, total_q, max_seqlen_q, hq, hkv, d, dtype, window) -> dict:
    """Host-only launch plan (rows_per_unit, block_n, kv_stages, ctas_per_sm,
    grid, max_units, q_tiles) for a call with these shapes."""
    p = _Plan()
    code = dtype if isinstance(dtype, int) else (GQA_BF16 if "bf16" in str(dtype) else GQA_F16)
    rc = load().gqa_prefill_plan(int(num_seqs), int(total_q), int(max_seqlen_q), int(hq),
                                 int(hkv), int(d), code, int(window), ctypes.byref(p))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_plan")
    return {f: getattr(p, f) for f, _ in _Plan._fields_}


def force_block_n(block_n: int) -> None:
    rc = load().gqa_prefill_force_block_n(int(block_n))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_force_block_n")


def force_q_tiles(q_tiles: int) -> None:
    """Pin 1 or 2 query tiles per work unit for later calls (0: the cache's choice)."""
    rc = load().gqa_prefill_force_q_tiles(int(q_tiles))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_force_q_tiles")


def set_tuning(enable: bool) -> None:
    """Turn the configuration cache's timed sweep on or off (see gqa_prefill.h)."""
    rc = load().gqa_prefill_set_tuning(1 if enable else 0)
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_set_tuning")


def clear_config_cache() -> None:
    load().gqa_prefill_clear_config_cache()


def config_block_n(total_q, max_seqlen_q, hq, hkv, d, dtype, window):
    """(block_n, q_tiles, tuned) cached for these shapes; block_n 0 = no entry
    yet."""
    bn, qt, tuned = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    code = dtype if isinstance(dtype, int) else (GQA_BF16 if "bf16" in str(dtype) else GQA_F16)
    rc = load().gqa_prefill_config_block_n(int(total_q), int(max_seqlen_q), int(hq), int(hkv),
                                           int(d), code, int(window), ctypes.byref(bn),
                                           ctypes.byref(qt), ctypes.byref(tuned))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_config_block_n")
    return bn.value, qt.value, bool(tuned.value)


def selftest_timeout(timeout_ms: int = 50, stream=None) -> int:
    """Run the bounded-wait self-test; returns the device status word it read."""
    st = ctypes.c_int(0)
    rc = load().gqa_prefill_selftest_timeout(int(timeout_ms), _stream_handle(stream),
                                             ctypes.byref(st))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_selftest_timeout")
    return st.value


def get_stream_status(stream=None) -> int:
    """Read and clear the device status word in the order of ``stream``
    (default: the current stream), waiting for that stream only."""
    v = ctypes.c_int(0)
    rc = load().gqa_prefill_get_stream_status(_stream_handle(stream), ctypes.byref(v))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_get_stream_status")
    return v.value


def get_device_status() -> int:
    """Read and clear the device status word (synchronises the device)."""
    v = ctypes.c_int(0)
    rc = load().gqa_prefill_get_device_status(ctypes.byref(v))
    if rc != GQA_OK:
        raise GQAError(rc, "gqa_prefill_get_device_status")
    return v.value
