"""Seeded synthetic inputs for the prefill path.

This module only draws random numbers and lays out ragged-batch metadata; it
holds none of the attention arithmetic, so both the CUDA path's tests and the
oracle can take their inputs from it.

Distributions follow the workloads the pages describe for gpt-oss-shaped
layers (hip-ep PR #622 sink/window harness: H=64, G=8, d=64, pure and chunked
prefill over past lengths 512/8192; SGLang PR #34468 microbench: prefix /
extend pairs, window 128, full and window-bounded prefix layouts): Q, K, V are
drawn i.i.d. N(0, 1) in fp32 and rounded to the 16-bit input type; per-head
sink logits are N(0, 1), rounded to the input type and handed over as fp32.
There are no model weights: these tensors stand in for a real model's
activations.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Batch:
    """One call's inputs, on the CPU unless moved with :meth:`to`."""
    q: torch.Tensor              # [total_q, hq, d]
    k: torch.Tensor              # [total_kv, hkv, d]
    v: torch.Tensor              # [total_kv, hkv, d]
    cu_seqlens_q: torch.Tensor   # int32 [B+1]
    prefix_lens: torch.Tensor    # int32 [B]
    kv_indptr: torch.Tensor      # int32 [B+1]
    hq: int
    hkv: int
    d: int
    window: int                  # <= 0: none
    sinks: Optional[torch.Tensor]  # fp32 [hq] or None
    smooth: bool
    scale: float
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.prefix_lens.numel())

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def total_kv(self) -> int:
        return int(self.k.shape[0])

    @property
    def max_seqlen_q(self) -> int:
        if "max_seqlen_q" not in self.meta:  # host copy, kept across .to()
            e = self.extend_lens
            self.meta["max_seqlen_q"] = max(e) if e else 0
        return self.meta["max_seqlen_q"]

    @property
    def extend_lens(self) -> List[int]:
        if "extend_lens" not in self.meta:
            cu = self.cu_seqlens_q.tolist()
            self.meta["extend_lens"] = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
        return self.meta["extend_lens"]

    @property
    def dtype_name(self) -> str:
        return "bf16" if self.q.dtype == torch.bfloat16 else "f16"

    def to(self, device) -> "Batch":
        self.max_seqlen_q  # cache host-side metadata before the move
        mv = lambda t: None if t is None else t.to(device)
        return Batch(mv(self.q), mv(self.k), mv(self.v), mv(self.cu_seqlens_q),
                     mv(self.prefix_lens), mv(self.kv_indptr), self.hq, self.hkv,
                     self.d, self.window, mv(self.sinks), self.smooth, self.scale,
                     self.name, dict(self.meta))


def _normal(gen, shape, dtype, device="cpu"):
    return torch.randn(*shape, generator=gen, dtype=torch.float32, device=device).to(dtype)


def make_batch(prefix_lens, extend_lens, hq, hkv, d, dtype="bf16", window=0,
               sink_mode="head", seed=0, scale=None, name="", device="cpu") -> Batch:
    """Ragged batch: sequence b has prefix_lens[b] cached keys followed by
    extend_lens[b] new tokens; its KV rows are packed [prefix | extend] back to
    back in sequence order.  sink_mode is "none", "head" or "smooth"."""
    assert len(prefix_lens) == len(extend_lens)
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    gen = torch.Generator(device=device).manual_seed(int(seed))
    b = len(prefix_lens)
    cu = [0]
    kvp = [0]
    for p, e in zip(prefix_lens, extend_lens):
        cu.append(cu[-1] + int(e))
        kvp.append(kvp[-1] + int(p) + int(e))
    total_q, total_kv = cu[-1], kvp[-1]
    q = _normal(gen, (total_q, hq, d), dt, device)
    k = _normal(gen, (total_kv, hkv, d), dt, device)
    v = _normal(gen, (total_kv, hkv, d), dt, device)
    sinks = None
    if sink_mode == "head":
        sinks = _normal(gen, (hq,), dt, device).to(torch.float32)
    elif sink_mode not in ("none", "smooth"):
        raise ValueError(sink_mode)
    return Batch(q, k, v,
                 torch.tensor(cu, dtype=torch.int32, device=device),
                 torch.tensor([int(p) for p in prefix_lens], dtype=torch.int32, device=device),
                 torch.tensor(kvp, dtype=torch.int32, device=device),
                 hq, hkv, d, int(window), sinks, sink_mode == "smooth",
                 float(scale if scale is not None else d ** -0.5), name,
                 {"seed": int(seed), "num_seqs": b})


def window_bounded(batch: Batch, window: int) -> Batch:
    """The same batch with each sequence's prefix cut to its last
    min(prefix, window) rows, the layout a serving stack hands a
    sliding-window layer (SGLang PR #34468, commit 1: window_kv_indptr).
    Positions inside the kernel are relative, so the result must not change."""
    cu = batch.cu_seqlens_q.tolist()
    kvp = batch.kv_indptr.tolist()
    pre = batch.prefix_lens.tolist()
    ks, vs, new_pre, new_kvp = [], [], [], [0]
    for i, p in enumerate(pre):
        e = cu[i + 1] - cu[i]
        keep = min(p, window) if window > 0 else p
        lo = kvp[i] + (p - keep)
        ks.append(batch.k[lo:kvp[i + 1]])
        vs.append(batch.v[lo:kvp[i + 1]])
        new_pre.append(keep)
        new_kvp.append(new_kvp[-1] + keep + e)
    return Batch(batch.q, torch.cat(ks), torch.cat(vs), batch.cu_seqlens_q,
                 torch.tensor(new_pre, dtype=torch.int32),
                 torch.tensor(new_kvp, dtype=torch.int32), batch.hq, batch.hkv,
                 batch.d, batch.window, batch.sinks, batch.smooth, batch.scale,
                 batch.name + "/window-bounded", dict(batch.meta))


# ---------------------------------------------------------------- named sets

def tiny(seed: int = 0) -> Batch:
    """Single sequence, 256 tokens, no prefix, Hq=4 / Hkv=1, d=64, fp16,
    window 32, per-head sinks."""
    return make_batch([0], [256], 4, 1, 64, "f16", window=32, sink_mode="head",
                      seed=seed, name="tiny-w32")


def layer_pair(seq: int = 4096, seed: int = 1) -> List[Batch]:
    """gpt-oss layer pair, pure prefill: one full-causal and one window-128
    layer at Hq=64 / Hkv=8, d=64, bf16, per-head sinks."""
    full = make_batch([0], [seq], 64, 8, 64, "bf16", window=0,
                      sink_mode="head", seed=seed, name=f"pair-full-s{seq}")
    win = make_batch([0], [seq], 64, 8, 64, "bf16", window=128,
                     sink_mode="head", seed=seed + 100, name=f"pair-w128-s{seq}")
    return [full, win]


def chunked_prefix(num_seqs: int = 8, prefix: int = 8192, extend: int = 8192,
                   window: int = 128, seed: int = 2) -> Batch:
    """Chunked prefill over a cached prefix, full-prefix KV layout; pass the
    result through window_bounded() for the min(prefix, window) layout."""
    return make_batch([prefix] * num_seqs, [extend] * num_seqs, 64, 8, 64,
                      "bf16", window=window, sink_mode="head", seed=seed,
                      name=f"chunked-p{prefix}-e{extend}x{num_seqs}-w{window}")


def oss20b_chunk(layer: int, chunk: int, chunk_len: int = 512,
                 seed: int = 3) -> Batch:
    """One call of a gpt-oss-20b-like 16k prefill processed in chunks of 512:
    layer parity picks full-causal (even) or window-128 (odd); the prefix is
    the chunk_len * chunk tokens already processed."""
    window = 0 if layer % 2 == 0 else 128
    return make_batch([chunk_len * chunk], [chunk_len], 64, 8, 64, "bf16",
                      window=window, sink_mode="head",
                      seed=seed * 100003 + layer * 1009 + chunk,
                      name=f"oss20b-L{layer}-c{chunk}")


@dataclass
class PrefillStack:
    """The per-layer tensors of a chunked prefill, each kind stacked over the
    layers: q [layers, seq, Hq, d], k and v [layers, seq, Hkv, d] (one KV
    cache per layer, filled up to the current chunk).  Rows [c*L, (c+1)*L) of
    every layer are then evenly spaced in memory, so one strided copy moves a
    chunk of all layers."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    sinks: List[torch.Tensor]
    windows: List[int]
    chunk_len: int
    scale: float

    @property
    def num_layers(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_chunks(self) -> int:
        return int(self.q.shape[1]) // self.chunk_len

    def chunk_meta(self, chunk: int, device=None) -> torch.Tensor:
        """int32 [5] = (cu_seqlens_q[0:2], prefix_lens[0], kv_indptr[0:2]) of chunk."""
        L = self.chunk_len
        return torch.tensor([0, L, L * chunk, 0, L * (chunk + 1)], dtype=torch.int32,
                            device=device if device is not None else self.q.device)

    def call(self, chunk: int, layer: int, meta: Optional[torch.Tensor] = None) -> Batch:
        """Chunk `chunk` of layer `layer`: query rows [c*L, (c+1)*L) over the
        first (c+1)*L keys.  `meta` (from chunk_meta) holds the metadata; the
        batch's metadata tensors are views of it."""
        L = self.chunk_len
        lo, hi = chunk * L, (chunk + 1) * L
        m = meta if meta is not None else self.chunk_meta(chunk)
        return Batch(self.q[layer, lo:hi], self.k[layer, :hi], self.v[layer, :hi],
                     m[0:2], m[2:3], m[3:5], int(self.q.shape[2]), int(self.k.shape[2]),
                     int(self.q.shape[3]), self.windows[layer], self.sinks[layer], False,
                     self.scale, f"oss20b-L{layer}-c{chunk}",
                     {"max_seqlen_q": L, "extend_lens": [L]})


def oss20b_stack(num_layers: int = 24, seq: int = 16384, chunk_len: int = 512,
                 seed: int = 3, device="cpu") -> PrefillStack:
    """The tensors of a gpt-oss-20b-like prefill of `seq` tokens in chunks of
    `chunk_len`: layers alternate full-causal (even) and window-128 (odd),
    64/8 heads, d 64, bf16, per-head sinks; layer l draws from its own seed."""
    layers = [make_batch([0], [seq], 64, 8, 64, "bf16", window=0 if layer % 2 == 0 else 128,
                         sink_mode="head", seed=seed * 100003 + layer, device=device,
                         name=f"oss20b-L{layer}")
              for layer in range(num_layers)]
    st = PrefillStack(torch.stack([t.q for t in layers]), torch.stack([t.k for t in layers]),
                      torch.stack([t.v for t in layers]), [t.sinks for t in layers],
                      [t.window for t in layers], chunk_len, layers[0].scale)
    return st


def oss20b_prefill(num_layers: int = 24, seq: int = 16384, chunk_len: int = 512,
                   seed: int = 3, device="cpu") -> List[List[Batch]]:
    """The calls of a gpt-oss-20b-like prefill of `seq` tokens in chunks of
    `chunk_len`: calls[c][layer] for chunk c and layer (see oss20b_stack);
    chunk c is a view of query rows [c*chunk_len, (c+1)*chunk_len) over the
    first (c+1)*chunk_len keys of its layer."""
    st = oss20b_stack(num_layers, seq, chunk_len, seed, device)
    calls = []
    for c in range(st.num_chunks):
        meta = st.chunk_meta(c)
        calls.append([st.call(c, layer, meta) for layer in range(num_layers)])
    return calls


def pack_custom_mask(keep_rows):
    """Packs per-sequence boolean matrices keep_rows[b] [E_b, E_b] (row i,
    extend key j') into the custom-mask layout: 32-bit words, row i of
    sequence b at words mask_indptr[b] + i * W_b .. + W_b - 1 with
    W_b = ceil(E_b / 32), key j' at bit j' % 32 of word j' / 32.  Returns
    (words int32 tensor, mask_indptr int32 tensor [B+1])."""
    import numpy as np
    words, indptr = [], [0]
    for m in keep_rows:
        m = np.asarray(m, dtype=bool)
        e = m.shape[0]
        wb = (e + 31) // 32
        padded = np.zeros((e, wb * 32), dtype=bool)
        padded[:, :m.shape[1]] = m
        packed = np.packbits(padded, axis=1, bitorder="little")  # bytes, key j' at bit j' % 8
        words.append(np.ascontiguousarray(packed).view("<u4").reshape(-1))
        indptr.append(indptr[-1] + e * wb)
    flat = np.concatenate(words) if words else np.zeros(0, dtype=np.uint32)
    return (torch.from_numpy(flat.astype(np.uint32).view(np.int32).copy()),
            torch.tensor(indptr, dtype=torch.int32))


def random_custom_mask(extend_lens, density=0.7, seed=0, diagonal=True):
    """Seeded random keep matrices [E_b, E_b] per sequence (each entry kept
    with probability `density`; the diagonal kept when `diagonal`), the way a
    speculative-decoding draft tree hands its verify step an arbitrary
    ancestor mask."""
    import numpy as np
    rng = np.random.default_rng(int(seed))
    out = []
    for e in extend_lens:
        m = rng.random((e, e)) < density
        if diagonal:
            np.fill_diagonal(m, True)
        out.append(m)
    return out


def random_tree_mask(num_tokens, seed=0):
    """Keep matrix [n, n] of a seeded random draft tree: token t > 0 hangs
    under a parent drawn uniformly from tokens 0 .. t-1 and keeps exactly its
    ancestors and itself (the shape of a speculative-decoding verify step)."""
    import numpy as np
    rng = np.random.default_rng(int(seed))
    parent = [-1] + [int(rng.integers(0, t)) for t in range(1, num_tokens)]
    m = np.zeros((num_tokens, num_tokens), dtype=bool)
    for t in range(num_tokens):
        a = t
        while a >= 0:
            m[t, a] = True
            a = parent[a]
    return m


RAGGED_WINDOWS = [1, 15, 64, 127, 128, 129, 4096, 0]


def ragged(num_seqs: int = 16, max_prefix: int = 16384, max_extend: int = 8192,
           hq: int = 64, hkv: int = 8, d: int = 64, dtype: str = "bf16",
           window: int = 0, sink_mode: str = "head", seed: int = 4) -> Batch:
    """Ragged varlen batch: prefixes uniform in [0, max_prefix], extends
    uniform in [1, max_extend], drawn once per seed."""
    gen = torch.Generator().manual_seed(int(seed) * 7919 + 17)
    pre = torch.randint(0, max_prefix + 1, (num_seqs,), generator=gen).tolist()
    ext = torch.randint(1, max_extend + 1, (num_seqs,), generator=gen).tolist()
    return make_batch(pre, ext, hq, hkv, d, dtype, window=window,
                      sink_mode=sink_mode, seed=seed,
                      name=f"ragged-{num_seqs}-h{hq}/{hkv}-d{d}-{dtype}-w{window}-{sink_mode}")


def decode(num_seqs: int = 128, min_prefix: int = 1024, max_prefix: int = 16384,
           hq: int = 64, hkv: int = 8, d: int = 64, dtype: str = "bf16", window: int = 128,
           sink_mode: str = "head", seed: int = 6, window_bounded_layout: bool = False) -> Batch:
    """Decode step: one new token per sequence over a cached prefix drawn
    uniformly in [min_prefix, max_prefix] (once per seed).  With
    window_bounded_layout the batch carries only the last min(prefix, window)
    prefix rows of each sequence."""
    gen = torch.Generator().manual_seed(int(seed) * 104729 + 3)
    pre = torch.randint(min_prefix, max_prefix + 1, (num_seqs,), generator=gen).tolist()
    b = make_batch(pre, [1] * num_seqs, hq, hkv, d, dtype, window=window, sink_mode=sink_mode,
                   seed=seed, name=f"decode-{num_seqs}-h{hq}/{hkv}-d{d}-{dtype}-w{window}")
    return window_bounded(b, window) if (window_bounded_layout and window > 0) else b


@dataclass
class PagedBatch:
    """A Batch whose K/V also live in a page pool: page p of the pool holds
    page_size consecutive keys of one sequence; the pages are placed in a
    seeded random order, and unused pool pages hold noise."""
    batch: Batch
    k_pages: torch.Tensor    # [num_pages, page_size, Hkv, d]
    v_pages: torch.Tensor
    page_indptr: torch.Tensor   # int32 [B+1]
    page_indices: torch.Tensor  # int32 [entries]
    page_size: int

    def to(self, device) -> "PagedBatch":
        return PagedBatch(self.batch.to(device), self.k_pages.to(device),
                          self.v_pages.to(device), self.page_indptr.to(device),
                          self.page_indices.to(device), self.page_size)


def paged(batch: Batch, page_size: int, spare_pages: int = 3, seed: int = 0,
          shuffle: bool = True) -> PagedBatch:
    """Lay a contiguous batch's K/V out as a page pool, the pages placed in a
    seeded random order (shuffle) or in order (the keys and their order per
    sequence are unchanged: only the placement differs)."""
    gen = torch.Generator().manual_seed(int(seed) * 31337 + page_size)
    kvp = batch.kv_indptr.tolist()
    counts = [-(-(kvp[b + 1] - kvp[b]) // page_size) for b in range(batch.num_seqs)]
    n_used = sum(counts)
    num_pages = n_used + spare_pages
    order = torch.randperm(num_pages, generator=gen) if shuffle else torch.arange(num_pages)
    place = order[:n_used]  # pool page of each used page
    hkv, d = batch.k.shape[1], batch.k.shape[2]
    k_pages = torch.randn(num_pages, page_size, hkv, d, generator=gen).to(batch.k.dtype)
    v_pages = torch.randn(num_pages, page_size, hkv, d, generator=gen).to(batch.v.dtype)
    indptr, indices, u = [0], [], 0
    for b in range(batch.num_seqs):
        for pg in range(counts[b]):
            page = int(place[u])
            u += 1
            lo = kvp[b] + pg * page_size
            hi = min(lo + page_size, kvp[b + 1])
            k_pages[page, : hi - lo] = batch.k[lo:hi]
            v_pages[page, : hi - lo] = batch.v[lo:hi]
            indices.append(page)
        indptr.append(len(indices))
    return PagedBatch(batch, k_pages, v_pages, torch.tensor(indptr, dtype=torch.int32),
                      torch.tensor(indices, dtype=torch.int32), page_size)
