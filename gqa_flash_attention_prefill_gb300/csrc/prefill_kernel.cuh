// prefill_kernel.cuh -- persistent, warp-specialised fused GQA flash-attention
// prefill for sm_103a: TMA-fed K/V ring shared by the G query heads of a KV
// head, tcgen05 MMAs into tensor memory for S = Q K^T and O += P V, online
// exp2 softmax with the mask applied only on edge tiles, and the sink folded
// into the denominator in the epilogue.
//
// Operation: hip-ep PR #622 "perf(gqa): support sliding windows in the fused
// flash prefill kernel" (sink fold, window bound, start-tile clamp, NaN guard)
// and SGLang PR #34468 "gfx950 SWA prefix trim" (one floored KV loop over
// prefix and extend).  The AMD kernels on those pages are prior art only; the
// structure here is GB300-specific.
//
// A work unit is QT consecutive 128-row query tiles of one KV head (QT = 1
// or 2).  With QT = 2 both tiles walk the same key tiles, so every K/V tile
// brought into shared memory serves 256 rows: half the L2 traffic per flop of
// QT = 1, and one CTA per SM can keep a K/V ring twice as deep.
//
// CTA = 4*QT + 2 warps.  Warps 0 .. 4*QT-1: softmax + epilogue; warpgroup t
// (warps 4t .. 4t+3) owns query tile t, thread r of it row r (tensor-memory
// lane r, in that tile's own 256-column region).  Warp 4*QT: TMA producer.
// Warp 4*QT+1: tensor memory allocation and the single-thread MMA issuer.
//
// Row packing: row r of a query tile is query head g*G + (r % G) at query
// position q0 + r / G, which is the [token][head] order of q in memory, so
// one 3-D TMA box (d-chunk, G heads, 128/G tokens) fills the tile and every
// K/V tile is loaded once for all G heads of the group.
#pragma once
#include <cuda.h>
#include <cstdint>

#include "ptx.cuh"
#include "tile_math.cuh"

namespace gqa {

constexpr int kMaxSeqs = 512;        // sequences per launch (shared-memory tables)
static_assert((kMaxSeqs & (kMaxSeqs - 1)) == 0, "the dealing-order sort packs indices below kMaxSeqs");
// Threads per CTA with QT query tiles: a softmax warpgroup per tile, one
// producer warp and one MMA warp.
__host__ __device__ constexpr int threads_for(int QT) { return 32 * (4 * QT + 2); }
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy rescale: the running max used as the exponent reference is only moved
// when a row's max grows by more than this many powers of two; probabilities
// are then bounded by 2^8, and the final division by the same-referenced
// denominator makes the result exact regardless of the reference.
constexpr float kRescaleThreshold = 8.0f;

struct PrefillParams {
  CUtensorMap tmap_q;  // [total_q, Hq, d]  box (64, G, 128/G), 128B swizzle
  CUtensorMap tmap_k;  // [total_kv, Hkv, d] box (64, 1, BN)
  CUtensorMap tmap_v;
  CUtensorMap tmap_o;  // out, same geometry as tmap_q (TMA store of full units)
  const int32_t* cu_seqlens_q;
  const int32_t* prefix_lens;
  const int32_t* kv_indptr;
  const float* sinks;
  void* out;
  float* lse;
  int32_t* unit_log;
  unsigned int* status;
  int num_seqs, total_q, total_kv;
  // Index of this launch's first sequence in the caller's batch: a call with
  // more sequences than the shared-memory tables hold runs as several
  // launches over consecutive groups of sequences, each given metadata
  // pointers offset to its group.  cu_seqlens_q[0] == 0 is checked only in
  // the first group.
  int first_seq;
  int Hq, Hkv, G, rows;  // rows = query positions per 128-row query tile = 128 / G
  int window;            // <= 0: none
  int smooth;
  float scale_log2;      // scale * log2(e)
  unsigned long long timeout_ns;
  // Split-KV (num_splits > 1): work item i is split i % num_splits of unit
  // i / num_splits, a contiguous range of the unit's key tiles.  Items write
  // fp32 partials instead of out / lse; merge_kernel combines them.
  int num_splits;
  float* part_o;      // unnormalised O: [item][d/4][QT*128 rows][4]
  float* part_ml;     // (m in the log2 domain, l) per row: [item][QT*128][2]
  int32_t* part_hdr;  // [0] units; [4 + 4 u ..] (first q row, KV head, valid positions, 0)
  // Paged KV: K/V are a pool of num_pages pages of page_size tokens; the keys
  // of sequence b are the pages kv_page_indices[kv_indptr[b] ..] in order, and
  // tmap_k / tmap_v address the pool as rows page * page_size + slot with
  // boxes of page_rows = min(BN, page_size) rows.
  const int32_t* kv_page_indices;
  int page_size, num_pages, page_rows;
  // Custom mask (the MASK instantiation): per sequence a bitmap over its
  // extend keys, ANDed with the causal and window conditions; row i of
  // sequence b holds words custom_mask[mask_indptr[b] + i W ..] with
  // W = ceil(E / 32), extend key j' at bit j' % 32 of word j' / 32.
  const uint32_t* custom_mask;
  const int32_t* mask_indptr;
  long long total_mask_words;
  // Balanced split (the SK instantiation): the key tiles of all units, laid
  // end to end in dealing order, are cut into gridDim.x equal shares, one per
  // CTA.  A unit cut by share boundaries runs as pieces; each piece writes a
  // partial to part_o / part_ml slot 2c (CTA c's first piece) or 2c + 1 (its
  // last) and counts itself, per softmax warp, in sk_count[unit * 4 + warp];
  // the warp that completes a count merges those rows.  Count words carry
  // the launch's epoch in their upper 48 bits, so stale words count as zero.
  unsigned long long* sk_count;
  unsigned long long epoch;
  // The caller declared the metadata arrays (cu_seqlens_q, prefix_lens,
  // kv_indptr, mask_indptr) ready before this kernel starts: the prologue
  // reads them before waiting on the previous kernel in the stream.
  int metadata_ready;
};

__host__ __device__ constexpr int pow2_cols(int n) {
  return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}
// P buffers in tensor memory: two when the allocation does not grow (then
// the softmax of tile j only waits for the PV of tile j-2), else one.
__host__ __device__ constexpr int p_buffers(int D, int BN) {
  return pow2_cols(BN + BN + D) == pow2_cols(BN + BN / 2 + D) ? 2 : 1;
}
// S (BN fp32 columns) + P buffers (BN 16-bit values = BN/2 columns each) + O
// (D columns): one query tile's tensor memory.
__host__ __device__ constexpr int tmem_cols_for(int D, int BN) {
  return pow2_cols(BN + p_buffers(D, BN) * (BN / 2) + D);
}
// A CTA's allocation: two query tiles take 256 columns each.
__host__ __device__ constexpr int tmem_alloc_for(int D, int BN, int QT) {
  return QT == 1 ? tmem_cols_for(D, BN) : 512;
}

// Q tiles in flight per CTA: two for d = 64 (the next unit's Q loads during
// the current unit and two CTAs still fit on an SM), one for larger d.
__host__ __device__ constexpr int q_buffers(int D) { return D == 64 ? 2 : 1; }

__host__ __device__ constexpr uint32_t smem_bytes_for(int D, int BN, int NS, int QT) {
  return 1024u                                          // alignment slack
         + (uint32_t)q_buffers(D) * QT * 128u * D * 2u  // Q tiles
         + 2u * NS * BN * D * 2u                        // K and V rings
         + 64u * 8u                                     // mbarriers
         + 16u                                          // misc words
         + 4u * (5 * kMaxSeqs + 2)                      // per-sequence tables
         + 4u * 16u;                                    // scan scratch (one word per warp)
}

// Barrier indices.  Each query tile t has a block of 8 at kSub + 8 t.
template <int NS>
struct Bar {
  static constexpr int kQFull = 0, kQEmpty = 2;  // two each (Q double buffer)
  static constexpr int kKFull = 4, kKEmpty = 4 + NS, kVFull = 4 + 2 * NS, kVEmpty = 4 + 3 * NS;
  static constexpr int kSub = 4 + 4 * NS;
  static constexpr int kSFull = 0, kSFree = 1;  // offsets inside a query tile's block
  static constexpr int kPFull = 2, kODone = 4;  // one per P buffer
  static constexpr int kEpi = 6;                // output tile staged in shared memory
  static constexpr int kDrain = kSub + 16;
  static constexpr int kCount = kDrain + 1;
};

struct Unit {
  int b, g, q0, q_last, P, E, kv_base, q_row0, kv_lo, n_tiles;
  int id;  // unit number (differs from the work item under split-KV)
};

// Per-sequence metadata copied into shared memory once per CTA, so that
// decoding a unit never waits on global memory.
struct SeqTab {
  const int32_t* tile_start;  // [B+1] exclusive scan of units per sequence, in dealing order
  const int32_t* cu0;         // [B+1] cu_seqlens_q
  const int32_t* pre;         // [B]   prefix_lens
  const int32_t* kvb;         // [B]   kv_indptr (first key row)
  const int32_t* order;       // [B]   sequence dealt r-th
};

// Unit u -> (sequence, KV head, unit of `urows` query positions).  Units are
// numbered with the KV head fastest, sequences in their dealing order and,
// inside a sequence, the last (costliest under causality) unit first.
__device__ __forceinline__ Unit decode_unit(const PrefillParams& p, const SeqTab& T, int u,
                                            int BN, int urows) {
  Unit U;
  U.g = u % p.Hkv;
  const int tau = u / p.Hkv;
  int lo = 0, hi = p.num_seqs;  // find r with tile_start[r] <= tau < tile_start[r+1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (T.tile_start[mid] <= tau) lo = mid; else hi = mid;
  }
  const int t = tau - T.tile_start[lo];
  const int tiles_b = T.tile_start[lo + 1] - T.tile_start[lo];
  const int b = T.order[lo];
  U.b = b;
  U.q0 = (tiles_b - 1 - t) * urows;
  U.P = T.pre[b];
  const int cu0 = T.cu0[b];
  U.E = T.cu0[b + 1] - cu0;
  U.q_last = min(U.q0 + urows, U.E) - 1;
  U.q_row0 = cu0 + U.q0;
  U.kv_base = T.kvb[b];
  const KvRange r = kv_range(U.P, U.q0, U.q_last, p.window, BN);
  U.kv_lo = r.kv_lo;
  U.n_tiles = r.n_tiles;
  return U;
}

// Work item -> unit and key-tile range.  Without split-KV an item is a unit;
// with it, split s of S takes the unit's tiles [s n / S, (s + 1) n / S), which
// may be empty when the unit has fewer than S tiles.
template <bool SPL>
__device__ __forceinline__ Unit decode_item(const PrefillParams& p, const SeqTab& T, int item,
                                            int BN, int urows) {
  if (!SPL) {
    Unit U = decode_unit(p, T, item, BN, urows);
    U.id = item;
    return U;
  }
  const int S = p.num_splits;
  const int unit = item / S, s = item - unit * S;
  Unit U = decode_unit(p, T, unit, BN, urows);
  U.id = unit;
  const int n = U.n_tiles;  // n * S < 2^31: at most 16 splits of a KV range below 2^27 tiles
  const int t0 = s * n / S, t1 = (s + 1) * n / S;
  U.kv_lo += t0 * BN;
  U.n_tiles = t1 - t0;
  return U;
}

// Issues the TMA loads of key tile [n0, n0 + BN) of unit U into `dst`
// (kv_chunk bytes per 64-column chunk, NCH chunks).  Contiguous KV: one box
// per chunk at row kv_base + n0.  Paged KV: BN / page_rows boxes per chunk,
// each from the page that holds its first key.  The tile's page numbers are
// read from the page table just before its copies, all of them before the
// first copy (prefetching them a tile ahead, into registers or into L1,
// measured slower); a box starting past the sequence's last key
// (masked keys of its last tile) reads the last page, and a page number
// outside the pool raises GQA_DEV_BAD_METADATA and reads page 0.
template <bool PAGED, int BN, int NCH>
__device__ __forceinline__ void load_kv_tile(const PrefillParams& p, const Unit& U, int n0,
                                             const CUtensorMap* tmap, uint32_t dst,
                                             uint32_t kv_chunk, uint32_t bar) {
  if constexpr (!PAGED) {
    for (int c = 0; c < NCH; ++c)
      tma_load_3d(dst + c * kv_chunk, tmap, bar, c * 64, U.g, U.kv_base + n0);
  } else {
    const int ps = p.page_size, boxr = p.page_rows;
    const int npg = (U.P + U.E + ps - 1) / ps;  // the sequence's pages
    if (boxr >= BN) {  // one box (page_size >= BN): one lookup
      int pg = __ldg(p.kv_page_indices + U.kv_base + min(n0 / ps, npg - 1));
      if (pg < 0 || pg >= p.num_pages) {
        atomicOr(p.status, 2u);  // GQA_DEV_BAD_METADATA
        pg = 0;
      }
      for (int c = 0; c < NCH; ++c)
        tma_load_3d(dst + c * kv_chunk, tmap, bar, c * 64, U.g, pg * ps + n0 % ps);
      return;
    }
    // All the tile's page numbers are loaded before the first copy, so their
    // latencies overlap (a box is at least 8 rows: at most BN / 8 boxes).
    constexpr int kMaxBoxes = BN / 8;
    int pgs[kMaxBoxes];
#pragma unroll
    for (int i = 0; i < kMaxBoxes; ++i)
      if (i * boxr < BN)
        pgs[i] = __ldg(p.kv_page_indices + U.kv_base + min((n0 + i * boxr) / ps, npg - 1));
#pragma unroll
    for (int i = 0; i < kMaxBoxes; ++i) {
      const int sub = i * boxr;
      if (sub >= BN) break;
      int pg = pgs[i];
      if (pg < 0 || pg >= p.num_pages) {
        atomicOr(p.status, 2u);  // GQA_DEV_BAD_METADATA
        pg = 0;
      }
      const int row = pg * ps + (n0 + sub) % ps;
      for (int c = 0; c < NCH; ++c)
        tma_load_3d(dst + c * kv_chunk + (uint32_t)sub * 128u, tmap, bar, c * 64, U.g, row);
    }
  }
}

// ---------------------------------------------------------------- balanced split
// A CTA's share of the key tiles is walked as pieces: the rest of the unit
// its share starts in (from local tile t0), the whole units after it, and
// the head of the unit its share ends in.
struct SkWalk {
  int u, t0, rem;  // next unit, its first tile, tiles left in the share
};

// Next piece of the walk: U is its unit with the key range narrowed to the
// piece's tiles [t0, t1); false when the share is used up.
__device__ __forceinline__ bool sk_next(const PrefillParams& p, const SeqTab& T, SkWalk& w, int BN,
                                        int urows, Unit& U) {
  if (w.rem <= 0) return false;
  U = decode_unit(p, T, w.u, BN, urows);
  U.id = w.u;
  const int t1 = min(U.n_tiles, w.t0 + w.rem);
  U.kv_lo += w.t0 * BN;
  U.n_tiles = t1 - w.t0;
  w.rem -= t1 - w.t0;
  w.u += 1;
  w.t0 = 0;
  return true;
}

// Share boundaries: CTA c of C takes global tiles [lo(c), lo(c + 1)) with
// lo(c) = floor(c W / C) = c q + floor(c r / C), q = W / C, r = W % C, in
// 32-bit arithmetic (c q <= W < 2^31 and c r < C^2 < 2^31 for C < 46341).
struct SkShares {
  int C, q, r;
  __device__ __forceinline__ SkShares(int W, int C_) : C(C_), q(W / C_), r(W - (W / C_) * C_) {}
  __device__ __forceinline__ int lo(int c) const {
    return c * q + (int)((unsigned)(c * r) / (unsigned)C);
  }
};

// Counts one piece of a unit (for one warp's rows) and returns the count
// including it.  The word holds epoch << 16 | count; a word tagged with
// another epoch (memory never written, or a launch that did not finish)
// counts as zero, and so does 0, the value a completed count is reset to.
// `guess` is the word's expected value (0: this piece is expected first).
// Lock-free: a failed compare-and-swap means another piece counted first.
// After 2^20 failed attempts (not expected: at most a few pieces race) the
// device status is raised and -1 returned (no merge).
__device__ __forceinline__ int sk_arrive(unsigned long long* word, unsigned long long epoch,
                                         unsigned long long guess, unsigned int* status) {
  unsigned long long old = guess;
  for (int n = 0; n < (1 << 20); ++n) {
    const unsigned long long cnt = (old >> 16) == epoch ? (old & 0xffffull) : 0ull;
    const unsigned long long got = atomicCAS(word, old, (epoch << 16) | (cnt + 1ull));
    if (got == old) return (int)(cnt + 1ull);
    old = got;
  }
  atomicOr(status, 1u);  // GQA_DEV_TIMEOUT
  return -1;
}

// Exclusive scan of a[0, n) in place by all nthreads threads of the CTA
// (contiguous segments per thread, warp scans, then the warp totals);
// a[n] receives the total.  `warp_tot` holds one word per warp.
__device__ __forceinline__ void cta_exclusive_scan(int32_t* a, int n, int32_t* warp_tot, int tid,
                                                   int nthreads) {
  const int per = (n + nthreads - 1) / nthreads;
  const int i0 = min(tid * per, n), i1 = min(i0 + per, n);
  int local = 0;
  for (int i = i0; i < i1; ++i) local += a[i];
  int incl = local;
  const int lane = tid & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[tid >> 5] = incl;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < nthreads / 32; ++w) {
      const int v = warp_tot[w];
      warp_tot[w] = acc;
      acc += v;
    }
    a[n] = acc;
  }
  __syncthreads();
  int acc = warp_tot[tid >> 5] + incl - local;
  for (int i = i0; i < i1; ++i) {
    const int v = a[i];
    a[i] = acc;
    acc += v;
  }
  __syncthreads();
}

// Custom-mask bits of a 64-key chunk for one query row: bit c is set when key
// jp0 + c of the extend part (jp0 may be negative: the chunk's first -jp0
// keys are prefix keys, which the mask does not cover) is kept.  `row` is
// the row's W words; words past the row's last are never needed (keys past
// the row's own position are masked causally), so reads clamp to it.
__device__ __forceinline__ uint64_t custom_keep_bits(const uint32_t* row, int W, int jp0) {
  if (jp0 + 64 <= 0) return ~0ull;
  const int lo = jp0 > 0 ? jp0 : 0;
  const int off = lo - jp0;  // prefix keys at the chunk's start (< 64)
  const int w0 = lo >> 5, sh = lo & 31;
  const uint32_t a = __ldg(row + min(w0, W - 1));
  const uint32_t b = __ldg(row + min(w0 + 1, W - 1));
  const uint32_t c = __ldg(row + min(w0 + 2, W - 1));
  uint64_t bits = (((uint64_t)b << 32) | a) >> sh;
  if (sh != 0) bits |= (uint64_t)c << (64 - sh);
  return off == 0 ? bits : ((bits << off) | ((1ull << off) - 1ull));
}

// k-th unit of this CTA: round k of a snake (boustrophedon) deal over the
// grid, so that with units ordered by decreasing cost every CTA alternates
// between the expensive and the cheap end of each round.
__device__ __forceinline__ int unit_of(int k) {
  const int g = gridDim.x, c = blockIdx.x;
  return k * g + ((k & 1) ? (g - 1 - c) : c);
}

// Bounded mbarrier wait.  Returns false (and raises the abort flag and the
// device status) when the phase does not complete within the time limit or
// when another role of this CTA has aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile uint32_t* abort_flag,
                                             unsigned int* status,
                                             unsigned long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1u;
        atomicOr(status, 1u);  // GQA_DEV_TIMEOUT
        return false;
      }
    }
  }
}

}  // namespace gqa

namespace gqa {

// Loads issued into ring slot s when `total` loads went round the ring in
// order (slot t % NS).  The paged instantiation drains with this instead of
// per-slot counters: those sit in local memory (the slot index is dynamic),
// and on the paged producer path, with a page lookup per box, that round
// trip measured 6-9% of the kernel's time.  The contiguous instantiations
// keep the counters, which measured faster for them.
template <int NS>
__device__ __forceinline__ uint32_t slot_loads(int s, uint32_t total) {
  return total / NS + ((uint32_t)s < total % NS ? 1u : 0u);
}

// Bounded wait used while draining at exit: ignores the abort flag, because
// its purpose is to let copies and MMAs already in flight land before the CTA
// releases its shared and tensor memory.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity,
                                           unsigned long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return;
    if ((n & 255u) == 0 && globaltimer_ns() - t0 > timeout_ns) return;
  }
}


// Dealing order of a batch's sequences, costliest first: keys[b] holds
// sequence b's costliest-unit tile count (-1: no units) and order[r]
// receives the sequence dealt r-th.  Sequences are sorted by decreasing key,
// ties by index, so the long units of every sequence go out before any
// short one (inside a sequence the units are already dealt costliest
// first).  A batch whose keys all lie within a factor of two (a windowed
// decode step) keeps its order: there the deal order does not matter.  The
// sort is a bitonic sort, descending, of the composites key * 512 +
// (511 - index) (keys clamped to 2^22 - 1; the padding up to a power of two
// holds -1 and sorts last).  Called by every thread of the CTA; `scratch`
// is two shared words.  deal_order keeps it out of line, so that the kernel
// body, and with it the placement of its hot loops, does not depend on it;
// the paged instantiation inlines it (a call there measured 10% slower on
// 16-token pages, where the page lookups run on the producer warp).
__device__ __forceinline__ void deal_order_body(const int32_t* keys, int32_t* order,
                                                int32_t* scratch, int nseq, int tid,
                                                int nthreads) {
  if (tid == 0) {
    scratch[0] = 0x7fffffff;
    scratch[1] = -1;
  }
  __syncthreads();
  int kmin = 0x7fffffff, kmax = -1;
  for (int b = tid; b < nseq; b += nthreads) {
    const int k = keys[b];
    if (k >= 0) {
      kmin = min(kmin, k);
      kmax = max(kmax, k);
    }
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if ((tid & 31) == 0) {
    atomicMin(&scratch[0], kmin);
    atomicMax(&scratch[1], kmax);
  }
  __syncthreads();
  if (scratch[1] < 2 * max(scratch[0], 1)) return;  // uniform: every thread reads the same words
  int n = 2;
  while (n < nseq) n <<= 1;
  for (int i = tid; i < n; i += nthreads)
    order[i] = i < nseq ? min(max(keys[i], 0), (1 << 22) - 1) * kMaxSeqs + (kMaxSeqs - 1 - i) : -1;
  for (int size = 2; size <= n; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = tid; i < n / 2; i += nthreads) {
        const int lo = 2 * stride * (i / stride) + (i % stride), hi = lo + stride;
        const bool desc = (lo & size) == 0;  // direction of this bitonic run
        const int x = order[lo], y = order[hi];
        if ((x < y) == desc) {
          order[lo] = y;
          order[hi] = x;
        }
      }
    }
  }
  __syncthreads();
  for (int r = tid; r < nseq; r += nthreads) order[r] = kMaxSeqs - 1 - (order[r] & (kMaxSeqs - 1));
  __syncthreads();
}
static __device__ __noinline__ void deal_order(const int32_t* keys, int32_t* order, int32_t* scratch,
                                               int nseq, int tid, int nthreads) {
  deal_order_body(keys, order, scratch, nseq, tid, nthreads);
}

// SPL: split-KV work items writing partials; PAGED: K/V from a page pool;
// MASK: the custom mask ANDed into the causal / window mask; SK: balanced
// split (equal shares of all key tiles per CTA, cut units merged in-kernel).
// Each is a separate instantiation, so the default kernel carries none of
// their code.
template <int D, int BN, int NS, bool WIN, bool BF16, int MINB, int QT, bool SPL, bool PAGED,
          bool MASK = false, bool SK = false>
__global__ void __launch_bounds__(threads_for(QT), MINB)
    prefill_kernel(const __grid_constant__ PrefillParams p) {
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
  static_assert(!MASK || (BN != 96 && !SPL && !PAGED && QT == 1), "custom-mask shapes");
  static_assert(!SK || (BN != 96 && !SPL && !PAGED && !MASK && QT == 1), "balanced-split shapes");
  static_assert(BN == 64 || BN == 96 || BN == 128, "key tile");
  static_assert(QT == 1 || (QT == 2 && tmem_cols_for(D, BN) <= 256), "query tiles per CTA");
  constexpr int kThr = threads_for(QT);
  constexpr int kSmWarps = 4 * QT;  // softmax warps
  constexpr int kProdWarp = kSmWarps, kMmaWarp = kSmWarps + 1;
  constexpr int NCH = D / 64;  // 128-byte swizzle chunks along d
  constexpr uint32_t kQBytes = 128u * D * 2u;  // one 128-row query tile
  constexpr uint32_t kKVBytes = (uint32_t)BN * D * 2u;
  constexpr uint32_t kQChunk = 128u * 128u;
  constexpr uint32_t kKVChunk = (uint32_t)BN * 128u;
  constexpr uint32_t kTmemCols = (uint32_t)tmem_alloc_for(D, BN, QT);
  constexpr uint32_t kSubCols = 256u;  // tensor-memory columns between query tiles
  constexpr uint32_t NP = (uint32_t)p_buffers(D, BN);
  constexpr uint32_t kColS = 0, kColP = BN, kColO = BN + NP * (BN / 2);
  constexpr uint32_t kIdescS = idesc_f16(BF16, 128, BN, false);  // Q, K both K-major
  constexpr uint32_t kIdescO = idesc_f16(BF16, 128, D, true);    // V is MN-major
  using B = Bar<NS>;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr uint32_t NQ = (uint32_t)q_buffers(D);  // Q buffers, each holding QT tiles
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + NQ * QT * kQBytes;
  const uint32_t sV = sK + NS * kKVBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NQ * QT * kQBytes + 2 * NS * kKVBytes);
  const uint32_t sBar = smem_u32(bars);
  uint32_t* misc = reinterpret_cast<uint32_t*>(bars + 64);  // [0] tmem base, [1] abort, [2] bad
  int32_t* tile_start = reinterpret_cast<int32_t*>(misc + 4);
  int32_t* seq_cu0 = tile_start + (kMaxSeqs + 1);
  int32_t* seq_pre = seq_cu0 + (kMaxSeqs + 1);
  int32_t* seq_kvb = seq_pre + kMaxSeqs;
  int32_t* seq_order = seq_kvb + kMaxSeqs;
  int32_t* scan = seq_order + kMaxSeqs;
  const SeqTab T{tile_start, seq_cu0, seq_pre, seq_kvb, seq_order};
  volatile uint32_t* abort_flag = misc + 1;
  const unsigned long long tmo = p.timeout_ns;
  const int win = WIN ? p.window : 0;
  const int urows = QT * p.rows;  // query positions per unit

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---------------------------------------------------------------- set-up
  // A second CTA of a kernel that allocates tensor memory is launched on an
  // SM only once the resident CTA has relinquished its allocation permit
  // (measured on GB300: the second wave starts right after it), so an
  // allocation after the prologue holds each SM's second CTA back by the
  // prologue's length (about 2.5 us).  The balanced split allocates first:
  // its shares are equal, so its second wave sets the call's end (chunk 31
  // of the 16k prefill 139.3 -> 135.9 us).  The other kernels allocate after
  // the prologue: allocating first made back-to-back full-causal calls 2-3%
  // slower under programmatic dependent launch (with earlier relinquishing,
  // the next call's CTAs pair up on the SMs that free first, and the costliest
  // units are dealt to the lowest CTAs).
  constexpr bool kEarlyTmem = SK;
  if (kEarlyTmem && warp == kMmaWarp) {
    tmem_alloc(smem_u32(misc), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < B::kCount; ++i) {
      uint32_t cnt = 1u;
      for (int t = 0; t < QT; ++t) {
        const int o = i - (B::kSub + 8 * t);
        if (o == B::kSFree || o == B::kPFull || o == B::kPFull + 1 || o == B::kEpi) cnt = 128u;
      }
      // A Q buffer is free once the unit's last QK^T is done (MMA commit) and
      // each query tile's epilogue has finished staging its output through it.
      if (i == B::kQEmpty || i == B::kQEmpty + 1) cnt = 1u + QT;
      mbar_init(sBar + 8u * i, cnt);
    }
    misc[1] = 0u;
    misc[2] = 0u;
    fence_barrier_init();
  }
  if (warp == kProdWarp && lane == 0) {
    tma_prefetch_desc(&p.tmap_q);
    tma_prefetch_desc(&p.tmap_k);
    tma_prefetch_desc(&p.tmap_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t tmem = kEarlyTmem ? misc[0] : 0u;
  // CTAs that end before any MMA hand early-allocated tensor memory back.
  auto release_tmem = [&]() {
    if (kEarlyTmem && warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  };
  // Everything above touches only this CTA's own shared memory and the
  // kernel parameters, so under programmatic dependent launch it overlaps
  // the previous kernel's tail.  The next kernel in the stream may start its
  // own set-up as soon as this grid's CTAs finish.  Nothing reads device
  // memory before the previous kernel's writes are visible, except, when the
  // caller declares them ready (metadata_ready), the metadata arrays the
  // prologue below reads; no global write comes before the wait either way.
  grid_dep_launch_dependents();
  if (!p.metadata_ready) grid_dep_wait();

  // Per-sequence tables and metadata checks (bad metadata: write nothing,
  // raise GQA_DEV_BAD_METADATA), the order in which sequences are dealt, and
  // the exclusive scan of their unit counts in that order.
  const int nseq = p.num_seqs;
  const int per = (nseq + kThr - 1) / kThr;
  const int b_lo = min(tid * per, nseq), b_hi = min(b_lo + per, nseq);
  bool bad = (tid == 0) && p.first_seq == 0 && (__ldg(p.cu_seqlens_q) != 0);
  for (int b = b_lo; b < b_hi; ++b) {
    const int c0 = __ldg(p.cu_seqlens_q + b), c1 = __ldg(p.cu_seqlens_q + b + 1);
    const int P = __ldg(p.prefix_lens + b);
    const int k0 = __ldg(p.kv_indptr + b), k1 = __ldg(p.kv_indptr + b + 1);
    const int E = c1 - c0;
    // KV rows (contiguous) or pages (paged) of the sequence: exactly P + E keys.
    const long long kv_need =
        PAGED ? ((long long)P + E + p.page_size - 1) / p.page_size : (long long)P + E;
    int key = -1;  // tiles of the sequence's costliest (last) unit; -1: no units
    bool mask_bad = false;
    if constexpr (MASK) {  // the sequence's bitmap: E rows of ceil(E / 32) words
      const long long m0 = __ldg(p.mask_indptr + b), m1 = __ldg(p.mask_indptr + b + 1);
      mask_bad = m0 < 0 || m1 > p.total_mask_words ||
                 m1 - m0 != (long long)E * ((E + 31) / 32);
    }
    if (E < 0 || P < 0 || c0 < 0 || c1 > p.total_q || k0 < 0 || k1 > p.total_kv ||
        (long long)k1 - k0 != kv_need || mask_bad)
      bad = true;
    else if (E > 0)
      key = kv_range(P, ((E - 1) / urows) * urows, E - 1, win, BN).n_tiles;
    seq_cu0[b] = c0;
    seq_pre[b] = P;
    seq_kvb[b] = k0;
    seq_order[b] = b;
    tile_start[b] = key;  // the keys wait here until the scan below
    if (b == nseq - 1) seq_cu0[nseq] = c1;
  }
  if (bad) misc[2] = 1u;
  __syncthreads();
  // Costliest sequences first (deal_order); one call whatever the batch, so
  // the kernel body stays the same size.
  if (nseq > 1) {
    if constexpr (PAGED)
      deal_order_body(tile_start, seq_order, scan + 14, nseq, tid, kThr);
    else
      deal_order(tile_start, seq_order, scan + 14, nseq, tid, kThr);
  }
  // Units per sequence in dealing order, then their exclusive scan: warp
  // scans, then warp totals.  tile_start[r] is the first unit (of one KV
  // head) of the r-th sequence dealt.
  auto units_of = [&](int b) {
    const int E = seq_cu0[b + 1] - seq_cu0[b];
    return E > 0 ? (E + urows - 1) / urows : 0;
  };
  int local = 0;
  for (int r = b_lo; r < b_hi; ++r) local += units_of(seq_order[r]);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int w = 0; w < kThr / 32; ++w) {
      const int v = scan[w];
      scan[w] = acc;
      acc += v;
    }
    tile_start[nseq] = acc;
  }
  __syncthreads();
  {
    int acc = scan[warp] + incl - local;
    for (int r = b_lo; r < b_hi; ++r) {
      tile_start[r] = acc;
      acc += units_of(seq_order[r]);
    }
  }
  __syncthreads();
  // This CTA's work, still from shared memory only: the units (times the
  // split count under split-KV), whether the CTA has any, the balanced
  // split's share, and the tensor memory.  With metadata_ready all of it
  // runs before the wait on the previous kernel, so each SM's second CTA is
  // not held back by the wait (it starts once this one has relinquished its
  // tensor-memory allocation permit).  Global writes (the bad-metadata
  // report, the split-KV header) come after the wait.
  const bool bad_meta = misc[2] != 0u;
  const int n_units = tile_start[nseq] * p.Hkv * (SPL ? p.num_splits : 1);
  bool run = !bad_meta && (SK || (int)blockIdx.x < n_units);
  // Balanced split: the key tiles of every query tile (in dealing order) into
  // the K/V rings, still unused, their exclusive scan, and this CTA's share:
  // sk[0] first unit, sk[1] its first tile, sk[2] tiles, sk[3] global index of
  // the first tile, sk[4] W (the host keeps W below 2^31 and the query tiles
  // within the rings).  Skipped on bad metadata, whose counts are not bounded.
  int32_t* const sk = scan + 8;
  if constexpr (SK) {
    static_assert(kThr / 32 <= 8, "scan words 8..12 hold the share");
    if (run) {
      int32_t* qn = reinterpret_cast<int32_t*>(smem + NQ * QT * kQBytes);
      const int nq = tile_start[nseq];
      for (int q = tid; q < nq; q += kThr) qn[q] = decode_unit(p, T, q * p.Hkv, BN, urows).n_tiles;
      __syncthreads();
      cta_exclusive_scan(qn, nq, scan, tid, kThr);
      if (tid == 0) {
        const int W = p.Hkv * qn[nq], c = blockIdx.x;
        const SkShares sh(W, (int)gridDim.x);
        const int lo = sh.lo(c), hi = sh.lo(c + 1);
        sk[0] = 0;
        sk[1] = 0;
        if (hi > lo) {  // query tile holding global tile lo: Hkv qn[a] <= lo < Hkv qn[a + 1]
          int a = 0, b = nq;
          while (b - a > 1) {
            const int mid = (a + b) >> 1;
            if (p.Hkv * qn[mid] <= lo) a = mid; else b = mid;
          }
          const int off = lo - p.Hkv * qn[a], n = qn[a + 1] - qn[a];  // n >= 1
          sk[0] = a * p.Hkv + off / n;
          sk[1] = off % n;
        }
        sk[2] = hi - lo;
        sk[3] = lo;
        sk[4] = W;
      }
      fence_proxy_async_smem();  // the rings were written here; TMA writes them next
      __syncthreads();
      run = sk[2] > 0;  // false: an empty share (fewer tiles than CTAs)
    }
  }
  if constexpr (!kEarlyTmem) {
    if (run) {
      if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(misc), kTmemCols);
        tmem_relinquish();
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      tmem = misc[0];
    }
  }
  if (p.metadata_ready) grid_dep_wait();  // before the first global write or other read
  if (bad_meta) {
    if (tid == 0) {
      atomicOr(p.status, 2u);  // GQA_DEV_BAD_METADATA
      if (SPL && blockIdx.x == 0) p.part_hdr[0] = 0;  // nothing to merge
    }
    release_tmem();
    return;
  }
  if (SPL && blockIdx.x == 0 && tid == 0) p.part_hdr[0] = tile_start[nseq] * p.Hkv;
  if (!run) {  // nothing for this CTA
    release_tmem();
    return;
  }

  // ---------------------------------------------------------------- producer
  // Two lanes of the producer warp, each with its own bounded waits: lane 0
  // walks the CTA's key tiles loading each unit's Q tiles and then its K
  // tiles, lane 1 walks the same tiles loading V.  K therefore runs as far
  // ahead as its ring allows (a K slot frees when its QK^T is done), however
  // late a V slot frees (when its PV is done).
  // One producer lane for the paged and the plain windowed instantiations,
  // two for the others (measured: one lane is 4-5% faster on windowed calls
  // and 0.4-0.7% slower on full-causal ones).
  constexpr bool kOneLane = PAGED || (WIN && !SPL && !SK && !MASK);
  if (warp == kProdWarp && kOneLane) {
    // One lane issues Q, K and V in the order the MMA warp consumes them (a
    // unit's Q, K0, K1, V0, K2, V1, ..., its last V, then the next unit's Q),
    // so every wait is for a slot freed by an MMA issued before anything this
    // lane issues later.  Paged KV: a tile's page numbers are fetched for its
    // K copy and again, from L1, for its V copy one step later; with two
    // lanes of one warp each fetching them, the divergent lanes' dependent
    // loads stalled each other.  (Prefetching the next tile's entries into L1
    // a step ahead measured 17% slower on 16-token pages.)
    if (lane == 0) {
      uint32_t nq = 0, itk = 0, itv = 0;
      bool ok = true;
      auto load_v = [&](const Unit& U, int j) -> bool {
        const uint32_t s = itv % NS, ph = (itv / NS) & 1u;
        if (!wait_bounded(sBar + 8u * (B::kVEmpty + s), ph ^ 1u, abort_flag, p.status, tmo))
          return false;
        mbar_arrive_expect_tx(sBar + 8u * (B::kVFull + s), kKVBytes);
        load_kv_tile<PAGED, BN, NCH>(p, U, U.kv_lo + j * BN, &p.tmap_v, sV + s * kKVBytes,
                                     kKVChunk, sBar + 8u * (B::kVFull + s));
        ++itv;
        return true;
      };
      for (int kk = 0; ok; ++kk) {
        const int uk = unit_of(kk);
        if (uk >= n_units) break;
        const Unit U = decode_item<SPL>(p, T, uk, BN, urows);
        const uint32_t qb = nq % NQ;
        if (!(ok = wait_bounded(sBar + 8u * (B::kQEmpty + qb), ((nq / NQ) & 1u) ^ 1u, abort_flag,
                                p.status, tmo)))
          break;
        mbar_arrive_expect_tx(sBar + 8u * (B::kQFull + qb), QT * kQBytes);
        for (int t = 0; t < QT; ++t)
          for (int c = 0; c < NCH; ++c)
            tma_load_3d(sQ + (qb * QT + t) * kQBytes + c * kQChunk, &p.tmap_q,
                        sBar + 8u * (B::kQFull + qb), c * 64, U.g * p.G, U.q_row0 + t * p.rows);
        ++nq;
        for (int j = 0; j < U.n_tiles; ++j, ++itk) {
          const uint32_t s = itk % NS, ph = (itk / NS) & 1u;
          if (!(ok = wait_bounded(sBar + 8u * (B::kKEmpty + s), ph ^ 1u, abort_flag, p.status, tmo)))
            break;
          mbar_arrive_expect_tx(sBar + 8u * (B::kKFull + s), kKVBytes);
          load_kv_tile<PAGED, BN, NCH>(p, U, U.kv_lo + j * BN, &p.tmap_k, sK + s * kKVBytes,
                                       kKVChunk, sBar + 8u * (B::kKFull + s));
          if (j > 0 && !(ok = load_v(U, j - 1))) break;
        }
        if (ok) ok = load_v(U, U.n_tiles - 1);
      }
      // Let every copy issued land before the CTA can exit.
      for (uint32_t b = 0; b < NQ; ++b) {
        if (nq > b) {
          const uint32_t last = nq - 1u - b;
          wait_drain(sBar + 8u * (B::kQFull + last % NQ), (last / NQ) & 1u, tmo);
        }
      }
      for (int s = 0; s < NS; ++s) {
        const uint32_t nk = slot_loads<NS>(s, itk), nv = slot_loads<NS>(s, itv);
        if (nk > 0) wait_drain(sBar + 8u * (B::kKFull + s), (nk - 1u) & 1u, tmo);
        if (nv > 0) wait_drain(sBar + 8u * (B::kVFull + s), (nv - 1u) & 1u, tmo);
      }
    }
    __syncwarp();
  }
  if (warp == kProdWarp && !kOneLane) {
    if (lane == 0) {
      uint32_t nq = 0, nk[NS];
      for (int s = 0; s < NS; ++s) nk[s] = 0u;
      uint32_t itk = 0;
      SkWalk wk{};
      if constexpr (SK) wk = SkWalk{sk[0], sk[1], sk[2]};
      for (int kk = 0;; ++kk) {
        Unit U;
        if constexpr (SK) {
          if (!sk_next(p, T, wk, BN, urows, U)) break;
        } else {
          const int uk = unit_of(kk);
          if (uk >= n_units) break;
          U = decode_item<SPL>(p, T, uk, BN, urows);
        }
        if (SPL && U.n_tiles == 0) continue;  // empty split: no loads, no Q buffer
        const uint32_t qb = nq % NQ;
        if (!wait_bounded(sBar + 8u * (B::kQEmpty + qb), ((nq / NQ) & 1u) ^ 1u, abort_flag,
                          p.status, tmo))
          break;
        mbar_arrive_expect_tx(sBar + 8u * (B::kQFull + qb), QT * kQBytes);
        // A query tile past the end of q (a unit's second tile at the end of
        // the batch) reads the tensor map's zero fill; its rows are never stored.
        for (int t = 0; t < QT; ++t)
          for (int c = 0; c < NCH; ++c)
            tma_load_3d(sQ + (qb * QT + t) * kQBytes + c * kQChunk, &p.tmap_q,
                        sBar + 8u * (B::kQFull + qb), c * 64, U.g * p.G, U.q_row0 + t * p.rows);
        ++nq;
        bool ok = true;
        for (int j = 0; j < U.n_tiles; ++j, ++itk) {
          const uint32_t s = itk % NS, ph = (itk / NS) & 1u;
          if (!(ok = wait_bounded(sBar + 8u * (B::kKEmpty + s), ph ^ 1u, abort_flag, p.status, tmo)))
            break;
          mbar_arrive_expect_tx(sBar + 8u * (B::kKFull + s), kKVBytes);
          load_kv_tile<PAGED, BN, NCH>(p, U, U.kv_lo + j * BN, &p.tmap_k, sK + s * kKVBytes,
                                       kKVChunk, sBar + 8u * (B::kKFull + s));
          if constexpr (!PAGED) ++nk[s];
        }
        if (!ok) break;
      }
      // Let every copy issued land before the CTA can exit.
      for (uint32_t b = 0; b < NQ; ++b) {
        if (nq > b) {
          const uint32_t last = nq - 1u - b;  // the last load into buffer (last % NQ)
          wait_drain(sBar + 8u * (B::kQFull + last % NQ), (last / NQ) & 1u, tmo);
        }
      }
      for (int s = 0; s < NS; ++s) {
        const uint32_t n = PAGED ? slot_loads<NS>(s, itk) : nk[s];
        if (n > 0) wait_drain(sBar + 8u * (B::kKFull + s), (n - 1u) & 1u, tmo);
      }
    } else if (lane == 1) {
      uint32_t nv[NS];
      for (int s = 0; s < NS; ++s) nv[s] = 0u;
      uint32_t itv = 0;
      bool ok = true;
      SkWalk wk{};
      if constexpr (SK) wk = SkWalk{sk[0], sk[1], sk[2]};
      for (int kv = 0; ok; ++kv) {
        Unit U;
        if constexpr (SK) {
          if (!sk_next(p, T, wk, BN, urows, U)) break;
        } else {
          const int uv = unit_of(kv);
          if (uv >= n_units) break;
          U = decode_item<SPL>(p, T, uv, BN, urows);
        }
        for (int j = 0; j < U.n_tiles; ++j, ++itv) {
          const uint32_t s = itv % NS, ph = (itv / NS) & 1u;
          if (!(ok = wait_bounded(sBar + 8u * (B::kVEmpty + s), ph ^ 1u, abort_flag, p.status, tmo)))
            break;
          mbar_arrive_expect_tx(sBar + 8u * (B::kVFull + s), kKVBytes);
          load_kv_tile<PAGED, BN, NCH>(p, U, U.kv_lo + j * BN, &p.tmap_v, sV + s * kKVBytes,
                                       kKVChunk, sBar + 8u * (B::kVFull + s));
          if constexpr (!PAGED) ++nv[s];
        }
      }
      for (int s = 0; s < NS; ++s) {
        const uint32_t n = PAGED ? slot_loads<NS>(s, itv) : nv[s];
        if (n > 0) wait_drain(sBar + 8u * (B::kVFull + s), (n - 1u) & 1u, tmo);
      }
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- MMA issuer
  // The whole warp runs this loop (the MMA helpers issue from one elected
  // lane), so the waits, the loop and the descriptors stay warp-uniform.
  if (warp == kMmaWarp) {
    // Q and K: K-major, 128-byte swizzle; the 16-wide k-step advances the
    // start address by 32 bytes inside a 128-byte swizzle row, the 64-wide
    // d-chunk by one chunk.  Stride between 8-row groups: 1024 bytes.
    // V: MN-major (d contiguous), 128-byte swizzle; a 16-key step is two
    // 8-key groups = 2048 bytes; d-chunks of 64 are kKVChunk apart.
    // Shared-memory addresses stay below 2^18, so moving a descriptor to
    // another buffer or k-step is an add to its start-address field.
    const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024);
    const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024);
    const uint64_t dV0 = smem_desc_sw128(sV, kKVChunk, 1024);
    auto kstep = [](int kk, uint32_t chunk) -> uint64_t {
      return (uint64_t)(((uint32_t)(kk >> 2) * chunk + (uint32_t)(kk & 3) * 32u) >> 4);
    };
    auto sub_bar = [&](int t, int o) { return sBar + 8u * (B::kSub + 8 * t + o); };
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort_flag, p.status, tmo));
    };
    // O_t += P_t V for every query tile t, once V and that tile's P are in.
    auto issue_pv = [&](uint32_t itp, bool first) -> bool {
      const uint32_t sp = itp % NS, php = (itp / NS) & 1u;
      if (!wait_all(sBar + 8u * (B::kVFull + sp), php)) return false;
      const uint32_t pb = itp % NP;
      const uint64_t dv = dV0 + sp * (kKVBytes >> 4);
      for (int t = 0; t < QT; ++t) {
        if (!wait_all(sub_bar(t, B::kPFull + pb), (itp / NP) & 1u)) return false;
        tc_fence_after();
        const uint32_t tb = tmem + t * kSubCols;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tb + kColO, tb + kColP + pb * (BN / 2) + kk * 8, dv + (uint64_t)(kk * 128),
                 kIdescO, (first && kk == 0) ? 0u : 1u);
        mma_commit(sub_bar(t, B::kODone + pb));
      }
      mma_commit(sBar + 8u * (B::kVEmpty + sp));
      return true;
    };
    uint32_t it = 0, uc = 0;
    bool ok = true;
    int u;
    Unit Un;
    SkWalk wk{};
    if constexpr (SK) {  // u: 0 while a piece is decoded ahead, n_units after the last
      wk = SkWalk{sk[0], sk[1], sk[2]};
      u = sk_next(p, T, wk, BN, urows, Un) ? 0 : n_units;
    } else {
      u = unit_of(0);
      if (u < n_units) Un = decode_item<SPL>(p, T, u, BN, urows);
    }
    for (int k = 0; ok && u < n_units; ++k) {
      const Unit U = Un;  // decoded one unit ahead: its loads overlap this unit
      if constexpr (SK) {
        u = sk_next(p, T, wk, BN, urows, Un) ? 0 : n_units;
      } else {
        const int u_next = unit_of(k + 1);
        if (u_next < n_units) Un = decode_item<SPL>(p, T, u_next, BN, urows);
        u = u_next;
      }
      if (SPL && U.n_tiles == 0) continue;  // empty split: nothing to issue
      const uint32_t qb = uc % NQ;
      if (!(ok = wait_all(sBar + 8u * (B::kQFull + qb), (uc / NQ) & 1u))) break;
      for (int j = 0; j < U.n_tiles; ++j) {
        const uint32_t cur = it + j;
        const uint32_t s = cur % NS, ph = (cur / NS) & 1u;
        const uint64_t dk = dK0 + s * (kKVBytes >> 4);
        if (!(ok = wait_all(sBar + 8u * (B::kKFull + s), ph))) break;
        for (int t = 0; t < QT && ok; ++t) {
          if (cur > 0 && !(ok = wait_all(sub_bar(t, B::kSFree), (cur - 1u) & 1u))) break;
          tc_fence_after();
          const uint64_t dq = dQ0 + (qb * QT + t) * (kQBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + t * kSubCols + kColS, dq + kstep(kk, kQChunk), dk + kstep(kk, kKVChunk),
                   kIdescS, kk > 0 ? 1u : 0u);
          mma_commit(sub_bar(t, B::kSFull));
        }
        if (!ok) break;
        mma_commit(sBar + 8u * (B::kKEmpty + s));
        if (j == U.n_tiles - 1) mma_commit(sBar + 8u * (B::kQEmpty + qb));
        // PV of the previous tile goes after this tile's QK^T, so the
        // tensor core works on S(j) while the softmax warps work on S(j-1).
        if (j > 0 && !(ok = issue_pv(cur - 1u, j == 1))) break;
      }
      if (ok) ok = issue_pv(it + U.n_tiles - 1u, U.n_tiles == 1);
      it += U.n_tiles;
      ++uc;
    }
    mma_commit(sBar + 8u * B::kDrain);  // completes when every MMA issued is done
    wait_drain(sBar + 8u * B::kDrain, 0u, tmo);
    __syncwarp();
  }

  // ---------------------------------------------------------------- softmax + epilogue
  if (warp < kSmWarps) {
    const int sub = warp >> 2;        // query tile of this warpgroup
    const int r = (warp & 3) * 32 + lane;  // tile row == tensor-memory lane
    const bool leader = r == 0;       // first thread of the warpgroup
    const uint32_t t_lane = tmem + sub * kSubCols + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t bsub = sBar + 8u * (B::kSub + 8 * sub);  // this tile's barrier block
    const float sl2 = p.scale_log2;
    uint32_t it = 0;
    bool ok = true;
    bool release_pending = false;  // Q buffer to hand back after the next P store
    uint32_t release_qb = 0;
    uint32_t n_full = 0;  // units whose output went through the TMA store
    uint32_t kq = 0;      // non-empty items done (they take Q buffers in turn)
    constexpr bool split = SPL;
    const int part_rows = QT * 128;  // partial rows per work item
    const int rr = sub * 128 + r;     // this thread's partial row
    int u;
    Unit Un;
    float sink_next = 0.f;
    SkWalk wk{};
    if constexpr (SK) {  // u: 0 while a piece is decoded ahead, n_units after the last
      wk = SkWalk{sk[0], sk[1], sk[2]};
      u = sk_next(p, T, wk, BN, urows, Un) ? 0 : n_units;
    } else {
      u = unit_of(0);
    }
    if (u < n_units) {
      if constexpr (!SK) Un = decode_item<SPL>(p, T, u, BN, urows);
      if (p.sinks != nullptr) sink_next = __ldg(p.sinks + Un.g * p.G + r % p.G);
    }
    for (int k = 0; ok && u < n_units; ++k) {
      // Unit metadata and the sink are fetched one unit ahead, so their
      // global-memory latency overlaps the previous unit.
      const Unit U = Un;
      const int cur_u = u;
      const float sink = sink_next;
      if constexpr (SK) {
        u = sk_next(p, T, wk, BN, urows, Un) ? 0 : n_units;
      } else {
        u = unit_of(k + 1);
      }
      if (u < n_units) {
        if constexpr (!SK) Un = decode_item<SPL>(p, T, u, BN, urows);
        if (p.sinks != nullptr) sink_next = __ldg(p.sinks + Un.g * p.G + r % p.G);
      }
      if (split && leader && sub == 0) {  // where the merge writes this unit's rows
        int32_t* hd = p.part_hdr + 4 + 4 * (size_t)U.id;
        hd[0] = U.q_row0;
        hd[1] = U.g;
        hd[2] = U.q_last - U.q0 + 1;
        hd[3] = 0;
      }
      if (split && U.n_tiles == 0) {  // empty split: a record the merge gives weight 0
        reinterpret_cast<float2*>(p.part_ml)[(size_t)cur_u * part_rows + rr] =
            make_float2(-INFINITY, 0.f);
        continue;
      }
      const uint32_t qb = (SPL ? kq : (uint32_t)k) % NQ;  // this unit's Q buffer
      ++kq;
      // This warpgroup's query tile: positions [q0s, qls] (empty when qls < q0s,
      // a unit's second tile past the end of its sequence).
      const int q0s = U.q0 + sub * p.rows;
      const int qls = min(q0s + p.rows, U.E) - 1;
      const int pl = q0s + r / p.G;  // query position inside the sequence
      const int h = U.g * p.G + r % p.G;
      const int pos = U.P + pl;
      const uint32_t* mrow = nullptr;  // this row's custom-mask words
      int mwords = 0;
      if constexpr (MASK) {
        mwords = (U.E + 31) / 32;
        if (pl <= qls)
          mrow = p.custom_mask + __ldg(p.mask_indptr + U.b) + (long long)pl * mwords;
      }
      float m = -INFINITY;  // exponent reference (log2 domain)
      float l = 0.f;        // running denominator, relative to m
      int n_masked = 0;     // tiles of the unit needing the mask (tile_needs_mask)
      for (int j = 0; j < U.n_tiles; ++j, ++it) {
        const int n0 = U.kv_lo + j * BN;
        ok = __all_sync(0xffffffffu,
                        wait_bounded(bsub + 8u * B::kSFull, it & 1u, abort_flag, p.status, tmo));
        if (!ok) break;
        tc_fence_after();
        // The S row is processed in 64-column chunks so that only one chunk
        // of fp32 scores is live in registers; the packed 16-bit P of earlier
        // chunks (half the size) waits in registers until the tile is done.
        // Edge tests are uniform over the warpgroup: the causal edge (a key
        // past the tile's first position) and the window edge (a key below
        // the tile's last position's lower bound).
        const bool edge_c = n0 + BN - 1 > U.P + q0s;
        const bool edge_w = WIN && n0 < U.P + qls - win + 1;
        const bool edge_m = MASK && n0 + BN - 1 >= U.P;  // the tile reaches the extend keys
        n_masked += tile_needs_mask(n0, BN, U.P, U.q0, U.q_last, win) ? 1 : 0;
        // S is processed in CW-column chunks (64, or 48 for 96-key tiles).
        constexpr int CW = (BN == 96) ? 48 : 64;
        constexpr int NCK = BN / CW;
        uint32_t pk[BN / 2];
        float alpha = 1.f;  // product of this tile's reference moves
        bool upd_any = false;
#pragma unroll
        for (int ch = 0; ch < NCK; ++ch) {
          uint32_t sr[64];
          // The reducing load also yields the row maximum of each 32-column
          // half; it stands for the chunk maximum on tiles without a mask.
          float red0 = tmem_ld32_max(t_lane + kColS + ch * CW, *reinterpret_cast<uint32_t(*)[32]>(sr));
          float red1 = -INFINITY;
          if constexpr (CW == 64)
            red1 = tmem_ld32_max(t_lane + kColS + ch * CW + 32,
                                 *reinterpret_cast<uint32_t(*)[32]>(sr + 32));
          else
            tmem_ld16(t_lane + kColS + ch * CW + 32, *reinterpret_cast<uint32_t(*)[16]>(sr + 32));
          tmem_wait_ld();
          if (ch == NCK - 1) {
            tc_fence_before();
            mbar_arrive(bsub + 8u * B::kSFree);  // S is in registers: next QK^T may overwrite it
          }
          // Per-element mask on edge tiles only: row `pos` keeps columns
          // [c_lo, c_hi] of this chunk; one-sided tiles test one bound.
          const int c_hi = pos - (n0 + ch * CW);
          const int c_lo = pos - win + 1 - (n0 + ch * CW);
          if (edge_c && edge_w) {
#pragma unroll
            for (int c = 0; c < CW; ++c)
              if (c > c_hi || c < c_lo) sr[c] = __float_as_uint(-INFINITY);
          } else if (edge_c) {
            if (c_hi < CW - 1) {
#pragma unroll
              for (int c = 0; c < CW; ++c)
                if (c > c_hi) sr[c] = __float_as_uint(-INFINITY);
            }
          } else if (edge_w) {
            if (c_lo > 0) {
#pragma unroll
              for (int c = 0; c < CW; ++c)
                if (c < c_lo) sr[c] = __float_as_uint(-INFINITY);
            }
          }
          if constexpr (MASK) {
            if (edge_m && mrow != nullptr) {
              const uint64_t keep = custom_keep_bits(mrow, mwords, n0 + ch * CW - U.P);
#pragma unroll
              for (int c = 0; c < CW; ++c)
                if (!((keep >> c) & 1ull)) sr[c] = __float_as_uint(-INFINITY);
            }
          }
          float mx = fmaxf(red0, red1);
          if (CW != 64 || edge_c || edge_w || edge_m) {
            // Masked (or 48-column) chunk: maximum over the kept values, over
            // independent chains (short dependency chains).
            float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < CW; c += 8) {
              mx0 = max3(mx0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
              mx1 = max3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
              mx2 = max3(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
              mx3 = max3(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
            }
            mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
          }
          const float m_cand = mx * sl2;
          if (m_cand > m + kRescaleThreshold) {  // move the reference (rare after the first tile)
            const float a = ex2(m - m_cand);     // m = -inf gives 0
            alpha *= a;
            l *= a;
            m = m_cand;
            upd_any = true;
#pragma unroll
            for (int i = 0; i < ch * (CW / 2); ++i) {  // earlier chunks of this tile
              const float lo = unpack_lo<BF16>(pk[i]) * a, hi = unpack_hi<BF16>(pk[i]) * a;
              pk[i] = pack2<BF16>(lo, hi);
            }
          }
          // NaN guard: a row that has seen no key keeps m = -inf; its scores
          // are all -inf, and with a zero offset every probability is exactly 0.
          const float neg_m = (m == -INFINITY) ? 0.f : -m;
          const uint64_t sc2 = f2(sl2, sl2), nm2 = f2(neg_m, neg_m);
          uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;  // packed partial sums
#pragma unroll
          for (int c = 0; c < CW; c += 8) {
            float x[8];
#pragma unroll
            for (int t = 0; t < 8; t += 2)
              unf2(ffma2(f2(__uint_as_float(sr[c + t]), __uint_as_float(sr[c + t + 1])), sc2, nm2),
                   x[t], x[t + 1]);
#pragma unroll
            for (int t = 0; t < 8; ++t) x[t] = ex2(x[t]);
            acc0 = fadd2(acc0, f2(x[0], x[1]));
            acc1 = fadd2(acc1, f2(x[2], x[3]));
            acc2 = fadd2(acc2, f2(x[4], x[5]));
            acc3 = fadd2(acc3, f2(x[6], x[7]));
#pragma unroll
            for (int t = 0; t < 8; t += 2)
              pk[ch * (CW / 2) + (c + t) / 2] = pack2<BF16>(x[t], x[t + 1]);
          }
          float r0, r1;
          unf2(fadd2(fadd2(acc0, acc1), fadd2(acc2, acc3)), r0, r1);
          l += r0 + r1;
        }

        // P buffer `pb` is rewritten once the PV that last read it is done.
        const uint32_t pb = it % NP;
        if (it >= NP)
          ok = __all_sync(0xffffffffu, wait_bounded(bsub + 8u * (B::kODone + pb),
                                                     ((it / NP) & 1u) ^ 1u, abort_flag, p.status,
                                                     tmo));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < BN / 64; ++c)
          tmem_st32(t_lane + kColP + pb * (BN / 2) + c * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(pk + c * 32));
        if constexpr (BN == 96)  // the last 16 packed columns
          tmem_st16(t_lane + kColP + pb * (BN / 2) + 32,
                    *reinterpret_cast<uint32_t(*)[16]>(pk + 32));
        const bool corr = upd_any && j > 0;
        if (__any_sync(0xffffffffu, corr)) {
          // Rescaling O needs every earlier PV done (PVs complete in order).
          if (NP > 1) {
            const uint32_t prev = it - 1u;
            ok = __all_sync(0xffffffffu,
                            wait_bounded(bsub + 8u * (B::kODone + prev % NP), (prev / NP) & 1u,
                                         abort_flag, p.status, tmo));
            if (!ok) break;
            tc_fence_after();
          }
          const float a = corr ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(t_lane + kColO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
            tmem_st32(t_lane + kColO + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bsub + 8u * (B::kPFull + pb));
        if (release_pending && leader) {
          // The previous unit's output store has read its staging buffer by now
          // (or shortly); hand that Q buffer back to the producer.
          bulk_wait_group_read0();
          mbar_arrive(sBar + 8u * (B::kQEmpty + release_qb));
          release_pending = false;
        }
      }
      if (!ok) break;

      // Epilogue: fold the sink into the denominator, normalise, store.
      ok = __all_sync(0xffffffffu, wait_bounded(bsub + 8u * (B::kODone + (it - 1u) % NP),
                                                 ((it - 1u) / NP) & 1u, abort_flag, p.status, tmo));
      if (!ok) break;
      tc_fence_after();
      if constexpr (SK) {
        // A cut unit runs as pieces: the one holding the unit's first tiles
        // (the last piece of its share) owns the unit, the later ones (each
        // the first piece of a later share) contribute.
        const int t0 = k == 0 ? sk[1] : 0;
        const int n_all = kv_range(U.P, U.q0, U.q_last, win, BN).n_tiles;
        if (t0 != 0 || U.n_tiles != n_all) {
          // A piece of a cut unit.  Each warp counts the piece for its 32 rows
          // in the unit's count word, after publishing its partial (O relative
          // to m, unnormalised, and (m, l)) to slot 2c (this CTA's first piece)
          // or 2c + 1 (its last); the warp whose count completes the unit's
          // pieces merges those rows with the log-sum-exp combine and writes
          // them.  No CTA waits on another.  The piece holding the unit's first
          // tiles (the last piece of its CTA, normally the last to finish) first
          // tries to complete the count without publishing: if every other
          // piece has counted, it merges at once.
          const SkShares sh(sk[4], (int)gridDim.x);
          const int gu = sk[3] + (int)(it - (uint32_t)U.n_tiles) - t0;  // the unit's first tile
          int c0 = (int)blockIdx.x, c1 = (int)blockIdx.x;
          while (sh.lo(c0) > gu) --c0;
          while (sh.lo(c1 + 1) <= gu + n_all - 1) ++c1;
          auto nonempty = [&](int c) { return sh.lo(c + 1) > sh.lo(c); };
          int npieces = 0;
          for (int c = c0; c <= c1; ++c) npieces += nonempty(c) ? 1 : 0;
          unsigned long long* word = p.sk_count + (size_t)U.id * 4 + (warp & 3);
          unsigned long long seen = 0ull;  // lane 0: the count word as last read
          int last = 0;
          if (t0 == 0 && lane == 0) {
            const unsigned long long want = (p.epoch << 16) | (unsigned long long)(npieces - 1);
            seen = atomicCAS(word, want, want + 1ull);
            last = seen == want;
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          if (!last) {
            const int slot = 2 * (int)blockIdx.x + (k == 0 ? 0 : 1);
            float4* po = reinterpret_cast<float4*>(p.part_o) + (size_t)slot * (D / 4) * 128;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(t_lane + kColO + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                po[(size_t)(c * 8 + i) * 128 + r] =
                    make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
            }
            reinterpret_cast<float2*>(p.part_ml)[(size_t)slot * 128 + r] = make_float2(m, l);
            fence_acq_rel_gpu();  // release: the partial before the count that publishes it
            __syncwarp();
            int cnt = 0;
            if (lane == 0) cnt = sk_arrive(word, p.epoch, seen, p.status);
            last = __shfl_sync(0xffffffffu, cnt == npieces ? 1 : 0, 0);
          }
          tc_fence_before();
          __syncwarp();
          if (leader) mbar_arrive(sBar + 8u * (B::kQEmpty + qb));  // nothing staged in Q
          if (!last) continue;  // another piece merges these rows
          if (lane == 0) fence_acq_rel_gpu();  // acquire: the other pieces' partials
          __syncwarp();
          // Merge in share order c0..c1 whichever piece merges (this piece's
          // values equal its partial's), so the result is the same run to run:
          // per 32 output columns, each piece's (m, l) and O loaded together
          // (one round trip to L2 per piece) and combined online against a
          // running maximum.
          auto slot_of = [&](int c) { return 2 * c + (sh.lo(c) >= gu ? 0 : 1); };
          const bool has_x = (p.sinks != nullptr) || (p.smooth != 0);
          const float ms = sink * kLog2e;  // 0 in smooth mode
          const float2* pml = reinterpret_cast<const float2*>(p.part_ml);
          const bool valid = pl <= qls;
          const size_t orow = (size_t)(U.q_row0 + sub * p.rows + r / p.G) * p.Hq + h;
          uint16_t* op = reinterpret_cast<uint16_t*>(p.out) + orow * D;
          float lse2 = -INFINITY;
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            float acc[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = 0.f;
            float M = -INFINITY, dsum = 0.f;
            // Uniform over the warp (tcgen05.ld is warp-wide); a piece that saw
            // no key of a row has m = -inf there and adds nothing.
            for (int c = c0; c <= c1; ++c) {
              if (!nonempty(c)) continue;
              float2 v;
              uint32_t x[32];
              if (c == (int)blockIdx.x) {
                v = make_float2(m, l);
                tmem_ld32(t_lane + kColO + cc * 32, x);
                tmem_wait_ld();
              } else {
                const size_t sc = (size_t)slot_of(c);
                const float4* src = reinterpret_cast<const float4*>(p.part_o) + sc * (D / 4) * 128;
                v = __ldcg(pml + sc * 128 + r);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                  const float4 f = __ldcg(src + (size_t)(cc * 8 + i) * 128 + r);
                  x[4 * i] = __float_as_uint(f.x);
                  x[4 * i + 1] = __float_as_uint(f.y);
                  x[4 * i + 2] = __float_as_uint(f.z);
                  x[4 * i + 3] = __float_as_uint(f.w);
                }
              }
              float a_run = 1.f, a_new = 0.f;
              if (v.x != -INFINITY) {
                if (v.x > M) {
                  a_run = (M == -INFINITY) ? 0.f : ex2(M - v.x);
                  a_new = 1.f;
                  M = v.x;
                } else {
                  a_new = ex2(v.x - M);
                }
              }
              dsum = dsum * a_run + v.y * a_new;
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = acc[i] * a_run + __uint_as_float(x[i]) * a_new;
            }
            // Fold the sink in once: den against mf = max(M, sink log2 e).
            float scl = 0.f;
            if (M != -INFINITY) {
              const float mf = has_x ? fmaxf(M, ms) : M;
              const float a = ex2(M - mf);
              float den = dsum * a + (has_x ? ex2(ms - mf) : 0.f);
              den = fmaxf(den, 1e-30f);
              scl = a / den;
              lse2 = mf + log2f(den);
            }
            if (valid) {
              uint4* dst = reinterpret_cast<uint4*>(op + cc * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pack2<BF16>(acc[8 * i] * scl, acc[8 * i + 1] * scl),
                                    pack2<BF16>(acc[8 * i + 2] * scl, acc[8 * i + 3] * scl),
                                    pack2<BF16>(acc[8 * i + 4] * scl, acc[8 * i + 5] * scl),
                                    pack2<BF16>(acc[8 * i + 6] * scl, acc[8 * i + 7] * scl));
            }
          }
          if (valid && p.lse != nullptr) p.lse[orow] = lse2 * kLn2;
          // Every piece has counted: zero the word (count 0 under any epoch),
          // so that the next launch, or a replay of this one (same epoch, e.g.
          // from a CUDA graph), starts from zero.
          if (lane == 0) *word = 0ull;
          continue;
        }
      }
      if constexpr (split) {
        // Partial of one key range: O relative to m, unnormalised, with (m, l);
        // float4 (c4, row) order so that a warp's stores are contiguous.
        float4* po = reinterpret_cast<float4*>(p.part_o) + (size_t)cur_u * (D / 4) * part_rows;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(t_lane + kColO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            po[(size_t)(c * 8 + i) * part_rows + rr] =
                make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                            __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
        }
        reinterpret_cast<float2*>(p.part_ml)[(size_t)cur_u * part_rows + rr] = make_float2(m, l);
        // Nothing staged in the Q buffer: hand it back once the O reads are done.
        tc_fence_before();
        __syncwarp();
        if (leader) mbar_arrive(sBar + 8u * (B::kQEmpty + qb));
        continue;
      }
      const bool has_x = (p.sinks != nullptr) || (p.smooth != 0);
      const float ms = sink * kLog2e;  // 0 in smooth mode
      float inv = 0.f, lse2 = -INFINITY;
      if (m != -INFINITY) {
        // Same value as l + exp2(ms - m) over the m-referenced sums, computed
        // against max(m, ms) so that a large sink cannot overflow.
        const float mf = has_x ? fmaxf(m, ms) : m;
        const float a = ex2(m - mf);
        float den = l * a + (has_x ? ex2(ms - mf) : 0.f);
        den = fmaxf(den, 1e-30f);
        inv = a / den;
        lse2 = mf + log2f(den);
      }
      const bool valid = pl <= qls;
      const int row0 = U.q_row0 + sub * p.rows;  // first q row of this query tile
      const size_t orow = (size_t)(row0 + r / p.G) * p.Hq + h;
      // A query tile whose rows all belong to its sequence is staged in its
      // own Q buffer (the unit's last QK^T is done) in the 128-byte-swizzled
      // layout of the output tensor map and written by one TMA store; a
      // ragged tail tile stores its valid rows directly.
      const bool full = (qls - q0s + 1) == p.rows;
      const uint32_t stage = sQ + (qb * QT + sub) * kQBytes;
      uint16_t* op = reinterpret_cast<uint16_t*>(p.out) + orow * D;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {  // 64 columns per round trip
        uint32_t o[64];
        tmem_ld32(t_lane + kColO + c * 64, *reinterpret_cast<uint32_t(*)[32]>(o));
        tmem_ld32(t_lane + kColO + c * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(o + 32));
        tmem_wait_ld();
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i)
          w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        if (full) {
          // 16-byte unit i of a 128-byte row sits at i ^ (row % 8) under the swizzle.
          const uint32_t row_addr = stage + c * kQChunk + (uint32_t)r * 128u;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_shared_v4(row_addr + ((uint32_t)(i ^ (r & 7)) << 4), w[4 * i], w[4 * i + 1],
                         w[4 * i + 2], w[4 * i + 3]);
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(op + c * 64);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      if (full) {
        fence_proxy_async_smem();  // generic-proxy writes -> visible to the TMA store
        mbar_arrive(bsub + 8u * B::kEpi);
        if (leader) {
          if (!wait_bounded(bsub + 8u * B::kEpi, n_full & 1u, abort_flag, p.status, tmo)) {
            ok = false;
          } else {
            for (int c = 0; c < NCH; ++c)
              tma_store_3d(&p.tmap_o, stage + c * kQChunk, c * 64, U.g * p.G, row0);
            bulk_commit_group();
          }
        }
        ++n_full;
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      if (valid && p.lse != nullptr) p.lse[orow] = lse2 * kLn2;
      if (leader) {
        if (NQ == 1) {
          bulk_wait_group_read0();
          mbar_arrive(sBar + 8u * (B::kQEmpty + qb));
        } else {
          release_pending = true;
          release_qb = qb;
        }
      }
      if (p.unit_log != nullptr && leader && sub == 0) {
        int32_t* rec = p.unit_log + 8 * (size_t)cur_u;
        rec[0] = U.b;
        rec[1] = U.g;
        rec[2] = U.q0;
        rec[3] = U.kv_lo;
        rec[4] = U.n_tiles;
        rec[5] = n_masked;
        rec[6] = (int)blockIdx.x;
        rec[7] = k;
      }
    }
    if (leader) {
      bulk_wait_group0();  // every output store complete before the CTA exits
      if (release_pending) mbar_arrive(sBar + 8u * (B::kQEmpty + release_qb));
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace gqa
