// tile_math.cuh -- the KV range a work unit walks.
//
// A work unit covers query positions [q0, q_last] of one sequence (all G query
// heads of one KV head).  Keys are tiled in blocks of BN counted from the
// sequence's first key, one loop over [cached prefix | extend]
// (SGLang PR #34468 "gfx950 SWA prefix trim", commit 2: one loop, one floor).
//
// Lower end (the loop floor): with a window w the lowest key any row of the
// unit may see is P + q0 - w + 1 (row q0 has the smallest lower bound, since
// the bound grows with the position: hip-ep PR #622 window commit), and the
// first tile that can hold a kept element is the BN-aligned tile containing
// it (SGLang commit 1: floor(A / BN) * BN, tight for every residue).  Without
// a window the loop starts at key 0.
//
// Upper end: the last real row q_last sees keys up to P + q_last (causal), so
// the loop stops at tile ceil((P + q_last + 1 - kv_lo) / BN).
//
// A tile needs the per-element mask only when some (real row, key) pair in it
// is masked: a key above the first row's position (causal edge) or, with a
// window, a key below the last row's lower bound (window edge).
#pragma once

namespace gqa {

struct KvRange {
  int kv_lo;    // first key of the first tile walked (multiple of BN)
  int n_tiles;  // tiles walked
};

__host__ __device__ __forceinline__ KvRange kv_range(int P, int q0, int q_last, int window,
                                                     int BN) {
  int lo = 0;
  if (window > 0) {
    const int a = P + q0 - window + 1;  // lowest key row q0 can see
    lo = a > 0 ? (a / BN) * BN : 0;
  }
  const int hi = P + q_last + 1;  // one past the last key row q_last can see
  KvRange r;
  r.kv_lo = lo;
  r.n_tiles = (hi - lo + BN - 1) / BN;
  return r;
}

// True when tile [n0, n0 + BN) holds a masked (real row, key) pair.
__host__ __device__ __forceinline__ bool tile_needs_mask(int n0, int BN, int P, int q0,
                                                         int q_last, int window) {
  if (n0 + BN - 1 > P + q0) return true;                      // causal edge
  if (window > 0 && n0 < P + q_last - window + 1) return true;  // window edge
  return false;
}

}  // namespace gqa
