// merge.cu -- split-KV merge: combines the fp32 partials that the split work
// items of one unit wrote (each over a contiguous range of the unit's key
// tiles) into out and lse, folding the sink in once.
//
// Split s of a row carries O_s (relative to its own reference m_s, log2
// domain) and l_s = sum of exp2(s' - m_s) over its keys.  With
// mf = max(max_s m_s, sink * log2 e) (the sink only when present):
//   den = sum_s l_s exp2(m_s - mf) + [sink] exp2(sink * log2 e - mf)
//   out = sum_s O_s exp2(m_s - mf) / den,   lse = (mf + log2 den) ln 2,
// the log-sum-exp combine of partial softmax results (the lse_extend merge of
// SGLang PR #34468's context-parallel path), and for one split the same value
// the unsplit epilogue computes.  A row no split saw (all m_s = -inf) gets
// out = 0, lse = -inf, as in the unsplit kernel.
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"

namespace gqa {

namespace {

struct MergeParams {
  const float* part_o;
  const float* part_ml;
  const int32_t* part_hdr;
  const float* sinks;
  void* out;
  float* lse;
  int num_splits, Hq, G, rows, part_rows, smooth;
};

// Columns per thread, as float4 groups: a thread merges one row's
// col_group<D>() float4 columns (8 values at d = 64, else 16), so a unit's
// rows spread over d / 8 or d / 16 blocks; the smaller group at d = 64 gives
// the short merges there twice the blocks (4-sequence decode 31.4 -> 28.8 us).
template <int D>
__host__ __device__ constexpr int col_group() { return D == 64 ? 2 : 4; }
// The largest split count the library accepts.
constexpr int kMaxMergeSplits = 16;

// Block = the 128 rows of one partial query tile for one group of output
// columns (thread = row, so every partial load of a warp is 32 consecutive
// float4s).  Grid = units x query tiles per unit x column groups; blocks past
// the units the split kernel recorded return at once.
template <int D, bool BF16>
__global__ void __launch_bounds__(128) merge_kernel(const __grid_constant__ MergeParams mp) {
  constexpr int kColGroup = col_group<D>();
  constexpr int kGroups = D / 4 / kColGroup;
  const int grp = blockIdx.x % kGroups;
  const int tile = blockIdx.x / kGroups;
  const int tiles_per_unit = mp.part_rows / 128;
  const int unit = tile / tiles_per_unit;
  if (unit >= mp.part_hdr[0]) return;
  const int32_t* hd = mp.part_hdr + 4 + 4 * (size_t)unit;
  const int row0 = hd[0], g = hd[1], nvalid = hd[2];
  const int S = mp.num_splits;
  const float2* ml = reinterpret_cast<const float2*>(mp.part_ml);
  const float4* po = reinterpret_cast<const float4*>(mp.part_o);
  const int rr = (tile % tiles_per_unit) * 128 + threadIdx.x;  // partial row
  const int r = threadIdx.x;
  const int off = (rr / 128) * mp.rows + r / mp.G;  // position inside the unit
  if (off >= nvalid) return;
  const int h = g * mp.G + r % mp.G;
  const size_t orow = (size_t)(row0 + off) * mp.Hq + h;
  uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(mp.out) + orow * D +
                                        grp * kColGroup * 4);
  // Every split's (m, l) of this row in one pass (independent loads).
  float2 mlv[kMaxMergeSplits];
  float M = -INFINITY;
#pragma unroll
  for (int s = 0; s < kMaxMergeSplits; ++s) {
    mlv[s] = make_float2(-INFINITY, 0.f);
    if (s < S) {
      mlv[s] = ml[((size_t)unit * S + s) * mp.part_rows + rr];
      M = fmaxf(M, mlv[s].x);
    }
  }
  if (M == -INFINITY) {  // no key reached this row in any split
#pragma unroll
    for (int i = 0; i < kColGroup / 2; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (grp == 0 && mp.lse != nullptr) mp.lse[orow] = -INFINITY;
    return;
  }
  const bool has_x = (mp.sinks != nullptr) || (mp.smooth != 0);
  const float ms = mp.sinks != nullptr ? mp.sinks[h] * kLog2e : 0.f;
  const float mf = has_x ? fmaxf(M, ms) : M;
  float den = has_x ? ex2(ms - mf) : 0.f;
#pragma unroll
  for (int s = 0; s < kMaxMergeSplits; ++s)
    if (s < S && mlv[s].x != -INFINITY) den += mlv[s].y * ex2(mlv[s].x - mf);
  den = fmaxf(den, 1e-30f);
  const float inv = 1.f / den;
  float4 acc[kColGroup];
#pragma unroll
  for (int i = 0; i < kColGroup; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int s = 0; s < kMaxMergeSplits; ++s) {
    // An empty split (m = -inf) wrote no O: its partial is not read.
    if (s < S && mlv[s].x != -INFINITY) {
      const size_t item = (size_t)unit * S + s;
      const float w = ex2(mlv[s].x - mf) * inv;
#pragma unroll
      for (int i = 0; i < kColGroup; ++i) {
        const float4 o = po[(item * (D / 4) + grp * kColGroup + i) * mp.part_rows + rr];
        acc[i].x += w * o.x;
        acc[i].y += w * o.y;
        acc[i].z += w * o.z;
        acc[i].w += w * o.w;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kColGroup / 2; ++i)
    dst[i] = make_uint4(pack2<BF16>(acc[2 * i].x, acc[2 * i].y),
                        pack2<BF16>(acc[2 * i].z, acc[2 * i].w),
                        pack2<BF16>(acc[2 * i + 1].x, acc[2 * i + 1].y),
                        pack2<BF16>(acc[2 * i + 1].z, acc[2 * i + 1].w));
  if (grp == 0 && mp.lse != nullptr) mp.lse[orow] = (mf + log2f(den)) * kLn2;
}

template <int D>
cudaError_t launch_merge_d(const MergeParams& mp, bool bf16, int grid, cudaStream_t st) {
  if (bf16)
    merge_kernel<D, true><<<grid, 128, 0, st>>>(mp);
  else
    merge_kernel<D, false><<<grid, 128, 0, st>>>(mp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const PrefillParams& p, int d, bool bf16, int part_rows, int grid,
                         cudaStream_t st) {
  MergeParams mp;
  mp.part_o = p.part_o;
  mp.part_ml = p.part_ml;
  mp.part_hdr = p.part_hdr;
  mp.sinks = p.sinks;
  mp.out = p.out;
  mp.lse = p.lse;
  mp.num_splits = p.num_splits;
  mp.Hq = p.Hq;
  mp.G = p.G;
  mp.rows = p.rows;
  mp.part_rows = part_rows;
  mp.smooth = p.smooth;
  if (grid < 1) return cudaSuccess;
  if (p.num_splits > kMaxMergeSplits) return cudaErrorInvalidValue;
  // Blocks: the units, times the 128-row query tiles of each, times the
  // column groups of a row.
  const int groups = d / 4 / (d == 64 ? col_group<64>() : col_group<128>());
  const long long blocks = (long long)grid * (part_rows / 128) * groups;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (d == 64) return launch_merge_d<64>(mp, bf16, (int)blocks, st);
  if (d == 128) return launch_merge_d<128>(mp, bf16, (int)blocks, st);
  if (d == 256) return launch_merge_d<256>(mp, bf16, (int)blocks, st);
  return cudaErrorInvalidValue;
}

}  // namespace gqa
