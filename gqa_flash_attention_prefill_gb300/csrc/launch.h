// launch.h -- internal interface between the host code and the per-head-dim
// kernel instantiations (one translation unit each, compiled in parallel).
#pragma once
#include <cuda_runtime.h>

#include <atomic>

#include "prefill_kernel.cuh"

namespace gqa {

constexpr int kMaxDevices = 64;

struct KernelShape {
  int block_n;      // keys per tile
  int q_tiles;      // 128-row query tiles per unit (1, or 2 sharing every K/V tile)
  int kv_stages;    // K/V ring depth
  int min_blocks;   // CTAs per SM the instantiation is compiled for
  unsigned smem;    // dynamic shared memory bytes
  int tmem_cols;    // tensor-memory columns a CTA allocates
};

// Shape of the instantiation used for (d, block_n, q_tiles); false if none exists.
bool kernel_shape(int d, int block_n, int q_tiles, KernelShape* out);

// Launches the instantiation for (d, block_n, q_tiles, windowed, bf16) with `grid` CTAs.
// `smem` is the dynamic shared memory requested per CTA: at least the
// instantiation's need, padded so that no more CTAs than planned fit on an SM
// (each resident CTA holds tensor memory for its whole life).
cudaError_t launch_d64(const PrefillParams& p, const KernelShape& ks, bool win, bool bf16,
                       int grid, unsigned smem, cudaStream_t st);
cudaError_t launch_d64_pair(const PrefillParams& p, const KernelShape& ks, bool win, bool bf16,
                            int grid, unsigned smem, cudaStream_t st);
cudaError_t launch_d128(const PrefillParams& p, const KernelShape& ks, bool win, bool bf16,
                        int grid, unsigned smem, cudaStream_t st);
cudaError_t launch_d256(const PrefillParams& p, const KernelShape& ks, bool win, bool bf16,
                        int grid, unsigned smem, cudaStream_t st);
// Split-KV instantiations (inst_split.cu); false from split_shape when (d,
// block_n, q_tiles) has none.
bool split_shape(int d, int block_n, int q_tiles);
cudaError_t launch_split(const PrefillParams& p, const KernelShape& ks, int d, bool win,
                         bool bf16, int grid, unsigned smem, cudaStream_t st);
// Paged-KV instantiations (inst_paged.cu), same shapes as split_shape.
cudaError_t launch_paged(const PrefillParams& p, const KernelShape& ks, int d, bool win,
                         bool bf16, int grid, unsigned smem, cudaStream_t st);

// Split-KV merge (merge.cu): one 128-thread block per unit, `grid` >= units.
cudaError_t launch_merge(const PrefillParams& p, int d, bool bf16, int part_rows, int grid,
                         cudaStream_t st);

// The launch helpers have internal linkage (one copy per translation unit):
// a function-local static in a template with external linkage is merged
// across shared objects by the dynamic linker, so two loaded copies of this
// library would share the cache below while owning different kernels.
namespace {

// Largest dynamic shared memory already allowed for one kernel on each device,
// so that the attribute is set once rather than on every launch.
struct SmemAttr {
  std::atomic<unsigned> allowed[kMaxDevices];
};

template <int D, int BN, int NS, bool WIN, bool BF16, int MINB, int QT, bool SPL, bool PAGED>
cudaError_t launch_one(const PrefillParams& p, int grid, unsigned smem, cudaStream_t st) {
  auto kern = prefill_kernel<D, BN, NS, WIN, BF16, MINB, QT, SPL, PAGED>;
  static SmemAttr attr{};
  if (smem < smem_bytes_for(D, BN, NS, QT)) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (attr.allowed[dev].load(std::memory_order_acquire) < smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr.allowed[dev].store(smem, std::memory_order_release);
  }
  kern<<<grid, threads_for(QT), smem, st>>>(p);
  return cudaGetLastError();
}

template <int D, int BN, int NS, int MINB, int QT, bool SPL = false, bool PAGED = false>
cudaError_t launch_variants(const PrefillParams& p, bool win, bool bf16, int grid, unsigned smem,
                            cudaStream_t st) {
  if (win)
    return bf16 ? launch_one<D, BN, NS, true, true, MINB, QT, SPL, PAGED>(p, grid, smem, st)
                : launch_one<D, BN, NS, true, false, MINB, QT, SPL, PAGED>(p, grid, smem, st);
  return bf16 ? launch_one<D, BN, NS, false, true, MINB, QT, SPL, PAGED>(p, grid, smem, st)
              : launch_one<D, BN, NS, false, false, MINB, QT, SPL, PAGED>(p, grid, smem, st);
}

}  // namespace

}  // namespace gqa
