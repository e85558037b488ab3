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

// Custom-mask instantiations (inst_mask.cu), same shapes as split_shape.
cudaError_t launch_mask(const PrefillParams& p, const KernelShape& ks, int d, bool win,
                        bool bf16, int grid, unsigned smem, cudaStream_t st);

// Balanced-split instantiations (inst_balanced.cu), same shapes as split_shape.
cudaError_t launch_balanced(const PrefillParams& p, const KernelShape& ks, int d, bool win,
                            bool bf16, int grid, unsigned smem, cudaStream_t st);

// Split-KV merge (merge.cu): one 128-thread block per unit, `grid` >= units.
cudaError_t launch_merge(const PrefillParams& p, int d, bool bf16, int part_rows, int grid,
                         cudaStream_t st);

// The CUDA context current on this thread (nullptr if none), from the
// driver's entry point: per-device caches of symbol addresses are keyed on it,
// since a device reset makes a new context that may load the module elsewhere.
void* current_context();

// Scratch provider of a split-KV call without a caller workspace: given the
// bytes the call's plan needs, stores the scratch address and its capacity,
// or returns GQA_ERR_UNSUPPORTED when the need exceeds the capacity.
typedef int (*ScratchFn)(size_t bytes, void** ptr, size_t* capacity);

// gqa_flash_prefill_splitkv with the workspace taken from `scratch` (host.cu).
int run_splitkv_scratch(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                        const int32_t* prefix_lens, const int32_t* kv_indptr, int num_seqs,
                        int total_q, int total_kv, int max_seqlen_q, int Hq, int Hkv, int d,
                        int dtype, float scale, int window, const float* sinks,
                        int smooth_softmax, void* out, float* lse, int num_splits, void* stream,
                        ScratchFn scratch);

// Whether kernels are launched with programmatic stream serialisation
// (host.cu; GQA_PREFILL_PDL=0 turns it off, read once per process).
bool pdl_enabled();

// Launches `kern(p)` on `st`.  With programmatic dependent launch on, the
// kernel may begin while the previous kernel in the stream finishes: its
// CTAs run their set-up, then wait (griddepcontrol.wait) for that kernel's
// writes before the first read of device memory.
template <typename Kern, typename Params>
cudaError_t launch_pdl(Kern kern, const Params& p, int grid, int threads, unsigned smem,
                       cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

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

template <int D, int BN, int NS, bool WIN, bool BF16, int MINB, int QT, bool SPL, bool PAGED,
          bool MASK = false, bool SK = false>
cudaError_t launch_one(const PrefillParams& p, int grid, unsigned smem, cudaStream_t st) {
  auto kern = prefill_kernel<D, BN, NS, WIN, BF16, MINB, QT, SPL, PAGED, MASK, SK>;
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
  return launch_pdl(kern, p, grid, threads_for(QT), smem, st);
}

template <int D, int BN, int NS, int MINB, int QT, bool SPL = false, bool PAGED = false,
          bool MASK = false, bool SK = false>
cudaError_t launch_variants(const PrefillParams& p, bool win, bool bf16, int grid, unsigned smem,
                            cudaStream_t st) {
  if (win)
    return bf16 ? launch_one<D, BN, NS, true, true, MINB, QT, SPL, PAGED, MASK, SK>(p, grid, smem, st)
                : launch_one<D, BN, NS, true, false, MINB, QT, SPL, PAGED, MASK, SK>(p, grid, smem, st);
  return bf16 ? launch_one<D, BN, NS, false, true, MINB, QT, SPL, PAGED, MASK, SK>(p, grid, smem, st)
              : launch_one<D, BN, NS, false, false, MINB, QT, SPL, PAGED, MASK, SK>(p, grid, smem, st);
}

}  // namespace

}  // namespace gqa
