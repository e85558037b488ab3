// noalloc.cu -- gqa_flash_prefill_splitkv_noalloc: the split-KV call with its
// scratch in a file-scope device array instead of a caller workspace, so a
// call allocates nothing (no cudaMalloc / cudaFree, no allocating library
// routine).  Declared in include/gqa_prefill.h.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "gqa_prefill.h"
#include "launch.h"

namespace gqa {
namespace {

// 32 MiB: e.g. 256 split work items of a d = 64 unit (33 KB of partials each).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, looked up once per device and context: the
// name g_noalloc_scratch is a host-side stand-in in host code, never an
// address a kernel may be given.  A new context (after a device reset) may
// hold the module elsewhere, so the address is looked up again then.
struct ScratchAddr {
  void* ctx = nullptr;
  void* addr = nullptr;
};
std::mutex g_scratch_mu;
ScratchAddr g_scratch_addr[kMaxDevices];

// ScratchFn for run_splitkv_scratch: declines a need above the array's size,
// else hands out the array's device address on the current device.
int scratch_for(size_t bytes, void** ptr, size_t* capacity) {
  if (bytes > kNoAllocScratchBytes) return GQA_ERR_UNSUPPORTED;  // declined: too large
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& e = g_scratch_addr[dev];
  if (e.addr == nullptr || e.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return GQA_ERR_CUDA;
    e.addr = p;
    e.ctx = ctx;
  }
  *ptr = e.addr;
  *capacity = kNoAllocScratchBytes;
  return GQA_OK;
}

}  // namespace
}  // namespace gqa

extern "C" {

int gqa_flash_prefill_splitkv_noalloc(const void* q, const void* k, const void* v,
                                      const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                                      const int32_t* kv_indptr, int num_seqs, int total_q,
                                      int total_kv, int max_seqlen_q, int Hq, int Hkv, int d,
                                      int dtype, float scale, int window, const float* sinks,
                                      int smooth_softmax, void* out, float* lse, int num_splits,
                                      void* stream) {
  // The same validation, plan and launch as gqa_flash_prefill_splitkv; when
  // the plan splits, the scratch comes from scratch_for, which checks the
  // plan's own workspace layout against the array.  Nothing in the scratch
  // has to start at zero: every value the merge reads (unit count, unit
  // headers, each split's (m, l) record and, for non-empty splits, its
  // partial O) is written earlier in the same call.
  return gqa::run_splitkv_scratch(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs,
                                  total_q, total_kv, max_seqlen_q, Hq, Hkv, d, dtype, scale,
                                  window, sinks, smooth_softmax, out, lse, num_splits, stream,
                                  gqa::scratch_for);
}

}  // extern "C"
