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

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // device address of the array, per device

// Address of the scratch array on the current device, looked up once.
int scratch_address(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return GQA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
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
  if (num_seqs == 0 || total_q == 0) return GQA_OK;  // no work, no launch
  int splits = 1;
  size_t bytes = 0;
  int rc = gqa_prefill_splitkv_workspace(num_seqs, total_q, max_seqlen_q, Hq, Hkv, d, dtype,
                                         window, num_splits, &splits, &bytes);
  if (rc != GQA_OK) return rc;
  if (bytes > gqa::kNoAllocScratchBytes) return GQA_ERR_UNSUPPORTED;  // declined: too large
  void* scratch = nullptr;
  if (splits > 1 && (rc = gqa::scratch_address(&scratch)) != GQA_OK) return rc;
  // Nothing in the scratch has to start at zero: every value the merge reads
  // (unit count, unit headers, each split's (m, l) record and, for non-empty
  // splits, its partial O) is written earlier in the same call.
  return gqa_flash_prefill_splitkv(q, k, v, cu_seqlens_q, prefix_lens, kv_indptr, num_seqs,
                                   total_q, total_kv, max_seqlen_q, Hq, Hkv, d, dtype, scale,
                                   window, sinks, smooth_softmax, out, lse, splits, scratch,
                                   splits > 1 ? gqa::kNoAllocScratchBytes : 0, stream);
}

}  // extern "C"
