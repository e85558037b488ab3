// Kernel instantiations for head dim 256 (one query tile per unit: two would
// need more than the SM's 512 tensor-memory columns).
#include "launch.h"

namespace gqa {
cudaError_t launch_d256(const PrefillParams& p, const KernelShape& ks, bool win, bool bf16,
                        int grid, unsigned smem, cudaStream_t st) {
  if (ks.block_n == 64 && ks.q_tiles == 1)
    return launch_variants<256, 64, 2, 1, 1>(p, win, bf16, grid, smem, st);
  return cudaErrorInvalidValue;
}
}  // namespace gqa
