// Kernel instantiations for head dim 128.
#include "launch.h"

namespace gqa {
cudaError_t launch_d128(const PrefillParams& p, const KernelShape& ks, bool win, bool bf16,
                        int grid, unsigned smem, cudaStream_t st) {
  if (ks.q_tiles == 2 && ks.block_n == 64)
    return launch_variants<128, 64, 4, 1, 2>(p, win, bf16, grid, smem, st);
  if (ks.q_tiles != 1) return cudaErrorInvalidValue;
  if (ks.block_n == 64) return launch_variants<128, 64, 2, 2, 1>(p, win, bf16, grid, smem, st);
  if (ks.block_n == 128) return launch_variants<128, 128, 2, 1, 1>(p, win, bf16, grid, smem, st);
  return cudaErrorInvalidValue;
}
}  // namespace gqa
