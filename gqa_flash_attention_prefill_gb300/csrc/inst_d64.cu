// Kernel instantiations for head dim 64.
#include "launch.h"

namespace gqa {
cudaError_t launch_d64(const PrefillParams& p, int block_n, bool win, bool bf16, int grid,
                       unsigned smem, cudaStream_t st) {
  if (block_n == 128) return launch_variants<64, 128, 2, 2>(p, win, bf16, grid, smem, st);
  if (block_n == 64) return launch_variants<64, 64, 4, 2>(p, win, bf16, grid, smem, st);
  if (block_n == 96) return launch_variants<64, 96, 2, 2>(p, win, bf16, grid, smem, st);
  return cudaErrorInvalidValue;
}
}  // namespace gqa
