// Kernel instantiations for head dim 128.
#include "launch.h"

namespace gqa {
cudaError_t launch_d128(const PrefillParams& p, int block_n, bool win, bool bf16, int grid,
                        unsigned smem, cudaStream_t st) {
  if (block_n == 64) return launch_variants<128, 64, 2, 2>(p, win, bf16, grid, smem, st);
  if (block_n == 128) return launch_variants<128, 128, 2, 1>(p, win, bf16, grid, smem, st);
  return cudaErrorInvalidValue;
}
}  // namespace gqa
