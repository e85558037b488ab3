// Kernel instantiations for head dim 256.
#include "launch.h"

namespace gqa {
cudaError_t launch_d256(const PrefillParams& p, int block_n, bool win, bool bf16, int grid,
                        unsigned smem, cudaStream_t st) {
  if (block_n == 64) return launch_variants<256, 64, 2, 1>(p, win, bf16, grid, smem, st);
  return cudaErrorInvalidValue;
}
}  // namespace gqa
