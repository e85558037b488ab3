// Kernel instantiations for head dim 64, one 128-row query tile per unit.
#include "launch.h"

namespace gqa {
cudaError_t launch_d64(const PrefillParams& p, const KernelShape& ks, bool win, bool bf16,
                       int grid, unsigned smem, cudaStream_t st) {
  if (ks.q_tiles == 2) return launch_d64_pair(p, ks, win, bf16, grid, smem, st);
  if (ks.block_n == 128) return launch_variants<64, 128, 2, 2, 1>(p, win, bf16, grid, smem, st);
  if (ks.block_n == 64) return launch_variants<64, 64, 4, 2, 1>(p, win, bf16, grid, smem, st);
  if (ks.block_n == 96) return launch_variants<64, 96, 2, 2, 1>(p, win, bf16, grid, smem, st);
  return cudaErrorInvalidValue;
}
}  // namespace gqa
