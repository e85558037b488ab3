// Kernel instantiations for head dim 64, two 128-row query tiles per unit
// sharing every K/V tile (one CTA per SM, deeper K/V ring).
#include "launch.h"

namespace gqa {
cudaError_t launch_d64_pair(const PrefillParams& p, const KernelShape& ks, bool win, bool bf16,
                            int grid, unsigned smem, cudaStream_t st) {
  if (ks.block_n == 128) return launch_variants<64, 128, 4, 1, 2>(p, win, bf16, grid, smem, st);
  if (ks.block_n == 64) return launch_variants<64, 64, 8, 1, 2>(p, win, bf16, grid, smem, st);
  return cudaErrorInvalidValue;
}
}  // namespace gqa
