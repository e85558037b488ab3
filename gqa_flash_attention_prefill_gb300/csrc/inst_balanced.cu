// Kernel instantiations of the balanced split (one query tile per unit; the
// key-tile sizes the configuration cache picks by default for each head dim).
#include "launch.h"

namespace gqa {
cudaError_t launch_balanced(const PrefillParams& p, const KernelShape& ks, int d, bool win,
                            bool bf16, int grid, unsigned smem, cudaStream_t st) {
  if (!split_shape(d, ks.block_n, ks.q_tiles)) return cudaErrorInvalidValue;
  if (d == 64 && ks.block_n == 128)
    return launch_variants<64, 128, 2, 2, 1, false, false, false, true>(p, win, bf16, grid, smem, st);
  if (d == 64)
    return launch_variants<64, 64, 4, 2, 1, false, false, false, true>(p, win, bf16, grid, smem, st);
  if (d == 128)
    return launch_variants<128, 64, 2, 2, 1, false, false, false, true>(p, win, bf16, grid, smem, st);
  return launch_variants<256, 64, 2, 1, 1, false, false, false, true>(p, win, bf16, grid, smem, st);
}
}  // namespace gqa
