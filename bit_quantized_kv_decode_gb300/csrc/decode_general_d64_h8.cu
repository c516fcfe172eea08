// General-geometry decode kernel instances for head dim 64, E4M3 operands, 8 query heads per unit.
#include "decode_general.cuh"

namespace kvq {

cudaError_t launch_general_d64_h8(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                  const GenLaunch& shape, cudaStream_t s) {
  if (bits == 4) {
    if (group == 32) return gen::launch_schemes<4, 64, 32, false, 8>(kcw, vcw, p, grid, shape, s);
    if (group == 64) return gen::launch_schemes<4, 64, 64, false, 8>(kcw, vcw, p, grid, shape, s);
  }
  if (bits == 2) {
    if (group == 32) return gen::launch_schemes<2, 64, 32, false, 8>(kcw, vcw, p, grid, shape, s);
    if (group == 64) return gen::launch_schemes<2, 64, 64, false, 8>(kcw, vcw, p, grid, shape, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
