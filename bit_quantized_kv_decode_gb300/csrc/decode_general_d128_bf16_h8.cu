// General-geometry decode kernel instances for head dim 128, BF16 operands, 8 query heads per unit.
#include "decode_general.cuh"

namespace kvq {

cudaError_t launch_general_d128_bf16_h8(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                        const GenLaunch& shape, cudaStream_t s) {
  if (bits == 4) {
    if (group == 32) return gen::launch_schemes<4, 128, 32, true, 8>(kcw, vcw, p, grid, shape, s);
    if (group == 64) return gen::launch_schemes<4, 128, 64, true, 8>(kcw, vcw, p, grid, shape, s);
    if (group == 128) return gen::launch_schemes<4, 128, 128, true, 8>(kcw, vcw, p, grid, shape, s);
  }
  if (bits == 2) {
    if (group == 32) return gen::launch_schemes<2, 128, 32, true, 8>(kcw, vcw, p, grid, shape, s);
    if (group == 64) return gen::launch_schemes<2, 128, 64, true, 8>(kcw, vcw, p, grid, shape, s);
    if (group == 128) return gen::launch_schemes<2, 128, 128, true, 8>(kcw, vcw, p, grid, shape, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
