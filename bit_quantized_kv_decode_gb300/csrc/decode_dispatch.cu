// Selects the decode-attention kernel instance for a cache configuration.
#include "kvq_internal.h"

namespace kvq {

cudaError_t launch_decode_i4(int k_scheme, int v_scheme, int mode, const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_i2(int k_scheme, int v_scheme, int mode, const DecodeParams& p, cudaStream_t s);

cudaError_t launch_decode(int bits, int k_scheme, int v_scheme, int mode, const DecodeParams& p, cudaStream_t s) {
  return bits == 4 ? launch_decode_i4(k_scheme, v_scheme, mode, p, s) : launch_decode_i2(k_scheme, v_scheme, mode, p, s);
}

int decode_ctas_per_sm() { return 2; }

}  // namespace kvq
