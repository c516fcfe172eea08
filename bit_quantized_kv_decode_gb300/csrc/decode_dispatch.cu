// Selects the decode-attention kernel instance for a cache configuration.
#include "kvq_internal.h"

namespace kvq {

cudaError_t launch_decode_i4(int k_scheme, int v_scheme, const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_i2(int k_scheme, int v_scheme, const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_i4_g(int k_scheme, int v_scheme, const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_i2_g(int k_scheme, int v_scheme, const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_i2_e2m1(int k_scheme, int v_scheme, const DecodeParams& p, cudaStream_t s);

cudaError_t launch_decode(int bits, int k_scheme, int v_scheme, const DecodeParams& p, cudaStream_t s) {
  if (p.flags & KVQ_FLAG_E2M1_V) return launch_decode_i2_e2m1(k_scheme, v_scheme, p, s);  // validated by the caller
  if (p.gq == kGroupQ && p.kv_shift == 0)  // 4 query heads per KV head
    return bits == 4 ? launch_decode_i4(k_scheme, v_scheme, p, s) : launch_decode_i2(k_scheme, v_scheme, p, s);
  return bits == 4 ? launch_decode_i4_g(k_scheme, v_scheme, p, s)
                   : launch_decode_i2_g(k_scheme, v_scheme, p, s);
}

int decode_ctas_per_sm() { return 2; }

}  // namespace kvq
