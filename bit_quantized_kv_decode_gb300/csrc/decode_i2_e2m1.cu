// Decode-attention kernel instances for 2-bit caches with the V codes placed
// as E2M1 values in shared memory (KVQ_FLAG_E2M1_V): FP8 operands, 4 query
// heads per KV head, every K/V scheme pair.
#include "decode.cuh"

namespace kvq {

cudaError_t launch_decode_i2_e2m1(int k_scheme, int v_scheme, const DecodeParams& p, cudaStream_t s) {
  const bool kcw = k_scheme == KVQ_CHANNELWISE, vcw = v_scheme == KVQ_CHANNELWISE;
  if (!kcw && !vcw) return launch_decode_instance<2, false, false, true, true>(p, s);
  if (!kcw && vcw) return launch_decode_instance<2, false, true, true, true>(p, s);
  if (kcw && !vcw) return launch_decode_instance<2, true, false, true, true>(p, s);
  return launch_decode_instance<2, true, true, true, true>(p, s);
}

}  // namespace kvq
