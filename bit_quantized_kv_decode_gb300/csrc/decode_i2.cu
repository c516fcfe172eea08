// Decode-attention kernel instances for 2-bit caches (all K/V scheme pairs, E4M3 operands);
// GQ4 selects 4 query heads per KV head (this file) or the other groupings
// (decode_i2_g.cu, which defines GQ4 false before including this one).
#include "decode.cuh"

#ifndef KVQ_GQ4
#define KVQ_GQ4 true
#define KVQ_FN launch_decode_i2
#endif

namespace kvq {

constexpr bool GQ4 = KVQ_GQ4;

cudaError_t KVQ_FN(int k_scheme, int v_scheme, const DecodeParams& p, cudaStream_t s) {
  const bool kcw = k_scheme == KVQ_CHANNELWISE, vcw = v_scheme == KVQ_CHANNELWISE;
  if (!kcw && !vcw) return launch_decode_instance<2, false, false, GQ4>(p, s);
  if (!kcw && vcw) return launch_decode_instance<2, false, true, GQ4>(p, s);
  if (kcw && !vcw) return launch_decode_instance<2, true, false, GQ4>(p, s);
  return launch_decode_instance<2, true, true, GQ4>(p, s);
}

}  // namespace kvq
