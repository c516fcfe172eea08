// Decode-attention kernel instances for 4-bit caches (all K/V scheme pairs, both operand modes).
#include "decode.cuh"

namespace kvq {

cudaError_t launch_decode_i4(int k_scheme, int v_scheme, int mode, const DecodeParams& p, cudaStream_t s) {
  const bool kcw = k_scheme == KVQ_CHANNELWISE, vcw = v_scheme == KVQ_CHANNELWISE, bf16 = mode == KVQ_OPERANDS_BF16;
  if (!bf16) {
    if (!kcw && !vcw) return launch_decode_instance<4, false, false, false>(p, s);
    if (!kcw && vcw) return launch_decode_instance<4, false, true, false>(p, s);
    if (kcw && !vcw) return launch_decode_instance<4, true, false, false>(p, s);
    return launch_decode_instance<4, true, true, false>(p, s);
  }
  if (!kcw && !vcw) return launch_decode_instance<4, false, false, true>(p, s);
  if (!kcw && vcw) return launch_decode_instance<4, false, true, true>(p, s);
  if (kcw && !vcw) return launch_decode_instance<4, true, false, true>(p, s);
  return launch_decode_instance<4, true, true, true>(p, s);
}

}  // namespace kvq
