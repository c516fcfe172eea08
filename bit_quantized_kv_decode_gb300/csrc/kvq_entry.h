// Decode entry points with a bound on the workspace, shared by the public
// entry points (kvq_api.cu) and the no-allocation entry (decode_static.cu).
#pragma once
#include "kvq_internal.h"

namespace kvq {

// kvq_decode_workspace_size / kvq_decode_attn for a caller whose workspace
// holds at most `limit` bytes (the static entry): a call the general kernel
// would take with a larger workspace goes to the specialised kernel when that
// one takes it (E4M3 operands, head dim 128, groups of 128).  The public
// entry points pass SIZE_MAX.
kvq_status decode_workspace_bounded(const kvq_attn_desc* desc, size_t limit, size_t* bytes);
kvq_status decode_attn_bounded(const kvq_attn_desc* desc, const uint16_t* q, const uint8_t* k_codes,
                               const uint16_t* k_scale, const uint16_t* k_zero, const uint8_t* v_codes,
                               const uint16_t* v_scale, const uint16_t* v_zero, const int32_t* seq_lens,
                               const int32_t* page_table, float* out, float* lse, void* workspace,
                               size_t workspace_bytes, size_t limit, uint32_t* dev_status, void* stream);

}  // namespace kvq
