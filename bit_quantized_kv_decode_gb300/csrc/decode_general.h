// Decode attention for the general cache geometry (head dim 64 / 128 / 256,
// groups of 32 / 64 / 128 elements): parameters, shared-memory and
// tensor-memory layout (one definition, used by the host launch and the
// kernel), launch entry.
#pragma once
#include "kvq_internal.h"

namespace kvq {

struct GenParams {
  const uint16_t* q;  // bf16 [B][Hq][D]
  const uint8_t* k_codes;
  const uint16_t* k_scale;
  const uint16_t* k_zero;
  const uint8_t* v_codes;
  const uint16_t* v_scale;
  const uint16_t* v_zero;
  const int32_t* seq_lens;
  const int32_t* page_table;
  float* part_o;    // [B * Hq][splits][D]: each range's output, normalised over the range
  float* part_lse;  // [B * Hq][splits]: its log-sum-exp (natural log; -inf for an empty range)
  uint32_t* dev_status;
  int batch, num_kv_heads, num_q_heads, max_blocks, num_pages;
  int gq, units_per_seq, kv_shift;  // units of work, as in DecodeParams
  int group, splits;                // G; block ranges per unit (grid = units * splits)
  float sm_scale_log2;
  uint32_t flags;
  uint64_t wait_limit_ns;
  uint32_t nibble_mul, minus_one;  // 2^28 and 2^32 - 1 (see DecodeParams)
};

// Byte offsets in shared memory and column offsets in tensor memory.
struct GenLayout {
  int nsz;          // s (and z) values per block: 128 * D / G
  int stage_bytes;  // K codes, V codes, K s, K z, V s, V z of one block
  int q_off, p_off, scratch_off, total_bytes;
  int col_ak, col_av, col_s, col_o, tmem_cols;
};

__host__ __device__ inline GenLayout gen_layout(int bits, int D, int G, bool kcw, bool vcw) {
  GenLayout L;
  const int halves = D > 128 ? 2 : 1, ngc = D / G, ngt = kBlockTokens / G;
  L.nsz = kBlockTokens * D / G;
  L.stage_bytes = 2 * (kBlockTokens * D * bits / 8) + 4 * L.nsz * 2;
  L.q_off = 2 * L.stage_bytes;                             // two stages
  L.p_off = L.q_off + D * 16 * (kcw ? ngt : 1);            // Q': D rows x (16-byte block per token group)
  L.scratch_off = L.p_off + kBlockTokens * 16 * (vcw ? 1 : ngc);  // P': 128 rows x (block per channel group)
  L.total_bytes = L.scratch_off + 512;                     // reductions, group sums, barriers
  L.col_ak = 0;                                            // K operand: D / 4 columns
  L.col_av = D / 4;                                        // V operand: 32 columns per channel half
  L.col_s = L.col_av + 32 * halves;                        // S: 16 columns per block
  L.col_o = L.col_s + 16 * (kcw ? ngt : ngc);              // O: 16 columns per block per half
  const int used = L.col_o + halves * 16 * (vcw ? ngt : ngc);
  int cols = 32;
  while (cols < used) cols *= 2;
  L.tmem_cols = cols;
  return L;
}

struct GenLaunch {
  int ctas_per_sm;  // resident CTAs per SM (tensor memory and shared memory)
  size_t smem;      // dynamic shared memory per CTA
};

// Launch shape of the general kernel on a device with `smem_per_sm` bytes of
// shared memory per SM (`smem_reserved_per_cta` of them taken per CTA).
GenLaunch general_launch_shape(int bits, int k_scheme, int v_scheme, int head_dim, int group, int smem_per_sm,
                               int smem_reserved_per_cta);

cudaError_t launch_decode_general(int bits, int k_scheme, int v_scheme, int head_dim, const GenParams& p, int grid,
                                  size_t smem, cudaStream_t stream);

}  // namespace kvq
