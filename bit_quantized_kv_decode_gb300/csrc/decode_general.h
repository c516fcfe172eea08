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
  float* part_o;    // [slots][gq][D]: each range's output, normalised over the range (slot = CTA)
  float* part_lse;  // [slots][gq]: its log-sum-exp (natural log)
  uint32_t* dev_status;
  int batch, num_kv_heads, num_q_heads, max_blocks, num_pages;
  int gq, units_per_seq, kv_shift;  // units of work, as in DecodeParams
  long long n_target;               // CTAs the plan aims at for max_blocks per unit (see gen_plan in decode_general.cuh)
  long long n_floor;                // ... and at least, when the lengths hold less work: one wave of resident CTAs
  const int4* assign;               // [grid]: per CTA {b | unit << 16, j0, j1, length}; x < 0: no work
  const int* plan_ps;               // [B + 1]: the plan's prefix (CTAs of sequences before b)
  float sm_scale_log2;
  uint32_t flags;
  uint64_t wait_limit_ns;
  uint32_t nibble_mul, minus_one;  // 2^28 and 2^32 - 1 (see DecodeParams)
};

// Byte offsets in shared memory and column offsets in tensor memory.
//   tensor memory: [A: K codes, then V codes of the block][S and O]
//   (the V codes replace the K codes once QK^T is done; O replaces S once
//   the scores are read), with the two M = 128 channel halves of a 256-dim
//   head run one after the other (gen_turn) when both would not fit in 256
//   columns, or when taking them in turn holds more CTAs per SM.
struct GenLayout {
  int nsz;          // s (and z) values per block: 128 * D / G
  int stage_bytes;  // K codes, V codes, K s, K z, V s, V z of one block
  int stages;
  int q_off, p_off, scratch_off, total_bytes;
  int col_a, col_so, tmem_cols;
  bool seq_halves;  // PV one channel half at a time
};

constexpr int kGenPlanInts = 2 * 1024 + 4;  // the plan kernel's prefix (B + 1) and lengths (B) ints
constexpr int kGenRangeBlocks = 20;         // blocks per range the plan aims at when the lengths are short of max_blocks
constexpr int kGenScratchBytes = 2304;       // reduction buffers, per-group values and barriers (2,168 used)
constexpr int kGenSmemPerSm = 228 * 1024, kGenSmemPerCta = 1024;  // shared memory per SM, reserved per CTA

__host__ __device__ constexpr int gen_pow2_cols(int used) {
  return used <= 32 ? 32 : used <= 64 ? 64 : used <= 128 ? 128 : used <= 256 ? 256 : 512;
}
__host__ __device__ constexpr int gen_min(int a, int b) { return a < b ? a : b; }

// bf16: codes as exact BF16 values (two bytes each: twice the operand
// columns) and Q' / P' as two BF16 parts (32-byte rows); else E4M3.
// nh: query heads per unit (4 or 8): one column block per quad of heads.
// turn: PV one channel half at a time even where both halves fit.
__host__ __device__ constexpr GenLayout gen_layout_turn(int bits, int D, int G, bool kcw, bool vcw, bool bf16, int nh,
                                                        int stages, bool turn) {
  const int halves = D > 128 ? 2 : 1, ngc = D / G, ngt = kBlockTokens / G, w = bf16 ? 2 : 1, hh = nh / 4;
  const int a_cols = w * ((D / 4 > 32 * halves) ? D / 4 : 32 * halves);
  const int s_cols = 16 * (kcw ? ngt : ngc) * hh;
  const int o_all = halves * 16 * (vcw ? ngt : ngc) * hh;
  const bool seq = (turn && halves > 1) || a_cols + (s_cols > o_all ? s_cols : o_all) > 256;
  const int o_cols = seq ? o_all / halves : o_all;
  const int nsz = kBlockTokens * D / G;
  const int stage_bytes = 2 * (kBlockTokens * D * bits / 8) + 4 * nsz * 2;
  const int q_off = stages * stage_bytes;
  const int p_off = q_off + D * 16 * w * (kcw ? ngt : 1) * hh;  // Q': D rows x (block per token group, quad)
  const int scratch_off = p_off + kBlockTokens * 16 * w * (vcw ? 1 : ngc) * hh;  // P': 128 rows x (block per channel group, quad)
  return GenLayout{nsz, stage_bytes, stages, q_off, p_off, scratch_off, scratch_off + kGenScratchBytes, 0, a_cols,
                   gen_pow2_cols(a_cols + (s_cols > o_cols ? s_cols : o_cols)), seq};
}

// Resident CTAs per SM of an instance: as many as tensor memory (512
// columns per SM) and shared memory (228 KB per SM, 1 KB of it reserved per
// CTA) hold, up to a cap.  More CTAs hide more of each CTA's serial chain
// (copy wait, conversion, QK^T, softmax, PV); the caps are where more
// stopped paying (measured: 4-head units up to 8, 8-head units 5 with 4-bit
// codes and 6 with 2-bit (+0.3-1.2 points of the peak over 5; 7 lost); at 5,
// the kernel keeps within 96 registers a thread by holding the channel-wise
// K multipliers in shared memory).  The kernel's launch bounds take the same
// count (never below 4 for 4-head units), so its registers always fit.
__host__ __device__ constexpr int gen_fit(int bits, int D, int G, bool kcw, bool vcw, bool bf16, int nh, int stages,
                                          bool turn) {
  const GenLayout l = gen_layout_turn(bits, D, G, kcw, vcw, bf16, nh, stages, turn);
  return gen_min(gen_min(512 / l.tmem_cols, kGenSmemPerSm / (l.total_bytes + kGenSmemPerCta)),
                 nh > 4 ? (bits == 2 ? 6 : 5) : 8);
}
// A 256-dim head takes its two channel halves' PV in turn, with a one-stage
// copy ring, where that holds more CTAs per SM than both halves at once
// with two stages (half the O columns in tensor memory; measured at groups
// of 64, 4-bit codes: K-cw/V-tw 59.0 -> 77.9% of the peak, K-/V-token-wise
// 72.6 -> 88.2, 2 -> 4 CTAs per SM).
__host__ __device__ constexpr bool gen_turn(int bits, int D, int G, bool kcw, bool vcw, bool bf16, int nh) {
  return D > 128 && gen_fit(bits, D, G, kcw, vcw, bf16, nh, 1, true) > gen_fit(bits, D, G, kcw, vcw, bf16, nh, 2, false);
}
__host__ __device__ constexpr GenLayout gen_layout(int bits, int D, int G, bool kcw, bool vcw, bool bf16, int nh,
                                                   int stages) {
  return gen_layout_turn(bits, D, G, kcw, vcw, bf16, nh, stages, gen_turn(bits, D, G, kcw, vcw, bf16, nh));
}

// The other exception to the 2-stage ring: 4-bit codes at head dim 128,
// groups of 128 (E4M3, 4 heads), except K channel-wise with V token-wise,
// run 8 CTAs with one stage each (measured against 5 CTAs with two stages:
// K-/V-token-wise 95.8% of the peak, K-tw/V-cw 91.6 against 88.1, K-cw/V-cw
// 82.5 against 77.2; K-cw/V-tw lost, 82.2 against 83.1).
__host__ __device__ constexpr bool gen_single_stage(int bits, int D, int G, bool kcw, bool vcw, bool bf16, int nh) {
  return (bits == 4 && D == 128 && G == 128 && (vcw || !kcw) && !bf16 && nh == 4) ||
         gen_turn(bits, D, G, kcw, vcw, bf16, nh);
}
__host__ __device__ constexpr int gen_ctas_per_sm(int bits, int D, int G, bool kcw, bool vcw, bool bf16, int nh) {
  return gen_fit(bits, D, G, kcw, vcw, bf16, nh, gen_single_stage(bits, D, G, kcw, vcw, bf16, nh) ? 1 : 2,
                 gen_turn(bits, D, G, kcw, vcw, bf16, nh));
}
__host__ __device__ constexpr int gen_min_ctas(int bits, int D, int G, bool kcw, bool vcw, bool bf16, int nh) {
  const int c = gen_ctas_per_sm(bits, D, G, kcw, vcw, bf16, nh);
  return nh > 4 ? c : (c > 4 ? c : 4);
}

struct GenLaunch {
  int ctas_per_sm;  // resident CTAs per SM (tensor memory and shared memory)
  int stages;       // copy-ring stages
  size_t smem;      // dynamic shared memory per CTA
};

// Launch shape of the general kernel on a device with `smem_per_sm` bytes of
// shared memory per SM (`smem_reserved_per_cta` of them taken per CTA).
GenLaunch general_launch_shape(int bits, int k_scheme, int v_scheme, int head_dim, int group, bool bf16, int nh,
                               int smem_per_sm, int smem_reserved_per_cta);

cudaError_t launch_decode_general(int bits, int k_scheme, int v_scheme, int head_dim, int group, bool bf16, int nh,
                                  const GenParams& p, int grid, const GenLaunch& shape, cudaStream_t stream);
// The plan of a call (gen_plan): prefix and per-CTA assignments into the
// workspace (p.plan_ps, p.assign), one CTA per 1,024 decode CTAs (64 at most);
// launched before the decode kernel.
cudaError_t launch_general_plan(const GenParams& p, long long grid, int4* assign, int* plan_ps, cudaStream_t stream);
// The log-sum-exp merge of the parts into out [B][Hq][head_dim] and lse [B][Hq].
cudaError_t launch_general_merge(const GenParams& p, int head_dim, float* out, float* lse, cudaStream_t stream);

}  // namespace kvq
