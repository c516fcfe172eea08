// Internal declarations shared by the kvq translation units (not installed).
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kBlockTokens = 128;  // tokens per block / page
constexpr int kHeadDim = 128;      // head dim of the specialised decode kernel (64 and 256: the general one)
constexpr int kGroupQ = 4;  // query heads per KV head
constexpr int kCounterGroups = 1;  // split-merge arrival counters per (sequence, kv head)

__device__ __forceinline__ void report(uint32_t* dev_status, uint32_t bits) {
  if (dev_status != nullptr) atomicOr(dev_status, bits);
}

struct PackParams {
  const float* x;    // pack: [batch][kv heads][max_seq_len][128]; append: the new tokens [batch][kv heads][128]
  float* window;     // append only: [batch][kv heads][128][128] raw rows of each current block
  const int32_t* seq_lens;
  const int32_t* page_table;
  uint8_t* codes;
  uint16_t* scale;
  uint16_t* zero;
  uint32_t* dev_status;
  int bits, k_scheme, v_scheme, which;
  int head_dim, group;  // D (64, 128, 256); group size G (32, 64, 128; <= D)
  int num_kv_heads, num_pages;
  int batch, max_seq_len, max_blocks, max_blocks_needed;
};

struct DequantParams {
  const uint8_t* codes;
  const uint16_t* scale;
  const uint16_t* zero;
  const int32_t* seq_lens;
  const int32_t* page_table;
  float* x_hat;
  uint32_t* dev_status;
  int bits, k_scheme, v_scheme, which;
  int head_dim, group;
  int num_kv_heads, num_pages;
  int batch, max_seq_len, max_blocks;
};

// Everything the decode kernel reads; built and validated on the host.
struct DecodeParams {
  const uint16_t* q;  // bf16 [B][Hq][128]
  const uint8_t* k_codes;
  const uint16_t* k_scale;
  const uint16_t* k_zero;
  const uint8_t* v_codes;
  const uint16_t* v_scale;
  const uint16_t* v_zero;
  const int32_t* seq_lens;
  const int32_t* page_table;
  float* out;
  float* lse;
  uint32_t* dev_status;
  int* counters;        // [B * Hkv] split-unit arrival counters (zeroed per call)
  float* part_o;        // [num_ctas][2][4][128]
  float* part_lse;      // [num_ctas][2][4]
  int batch, num_kv_heads, num_q_heads, max_blocks, num_pages;
  // units of work: up to 4 query heads of one KV head each.  gq = query heads
  // per unit (1, 2 or 4); units_per_seq = units per sequence (num_kv_heads,
  // or 2 * num_kv_heads with 8 query heads per KV head); unit head u reads KV
  // head u >> kv_shift.
  int gq, units_per_seq, kv_shift;
  int num_ctas;
  float sm_scale_log2;  // sm_scale * log2(e)
  uint32_t flags;
  uint64_t wait_limit_ns;
  // 2^28 and 2^32 - 1, passed at run time so that the compiler keeps the
  // code unpacking's shift and subtraction as integer multiply-adds (the
  // FMA pipe) instead of turning them back into shifts and logic ops (the
  // ALU pipe, the busier of the two in the converter warps)
  uint32_t nibble_mul, minus_one;
  unsigned long long* prof;  // cycle counters [grid][32] in profiling builds, else null
};

// KVQ_OK when the current device is an sm_103 GPU (and its SM count in
// *sm_count when non-null), else KVQ_ERR_DEVICE; launches nothing.
kvq_status check_device(int* sm_count);

size_t pack_smem_bytes(int head_dim, int group);
cudaError_t launch_pack(const PackParams& p, cudaStream_t stream);
cudaError_t launch_append(const PackParams& p, cudaStream_t stream);
cudaError_t launch_dequant(const DequantParams& p, cudaStream_t stream);
cudaError_t launch_merge(const float* o_parts, const float* lse_parts, int rows, int splits, int head_dim, float* out,
                         float* lse, cudaStream_t stream);

// Specialised decode kernel instances (head dim 128, groups of 128, E4M3
// operands): bits in {2, 4}, K/V scheme.
cudaError_t launch_decode(int bits, int k_scheme, int v_scheme, const DecodeParams& p, cudaStream_t stream);
int decode_ctas_per_sm();

}  // namespace kvq
