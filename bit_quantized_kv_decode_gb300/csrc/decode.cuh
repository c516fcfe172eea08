// Affine-folded decode attention over a packed INT2/INT4 KV cache, sm_103a.
//
// Method (cited by page title and section):
//  * "FOSCAR: Accelerating Decode Attention over 2- and 4-Bit KV Caches
//    through Affine Folding" (papers.pytorch.kr), abstract: scale/offset are
//    applied to the other operand or to the output of the two products, not
//    to each KV value; packed bits feed the tensor cores directly.
//  * rag-lover.com summary of arXiv 2611.09722, section "解説": QK^T contracts
//    over channels (token-wise K: scale the partial result by s, add z*sum(q);
//    channel-wise K: fold s into Q, add q.z after), PV contracts over tokens
//    (token-wise V: fold s into P; channel-wise V: scale the partial result
//    and add z*sum(p)); a 4-bit code in the low bits of an E4M3 element reads
//    as q*2^-9.  Section "限界と未検証の範囲": accumulator folds are applied one
//    quantization group at a time.
//
// kvq_decode_attn runs this kernel for small calls (its persistent CTAs start
// faster) and for the E2M1 V placement; calls of real size take the
// block-range kernel of decode_general.cuh, measured faster there.
//
// GB300 design (this library's; the pages' Blackwell pipeline is prior art):
//  * swap-AB MMAs: tokens (QK^T) or channels (PV) are the M = 128 rows, the
//    4 GQA query heads x operand splits are N = 16 columns;
//  * the KV operand (A) is written by converter warps straight into tensor
//    memory (tcgen05.st) and read by tcgen05.mma from there, so the hot
//    operand never passes through shared memory: packed codes are the only
//    KV bytes staged in shared memory (by cp.async.bulk);
//  * INT4 and INT2 codes both become E4M3 bytes (code * 2^-9): 3 integer ops
//    per 8 INT4 codes, 7 per 16 INT2 codes;
//  * Q' and P' are sums of three E4M3 parts stacked along N, so precision
//    costs no extra MMA (the BF16-operand mode runs in the block-range kernel
//    of decode_general.cuh);
//  * persistent CTAs take equal ranges of (sequence, kv head, 128-token tile);
//    a (sequence, kv head) cut by a range boundary is merged by the last CTA
//    to finish a part (log-sum-exp over the parts, no waiting);
//  * every wait is bounded; on a timeout the CTA records KVQ_DEV_TIMEOUT,
//    drains its copies and MMAs, frees tensor memory and returns.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

// Optional cycle accounting per CTA and pipeline role (built only when
// KVQ_PROFILE is defined; the library build never defines it).  Probes add
// into shared memory: a global atomic per probe would stall the next
// mbarrier arrive, whose release semantics wait for it to complete.
#if defined(KVQ_PROFILE) && !defined(KVQ_TRACE)
#define KVQ_PT(n) long long kvq_pt_##n = clock64();
#define KVQ_PA(slot, n) \
  if (p.prof != nullptr && (threadIdx.x & 31) == 0) atomicAdd(&sh.prof[slot], (unsigned long long)(clock64() - kvq_pt_##n));
#else
#define KVQ_PT(n)
#define KVQ_PA(slot, n)
#endif
// Optional per-tile event timeline (KVQ_TRACE with KVQ_PROFILE): lane 0 of
// the recording warp stamps event ev of tile t (a window of tiles) in shared
// memory; the CTA dumps it to the profiling buffer at exit.
constexpr int kTrT0 = 200, kTrN = 64, kTrEv = 24;
#ifdef KVQ_TRACE
#define KVQ_TR(ev, t) \
  { if ((threadIdx.x & 31) == 0 && (t) >= kTrT0 && (t) < kTrT0 + kTrN) sh.trace[((t) - kTrT0) * kTrEv + (ev)] = clock64(); }
#else
#define KVQ_TR(ev, t) {}
#endif

constexpr int kDecodeThreads = 384;  // 12 warps: three warpgroups (warps 10, 11 only complete the third)
constexpr int kMaxBatch = 1024;      // sequences per call (prefix table in shared memory)
constexpr uint32_t FULL = 0xffffffffu;

// Warp roles.  Registers are rebalanced per warpgroup at the start of the
// role code (setmaxnreg): the launch gives every thread kRegsLaunch; the
// loader / MMA warpgroup gives back down to kRegsLight, and the converter and
// softmax warpgroups take them (kRegsConvert, kRegsSoftmax).  The three add
// up to the launch total, so the increases never wait on registers that
// will not come.
constexpr int kWarpConvert0 = 0;  // warps 0-3: KV codes -> tensor memory, Q' operand
constexpr int kWarpSoftmax0 = 4;  // warps 4-7: fold, online softmax, P' operand, epilogue (two tiles per step)
constexpr int kWarpLoad = 8;      // packed tiles HBM -> shared memory
constexpr int kWarpMma = 9;       // tcgen05.mma issue, tensor memory owner
constexpr int kRegsLaunch = 80, kRegsLight = 24, kRegsSoftmax = 112, kRegsConvert = 104;
static_assert(128 * kRegsConvert + 128 * kRegsSoftmax + 128 * kRegsLight == kDecodeThreads * kRegsLaunch,
              "setmaxnreg split must add up to the launch allocation");

// E2V: 2-bit V codes as E2M1 values (code / 2) in shared memory (the
// KVQ_FLAG_E2M1_V placement); otherwise codes are E4M3 bytes in tensor memory.
template <int BITS, bool E2V = false>
struct DecodeCfg {
  static constexpr int kBlockBytes = kBlockTokens * kHeadDim * BITS / 8;  // 8192 / 4096
  static constexpr int kChunks = kHeadDim * BITS / 8 / 16;                // 16-byte chunks per row
  static constexpr bool kE2V = E2V;
  static_assert(!E2V || BITS == 2, "E2M1 placement: 2-bit codes");
  // (four stages with the E2M1 tiles: two CTAs per SM must still fit)
  static constexpr int kStages = (BITS == 4) ? 4 : (E2V ? 4 : 6);
  static constexpr int kSzBytes = kBlockTokens * 2;                       // one fp16 [128] array
  static constexpr int kStageBytes = 2 * kBlockBytes + 4 * kSzBytes;
  static constexpr int kACols = 32;      // tensor-memory columns of one 128 x 128 A tile (E4M3 bytes)
  static constexpr int kNAK = 2;         // A tile buffers: K codes
  static constexpr int kNAV = 3;         // A tile buffers: V codes (the converters run ahead of PV)
  static constexpr int kSplits = 3;      // E4M3 parts of Q' and P'
  static constexpr int kBBytes = 2048;   // one B operand (128 K-rows x N=16)
  static constexpr int kKSteps = 4;
  static constexpr uint32_t kKStepBBytes = 512;
  static constexpr uint32_t kLbo = 128;  // K-direction core-matrix stride
  static constexpr uint32_t kSbo = 128;  // N-direction core-matrix stride
  static constexpr uint32_t kIdesc = make_idesc(0, 0, 0, 1, 128, 16);
  static constexpr int kSlots = 3;       // score / probability / output buffers in flight
  static constexpr int kColAK = 0;
  static constexpr int kColAV = kNAK * kACols;
  static constexpr int kColS = kColAV + kNAV * kACols;
  static constexpr int kColO = kColS + 16 * kSlots;
  static constexpr int kTmemCols = 256;
  // code = operand value * code scale (E4M3: code * 2^-9; E2M1: code / 2)
  static constexpr float kCodeInv = 512.0f;  // K: code = operand value * 2^9
  static constexpr int kVCodeLog2 = E2V ? 1 : 9;
  static constexpr uint32_t kIdescV = E2V ? make_idesc(5, 0, 0, 1, 128, 16) : kIdesc;  // A = E2M1, B = E4M3
  // E2M1 tiles in shared memory: canonical K-major layout without swizzle;
  // a 16-byte unit holds 16 codes of one row as packed nibbles (8 bytes) and
  // 8 bytes of padding; K-groups of 16 codes kALbo apart, 8-row groups kASbo
  static constexpr uint32_t kALbo = 2048, kASbo = 128;
  static constexpr int kASmBytes = 16384;  // one 128 x 128 tile
  static constexpr int kASmTiles = E2V ? kNAV : 0;
  static_assert(kColO + 16 * kSlots <= kTmemCols, "tensor memory budget");
};

// Position of element e (channel of a K row, token of a V row) along the
// contraction dimension of the A operand, i.e. where the converter's masks
// put it.  The B operand rows (Q' channels, P' tokens) use the same order.
template <int BITS, bool BF16, bool E2 = false>
__device__ __forceinline__ int a_pos(int e) {
  if (E2) return (e & ~15) + ((e & 1) << 3) + ((e & 15) >> 1);  // even codes, then odd codes
  if (!BF16) {
    if (BITS == 4) return (e & ~7) + ((e & 1) << 2) + ((e & 7) >> 1);
    return (e & ~15) + ((e & 3) << 2) + ((e & 15) >> 2);
  } else {
    if (BITS == 4) return (e & ~7) + ((e & 3) << 1) + ((e & 7) >> 2);
    return (e & ~15) + ((e & 7) << 1) + ((e & 15) >> 3);
  }
}

// The used columns of one S / O slot (4 heads x 3 parts): a single
// 12-column load instead of all 16.
__device__ __forceinline__ void tmem_ld_parts(uint32_t taddr, uint32_t (&r)[12]) {
  tmem_ld_32x32b_x8(taddr, r);
  tmem_ld_32x32b_x4(taddr + 8, r + 8);
}

// Byte offset of B-operand row p (MN-major, no swizzle, E4M3: one core
// matrix per 8 rows).
__device__ __forceinline__ uint32_t b_row_off(int p) { return (uint32_t)(p * 16); }

// B-operand row factor matching Convert: 2-bit codes at odd positions e are
// stored as 4 * code, so their Q' / P' rows are scaled by 1/4 (exact).
template <int BITS, bool BF16, bool E2 = false>
__device__ __forceinline__ float odd_quarter(int e) {
  return (BITS == 2 && !BF16 && !E2 && (e & 1)) ? 0.25f : 1.0f;
}

// ---------------------------------------------------------------- operands
// 4 floats -> 4 E4M3 bytes (element i in byte i), round to nearest, saturate.
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}
__device__ __forceinline__ float4 unpack4_e4m3(uint32_t w) {
  __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
  __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  float2 a = __half22float2(*reinterpret_cast<__half2*>(&h01));
  float2 b = __half22float2(*reinterpret_cast<__half2*>(&h23));
  return make_float4(a.x, a.y, b.x, b.y);
}
// x ~= hi + mid + lo, each part E4M3 (greedy residual split).
__device__ __forceinline__ uint4 split3_e4m3(float4 v) {
  uint4 r;
  r.x = pack4_e4m3(v.x, v.y, v.z, v.w);
  float4 f = unpack4_e4m3(r.x);
  v = make_float4(v.x - f.x, v.y - f.y, v.z - f.z, v.w - f.w);
  r.y = pack4_e4m3(v.x, v.y, v.z, v.w);
  f = unpack4_e4m3(r.y);
  v = make_float4(v.x - f.x, v.y - f.y, v.z - f.z, v.w - f.w);
  r.z = pack4_e4m3(v.x, v.y, v.z, v.w);
  r.w = 0u;
  return r;
}
// x ~= hi + lo, each part BF16: {hi01, hi23, lo01, lo23}.
__device__ __forceinline__ uint4 split2_bf16(float4 v) {
  __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y), h23 = __floats2bfloat162_rn(v.z, v.w);
  float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
  __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
  __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
  uint4 r;
  r.x = *reinterpret_cast<uint32_t*>(&h01);
  r.y = *reinterpret_cast<uint32_t*>(&h23);
  r.z = *reinterpret_cast<uint32_t*>(&l01);
  r.w = *reinterpret_cast<uint32_t*>(&l23);
  return r;
}

// Power of two 2^k with m * 2^k in [128, 256); 1 when m < 2^-120 (the
// factor would leave the fp32 exponent range) or m is non-finite.
__device__ __forceinline__ float pow2_prescale(float m) {
  int e = (int)((__float_as_uint(m) >> 23) & 0xffu);
  if (e < 7 || e == 0xff) return 1.0f;
  return __uint_as_float((uint32_t)(261 - e) << 23);  // 2^(7 - (e - 127))
}
// 1 / pow2_prescale(m), exactly (no division).
__device__ __forceinline__ float pow2_prescale_inv(float m) {
  int e = (int)((__float_as_uint(m) >> 23) & 0xffu);
  if (e < 7 || e == 0xff) return 1.0f;
  return __uint_as_float((uint32_t)(e - 7) << 23);  // 2^((e - 127) - 7)
}

// Channel-wise K prescale of Q', split into a per-segment head factor and a
// per-tile group factor.  With E_q = floor(log2 qmax) and E_s the exponent
// of the group's largest fp16 scale, Q' = q * s * 2^(6 - E_q) * 2^(-E_s)
// stays below 2^(E_q+1) * 2^(E_s+1) * 2^(6 - E_q - E_s) = 256 (no E4M3
// overflow); the score multiplier 2^(E_q - 6) * 2^(E_s) undoes it exactly.
// A query with qmax < 2^-120 (or non-finite) uses factor 1 on both sides.
__device__ __forceinline__ float pow2_head(float qmax) {
  const int e = (int)((__float_as_uint(qmax) >> 23) & 0xffu);
  return (e < 7 || e == 0xff) ? 1.0f : __uint_as_float((uint32_t)(260 - e) << 23);  // 2^(6 - E_q)
}
__device__ __forceinline__ float pow2_head_inv(float qmax) {
  const int e = (int)((__float_as_uint(qmax) >> 23) & 0xffu);
  return (e < 7 || e == 0xff) ? 1.0f : __uint_as_float((uint32_t)(e - 6) << 23);  // 2^(E_q - 6)
}
// Exponent field of an fp16 maximum, clamped to the normal range [1, 30].
__device__ __forceinline__ uint32_t f16_exp_field(uint32_t h) {
  const uint32_t e = (h >> 10) & 31u;
  return e < 1u ? 1u : (e > 30u ? 30u : e);
}
__device__ __forceinline__ float pow2_group(uint32_t e16) { return __uint_as_float((142u - e16) << 23); }      // 2^(-E_s)
__device__ __forceinline__ float pow2_group_inv(uint32_t e16) { return __uint_as_float((112u + e16) << 23); }  // 2^(E_s)

// P' prescale of one head: with x = (pair maximum - running maximum) in log2
// units (<= 0) and e_v the exponent of the pair's largest V scale (0 for
// channel-wise V), E = floor(x) + e_v bounds log2 of the head's largest
// p * s; the scale 2^(6 - E) keeps max |P'| below 256 and is undone exactly
// by 2^(E - 6).  E is clamped to [-120, 120] (-inf / NaN x included); the
// four heads' E are kept as signed bytes of one word.
__device__ __forceinline__ int p_exponent(float x, int e_v) {
  const int fx = (x > -100.0f) ? __float2int_rd(x) : -100;
  const int e = fx + e_v;
  return e < -120 ? -120 : (e > 120 ? 120 : e);
}
// Signed byte k of a packed word, sign-extended (one byte permute: selector
// nibbles k for byte 0 and 8 + k, "replicate the sign of byte k", above it).
__device__ __forceinline__ int p_exp_of(uint32_t packed, int k) {
  int r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(packed), "r"(k | ((8 | k) << 4) | ((8 | k) << 8) | ((8 | k) << 12)));
  return r;
}
// 2^(6 - E) and 2^(E - 6 + code_log2) for head k of a packed word.
__device__ __forceinline__ float p_scale(uint32_t packed, int k) {
  return __uint_as_float((uint32_t)(133 - p_exp_of(packed, k)) << 23);
}
__device__ __forceinline__ float p_inverse(uint32_t packed, int k, int code_log2) {
  return __uint_as_float((uint32_t)(121 + code_log2 + p_exp_of(packed, k)) << 23);
}

// Packed pairs of fp32 values (two heads at once): one sm_100-family
// instruction per pair instead of two, with the same IEEE round-to-nearest
// results as the scalar operations.
__device__ __forceinline__ float2 f2u(uint32_t a, uint32_t b) {
  return make_float2(__uint_as_float(a), __uint_as_float(b));
}
__device__ __forceinline__ float2 f2s(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// 2^x (hardware approximation, flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// x ~= hi + mid + lo (each E4M3), with the residuals taken in f16x2
// arithmetic: {hi, mid, lo, 0} words, element i in byte i.  Used for P'
// (the fp16 rounding of x stays below the operand's own error).
__device__ __forceinline__ uint4 split3_e4m3_via_f16(float4 v) {
  __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
  uint32_t w[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const __nv_fp8x2_storage_t ea = __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<__half2_raw*>(&a), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t eb = __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<__half2_raw*>(&b), __NV_SATFINITE, __NV_E4M3);
    w[k] = (uint32_t)ea | ((uint32_t)eb << 16);
    if (k < 2) {
      __half2_raw ra = __nv_cvt_fp8x2_to_halfraw2(ea, __NV_E4M3), rb = __nv_cvt_fp8x2_to_halfraw2(eb, __NV_E4M3);
      a = __hsub2(a, *reinterpret_cast<__half2*>(&ra));
      b = __hsub2(b, *reinterpret_cast<__half2*>(&rb));
    }
  }
  return make_uint4(w[0], w[1], w[2], 0u);
}

// Converted code words of one packed 32-bit word.  `mul` = 2^28 and
// `m1` = 2^32 - 1 arrive as run-time values: x >> 4 is taken as the high
// word of x * 2^28 and x - y as x + y * m1, integer multiply-adds that issue
// on the FMA pipe, which the converter warps leave mostly idle, while the
// masks stay on the ALU pipe.
template <int BITS, bool BF16>
struct Convert {
  static constexpr int kOut = BF16 ? (BITS == 4 ? 4 : 8) : (BITS == 4 ? 2 : 4);
  __device__ __forceinline__ static void run(uint32_t x, uint32_t* o, uint32_t mul, uint32_t m1) {
    if (!BF16) {
      if (BITS == 4) {  // codes e = 0,2,4,6 then 1,3,5,7 as E4M3 0x0q
        o[0] = x & 0x0F0F0F0Fu;
        o[1] = __umulhi(x + o[0] * m1, mul);  // high nibbles (low ones cleared), shifted down
      } else {  // word k holds codes e = k, k+4, k+8, k+12; words 1 and 3 hold 4 * code
        // (E4M3 byte b is b * 2^-9 exactly for b < 16, so the shift is left to
        // the B operand: its rows for odd e carry a factor 1/4, see odd_quarter)
        const uint32_t y = __umulhi(x, mul);  // x >> 4
        o[0] = x & 0x03030303u;
        o[1] = x & 0x0C0C0C0Cu;
        o[2] = y & 0x03030303u;
        o[3] = y & 0x0C0C0C0Cu;
      }
    } else {  // exact BF16 integers: bits of (128 + q) minus 128
      const __nv_bfloat162 base = __floats2bfloat162_rn(128.0f, 128.0f);
      constexpr uint32_t mask = (BITS == 4) ? 0x000F000Fu : 0x00030003u;
#pragma unroll
      for (int k = 0; k < kOut; ++k) {
        uint32_t u = ((x >> (BITS * k)) & mask) | 0x43004300u;
        __nv_bfloat162 v = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&u), base);
        o[k] = *reinterpret_cast<uint32_t*>(&v);
      }
    }
  }
};

// ------------------------------------------------------------ shared state
template <int BITS, bool E2V>
struct alignas(16) DecodeBarriers {
  using C = DecodeCfg<BITS, E2V>;
  uint64_t stg_full[C::kStages], stg_empty[C::kStages];
  // *_empty of the A buffers, Q' slots and P' slots are committed only by
  // kernels that do not wait on the product's own full barrier instead (see
  // kLeanCommits in decode_kernel)
  uint64_t ak_full[C::kNAK], ak_empty[C::kNAK], av_full[C::kNAV], av_empty[C::kNAV];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[C::kSlots], s_empty[C::kSlots], p_full[C::kSlots], p_empty[C::kSlots];
  uint64_t o_full[C::kSlots], o_empty[C::kSlots];
  uint64_t sw_grp, drain;
  float sw_red[2][4][32];  // softmax-group reduction scratch [parity][warp][value]
  int flag;                // split-unit "last arriver" broadcast
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
#ifdef KVQ_PROFILE
  unsigned long long prof[32];  // cycle accounting, flushed to global memory at exit
#endif
#ifdef KVQ_TRACE
  long long trace[kTrN * kTrEv];
#endif
};

template <int BITS, bool E2V>
constexpr size_t decode_smem_layout_bytes() {
  using C = DecodeCfg<BITS, E2V>;
  size_t b = (size_t)C::kStages * C::kStageBytes + (2 + C::kSlots) * (size_t)C::kBBytes +
             (size_t)C::kASmTiles * C::kASmBytes + sizeof(DecodeBarriers<BITS, E2V>) +
             (2 * kMaxBatch + 1) * sizeof(int) + 1024;
  return b < 80 * 1024 ? 80 * 1024 : b;  // >= 80 KB keeps at most two CTAs per SM
}

// --------------------------------------------------------------- helpers
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// All lanes wait (sleeping inside try_wait until the phase completes); the
// warp gives up together, after the time limit or when the CTA has been told
// to abort.
// The slow path (sleeping waits, time limit, abort check) is out of line so
// that the hot loops stay compact in the instruction cache.
static __device__ __noinline__ bool warp_wait_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                            uint64_t limit_ns) {
  uint64_t t0 = 0;
  for (;;) {
    bool ok = mbar_try_wait_sleep(bar, parity, 20000u);
    if (__all_sync(FULL, ok)) return true;
    int stop = 0;
    if (lane_id() == 0) {
      uint64_t now = globaltimer_ns();
      if (t0 == 0) t0 = now;
      stop = (*abort_flag != 0) || (now - t0 > limit_ns);
    }
    if (__shfl_sync(FULL, stop, 0)) return false;
  }
}
// The same loop written in place, for code that runs under a changed
// register budget (setmaxnreg), where no calls can be made.  Kept small:
// several phases share one copy (their barriers and parities go through a
// small local array, touched only on this rare path).
template <int N>
__device__ __forceinline__ bool warp_wait_slow_inline(uint64_t* const (&bars)[N], const uint32_t (&pars)[N],
                                                      volatile int* abort_flag, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
  for (int k = 0; k < N; ++k) {
    for (;;) {
      if (__all_sync(FULL, mbar_try_wait_sleep(bars[k], pars[k], 20000u))) break;
      const bool stop = (*abort_flag != 0) || (globaltimer_ns() - t0 > limit_ns);
      if (__any_sync(FULL, stop)) return false;  // the warp gives up together
    }
  }
  return true;
}

// IL: slow path written in place (true) or out of line (false).
template <bool IL = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
  if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
  if (IL) {
    uint64_t* const bars[1] = {bar};
    const uint32_t pars[1] = {parity};
    return warp_wait_slow_inline<1>(bars, pars, abort_flag, limit_ns);
  }
  return warp_wait_slow(bar, parity, abort_flag, limit_ns);
}

// Two or four phases: one overlapped probe of all of them, then (rarely) the
// one-by-one slow path.
template <bool IL = false>
__device__ __forceinline__ bool warp_wait2(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1,
                                           volatile int* abort_flag, uint64_t limit_ns) {
  if (__all_sync(FULL, mbar_try_wait2(b0, p0, b1, p1))) return true;
  if (IL) {
    uint64_t* const bars[2] = {b0, b1};
    const uint32_t pars[2] = {p0, p1};
    return warp_wait_slow_inline<2>(bars, pars, abort_flag, limit_ns);
  }
  return warp_wait_slow(b0, p0, abort_flag, limit_ns) && warp_wait_slow(b1, p1, abort_flag, limit_ns);
}
template <bool IL = false>
__device__ __forceinline__ bool warp_wait4(uint64_t* b0, uint32_t p0, uint64_t* b1, uint32_t p1, uint64_t* b2,
                                           uint32_t p2, uint64_t* b3, uint32_t p3, volatile int* abort_flag,
                                           uint64_t limit_ns) {
  if (__all_sync(FULL, mbar_try_wait4(b0, p0, b1, p1, b2, p2, b3, p3))) return true;
  if (IL) {
    uint64_t* const bars[4] = {b0, b1, b2, b3};
    const uint32_t pars[4] = {p0, p1, p2, p3};
    return warp_wait_slow_inline<4>(bars, pars, abort_flag, limit_ns);
  }
  return warp_wait_slow(b0, p0, abort_flag, limit_ns) && warp_wait_slow(b1, p1, abort_flag, limit_ns) &&
         warp_wait_slow(b2, p2, abort_flag, limit_ns) && warp_wait_slow(b3, p3, abort_flag, limit_ns);
}

__device__ __forceinline__ void set_abort(volatile int* abort_flag, uint32_t* dev_status) {
  *abort_flag = 1;
  report(dev_status, KVQ_DEV_TIMEOUT);
}

// A four-warp group barrier on an mbarrier (count 4), bounded.
template <bool IL = false>
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, volatile int* abort_flag,
                                           uint64_t limit_ns) {
  __syncwarp();
  if (lane_id() == 0) mbar_arrive(bar);
  bool ok = warp_wait<IL>(bar, phase, abort_flag, limit_ns);
  phase ^= 1u;
  return ok;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
// Warp sums of eight per-lane values in 9 shuffles (a transposing butterfly):
// on return lane l holds the sum of value (l >> 2) & 7.
__device__ __forceinline__ float warp_sum8_transposed(const float (&a)[8]) {
  const int l = lane_id();
  const bool b4 = (l & 16) != 0, b3 = (l & 8) != 0, b2 = (l & 4) != 0;
  float h[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float keep = b4 ? a[4 + j] : a[j], send = b4 ? a[j] : a[4 + j];
    h[j] = keep + __shfl_xor_sync(FULL, send, 16);
  }
  float g[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float keep = b3 ? h[2 + j] : h[j], send = b3 ? h[j] : h[2 + j];
    g[j] = keep + __shfl_xor_sync(FULL, send, 8);
  }
  float f = (b2 ? g[1] : g[0]) + __shfl_xor_sync(FULL, b2 ? g[0] : g[1], 4);
  f += __shfl_xor_sync(FULL, f, 2);
  f += __shfl_xor_sync(FULL, f, 1);
  return f;
}

__device__ __forceinline__ float warp_maxf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

__device__ __forceinline__ float h2f(uint16_t bits) { return __half2float(__ushort_as_half(bits)); }

// Warp maximum of a float in one instruction (NaN inputs are ignored).
__device__ __forceinline__ float warp_max_redux(float f) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(f));
  return r;
}

// Largest of 128 non-negative fp16 values in shared memory; every warp that
// calls it gets the same value without talking to the other warps.
__device__ __forceinline__ uint32_t max_f16_bits_128(const uint16_t* v) {
  uint2 w = *reinterpret_cast<const uint2*>(v + 4 * lane_id());
  const uint32_t m = __vmaxu2(w.x, w.y);  // two 16-bit maxima at once
  return __reduce_max_sync(FULL, max(m & 0xffffu, m >> 16));
}
__device__ __forceinline__ float max_f16_128(const uint16_t* v) { return h2f((uint16_t)max_f16_bits_128(v)); }

__device__ __forceinline__ float bf2f(uint16_t bits) { return __uint_as_float((uint32_t)bits << 16); }

// Per-unit query statistics, computed by each warp on its own (identical in
// every warp): qmax[h] = max_d |q[h, d]|, qsum[h] = sum_d q[h, d] for the
// unit's `rows` consecutive query heads starting at qb (16-byte aligned rows
// of 128 bf16); heads rows..NH-1 do not exist (fewer query heads per KV head)
// and read as zero.
template <int NH>
__device__ __forceinline__ void unit_q_stats(const uint16_t* qb, int rows, bool need_sum, float (&qmax)[NH],
                                             float (&qsum)[NH]) {
#pragma unroll
  for (int h = 0; h < NH; ++h) {
    // an empty slot re-reads row 0 (always valid memory) and is zeroed: no branch
    const float keep = h < rows ? 1.0f : 0.0f;
    uint2 w = *reinterpret_cast<const uint2*>(qb + (h < rows ? h : 0) * kHeadDim + 4 * lane_id());
    float x0 = bf2f((uint16_t)(w.x & 0xffffu)) * keep, x1 = bf2f((uint16_t)(w.x >> 16)) * keep;
    float x2 = bf2f((uint16_t)(w.y & 0xffffu)) * keep, x3 = bf2f((uint16_t)(w.y >> 16)) * keep;
    float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3)));
    qmax[h] = __uint_as_float(__reduce_max_sync(FULL, __float_as_uint(m)));
    qsum[h] = need_sum ? warp_sum((x0 + x1) + (x2 + x3)) : 0.0f;
  }
}

// Walks the global tile order (sequence-major, then KV head, then block).
struct TileIter {
  int b, h, j, nblk;
  __device__ __forceinline__ void init(const int* prefix, int B, int Hkv, int g) {
    int lo = 0, hi = B;  // prefix[lo] <= g < prefix[hi]
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (prefix[mid] <= g) lo = mid; else hi = mid;
    }
    b = lo;
    nblk = (prefix[b + 1] - prefix[b]) / Hkv;
    int r = g - prefix[b];
    h = r / nblk;
    j = r - h * nblk;
  }
  template <bool IL = false>
  __device__ __forceinline__ void next(const int* prefix, int B, int Hkv);
};

// Next (sequence, kv head) unit after (b, h): {b, h, nblk}; out of line (it
// runs once per unit) to keep the hot loops compact.
__device__ __forceinline__ int3 next_unit_inline(int b, int h, int nblk, const int* prefix, int B, int Hkv) {
  if (++h < Hkv) return make_int3(b, h, nblk);
  h = 0;
  do { ++b; } while (b < B && prefix[b + 1] == prefix[b]);
  if (b < B) nblk = (prefix[b + 1] - prefix[b]) / Hkv;
  return make_int3(b, h, nblk);
}
static __device__ __noinline__ int3 next_unit(int b, int h, int nblk, const int* prefix, int B, int Hkv) {
  return next_unit_inline(b, h, nblk, prefix, B, Hkv);
}
template <bool IL>
__device__ __forceinline__ void TileIter::next(const int* prefix, int B, int Hkv) {
  if (++j < nblk) return;
  j = 0;
  const int3 u = IL ? next_unit_inline(b, h, nblk, prefix, B, Hkv) : next_unit(b, h, nblk, prefix, B, Hkv);
  b = u.x; h = u.y; nblk = u.z;
}

__device__ __forceinline__ int cta_of_tile(long long t, long long T, int C) {
  return (int)(((t + 1) * C - 1) / T);
}
__device__ __forceinline__ long long range_start(int c, long long T, int C) { return (long long)c * T / C; }

// Per-unit set-up, out of line (once per unit).
// Converter thread r: q[i, r] of the unit's query head i times that head's Q'
// prescale (0 for the head slots a unit with fewer than 4 heads leaves empty).
template <bool KCW>
static __device__ __noinline__ float4 converter_unit_q(const uint16_t* qb, int rows, int r) {
  float qmax[4], qsum[4];
  unit_q_stats<4>(qb, rows, false, qmax, qsum);
  float qh[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    qh[i] = bf2f(qb[(i < rows ? i : 0) * kHeadDim + r]) * (i < rows ? 1.0f : 0.0f) *
            (KCW ? pow2_head(qmax[i]) : pow2_prescale(qmax[i]));
  return make_float4(qh[0], qh[1], qh[2], qh[3]);
}
// Softmax thread i: per-head score constants of the unit.  Channel-wise K:
// add = the unit's part of the score multiplier, qi = q[k, i] of the unit's
// head k; token-wise K: S = s_l * (q . code) * mult + z_l * add.  Empty head
// slots get zero constants (their scores are 0 and never written out).
struct SegConsts {
  float qi[4], mult[4], add[4];
};
template <bool KCW>
static __device__ __forceinline__ SegConsts softmax_unit_consts(const uint16_t* qb, int rows, int i,
                                                               float sm_scale_log2, float code_inv) {
  float qmax[4], qsum[4];
  unit_q_stats<4>(qb, rows, !KCW, qmax, qsum);
  SegConsts c;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (KCW) {
      c.qi[k] = bf2f(qb[(k < rows ? k : 0) * kHeadDim + i]) * (k < rows ? 1.0f : 0.0f);
      c.mult[k] = 0.f;
      c.add[k] = code_inv * pow2_head_inv(qmax[k]) * sm_scale_log2;
    } else {
      c.qi[k] = 0.f;
      c.mult[k] = code_inv * pow2_prescale_inv(qmax[k]) * sm_scale_log2;
      c.add[k] = qsum[k] * sm_scale_log2;
    }
  }
  return c;
}

// ================================================================= kernel
// GQ4: exactly 4 query heads per KV head (one unit per KV head, no empty
// head slots); the other groupings (1, 2, 8) take the run-time values in p.
template <int BITS, bool KCW, bool VCW, bool GQ4, bool E2V>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_kernel(const DecodeParams p) {
  using C = DecodeCfg<BITS, E2V>;
  using Bars = DecodeBarriers<BITS, E2V>;
  // Lean commits: each product commits only its full barrier (S or O slot)
  // and the buffers it read are reused on that phase.  Measured faster with
  // token-wise K (INT2: +6% K-tw/V-tw, +2% K-tw/V-cw) and slower with
  // channel-wise K (-3%), which keeps the separate release barriers.
  constexpr bool kLeanCommits = !KCW;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* stages = smem_raw;
  unsigned char* qop = stages + (size_t)C::kStages * C::kStageBytes;  // [2][kBBytes]
  unsigned char* pop = qop + 2 * C::kBBytes;                          // [kSlots][kBBytes]
  unsigned char* asm_tiles = pop + C::kSlots * C::kBBytes;             // [kASmTiles][kASmBytes] E2M1 codes
  Bars& sh = *reinterpret_cast<Bars*>(asm_tiles + C::kASmTiles * C::kASmBytes);
  int* prefix = reinterpret_cast<int*>(&sh + 1);  // [B + 1] tile offsets
  int* lens = prefix + (kMaxBatch + 1);           // [B] validated sequence lengths

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Units: (sequence, unit head) pairs.  A unit holds up to 4 query heads
  // (gq) of one KV head; with 8 query heads per KV head there are two units
  // per KV head (unit head u reads KV head u >> kv_shift).
  const int B = p.batch, Hkv = GQ4 ? p.num_kv_heads : p.units_per_seq;
  const int gq = GQ4 ? kGroupQ : p.gq, kv_shift = GQ4 ? 0 : p.kv_shift;
  const int cta = blockIdx.x;
  volatile int* abort_flag = &sh.abort_flag;
  const uint64_t limit = p.wait_limit_ns;

  // ------------------------------------------------------------ set-up
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) { mbar_init(&sh.stg_full[s], 1); mbar_init(&sh.stg_empty[s], 8); }
    for (int a = 0; a < C::kNAK; ++a) { mbar_init(&sh.ak_full[a], 4); mbar_init(&sh.ak_empty[a], 1); }
    for (int a = 0; a < C::kNAV; ++a) { mbar_init(&sh.av_full[a], 4); mbar_init(&sh.av_empty[a], 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(&sh.q_full[s], 4); mbar_init(&sh.q_empty[s], 1); }
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&sh.s_full[s], 1); mbar_init(&sh.s_empty[s], 4);
      mbar_init(&sh.p_full[s], 4); mbar_init(&sh.p_empty[s], 1);
      mbar_init(&sh.o_full[s], 1); mbar_init(&sh.o_empty[s], 4);
    }
    mbar_init(&sh.sw_grp, 4);
#ifdef KVQ_PROFILE
    for (int s = 0; s < 32; ++s) sh.prof[s] = 0ull;
#endif
#ifdef KVQ_TRACE
    for (int j = 0; j < kTrN * kTrEv; ++j) sh.trace[j] = 0;
#endif
    mbar_init(&sh.drain, 1);
    sh.abort_flag = 0;
    fence_barrier_init();
  }
  // validated lengths and the tile prefix (sequence-major)
  for (int b = tid; b < B; b += kDecodeThreads) {
    int len = p.seq_lens[b];
    if (len < 0 || len > p.max_blocks * kBlockTokens) {
      if (cta == 0) report(p.dev_status, KVQ_DEV_BAD_SEQ_LEN);
      len = 0;
    }
    lens[b] = len;
  }
  // operand columns nobody writes (N = 12..15) stay zero
  // (and the padding half of every E2M1 unit, which the converters never write)
  for (int i = tid; i < ((2 + C::kSlots) * C::kBBytes + C::kASmTiles * C::kASmBytes) / 16; i += kDecodeThreads)
    reinterpret_cast<uint4*>(qop)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (warp == kWarpMma) { tmem_alloc(&sh.tmem_base, C::kTmemCols); tmem_relinquish(); }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      prefix[b] = acc;
      acc += Hkv * ((lens[b] + kBlockTokens - 1) / kBlockTokens);
    }
    prefix[B] = acc;
    sh.total_tiles = acc;
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  const long long T = sh.total_tiles;
  // Tile ranges are cut over min(grid, T) CTAs so that every active CTA owns
  // at least one tile (the split-unit merge counts one part per CTA between a
  // unit's first and last owner); the remaining CTAs only write empty rows.
  const int Cn = (int)(T < (long long)gridDim.x ? T : (long long)gridDim.x);
  const bool active = cta < Cn;
  const long long g0 = active ? range_start(cta, T, Cn) : 0;
  const long long g1 = active ? range_start(cta + 1, T, Cn) : 0;
  const int ntiles = (int)(g1 - g0);

  // Each role leaves through finish_cta() and returns: code after the role
  // branches would be shared by warps with different register budgets.
  auto finish_cta = [&]() {
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
      tc_fence_after();
      tmem_dealloc(tmem, C::kTmemCols);
    }
#if defined(KVQ_PROFILE) && !defined(KVQ_TRACE)
    if (p.prof != nullptr && tid < 32) atomicAdd(&p.prof[blockIdx.x * 32 + tid], sh.prof[tid]);
#endif
#ifdef KVQ_TRACE
    if (p.prof != nullptr)
      for (int j = tid; j < kTrN * kTrEv; j += kDecodeThreads) p.prof[(size_t)blockIdx.x * kTrN * kTrEv + j] = sh.trace[j];
#endif
  };

  if (warp >= kWarpLoad) {
    setmaxnreg_dec<kRegsLight>();
    // ========================================================== loader
    if (warp == kWarpLoad && lane == 0 && ntiles > 0) {
      const uint64_t policy = l2_policy_evict_first();
      uint32_t issued = 0u, issued_par = 0u;  // per stage: a copy was issued / its phase parity
      TileIter it;
      it.init(prefix, B, Hkv, (int)g0);
      for (int t = 0; t < ntiles; ++t, it.next<true>(prefix, B, Hkv)) {
        const int s = t % C::kStages;
        const uint32_t ph = (uint32_t)(t / C::kStages) & 1u;
        KVQ_PT(le)
        if (!mbar_wait_bounded<true>(&sh.stg_empty[s], ph ^ 1u, abort_flag, limit)) {
          set_abort(abort_flag, p.dev_status);
          break;
        }
        KVQ_PA(0, le)
        if ((p.flags & KVQ_FLAG_TEST_STALL) && cta == 0 && t == 1) continue;  // withhold one tile
        int page = p.page_table ? p.page_table[(size_t)it.b * p.max_blocks + it.j] : it.b * p.max_blocks + it.j;
        if (page < 0 || page >= p.num_pages) {
          report(p.dev_status, KVQ_DEV_BAD_PAGE);
          page = 0;
        }
        const size_t blk = (size_t)page * p.num_kv_heads + (it.h >> kv_shift);
        unsigned char* st = stages + (size_t)s * C::kStageBytes;
        mbar_arrive_expect_tx(&sh.stg_full[s], C::kStageBytes);
        bulk_g2s_evict_first(st, p.k_codes + blk * C::kBlockBytes, C::kBlockBytes, &sh.stg_full[s], policy);
        bulk_g2s_evict_first(st + C::kBlockBytes, p.v_codes + blk * C::kBlockBytes, C::kBlockBytes, &sh.stg_full[s],
                             policy);
        unsigned char* sz = st + 2 * C::kBlockBytes;
        bulk_g2s_evict_first(sz, p.k_scale + blk * kBlockTokens, C::kSzBytes, &sh.stg_full[s], policy);
        bulk_g2s_evict_first(sz + C::kSzBytes, p.k_zero + blk * kBlockTokens, C::kSzBytes, &sh.stg_full[s], policy);
        bulk_g2s_evict_first(sz + 2 * C::kSzBytes, p.v_scale + blk * kBlockTokens, C::kSzBytes, &sh.stg_full[s],
                             policy);
        bulk_g2s_evict_first(sz + 3 * C::kSzBytes, p.v_zero + blk * kBlockTokens, C::kSzBytes, &sh.stg_full[s],
                             policy);
        issued |= 1u << s;
        issued_par = (issued_par & ~(1u << s)) | (ph << s);
        KVQ_TR(21, t)
      }
      // never leave a copy in flight: wait for every issued stage to land
      for (int s = 0; s < C::kStages; ++s)
        if (issued & (1u << s)) mbar_wait_bounded<true>(&sh.stg_full[s], (issued_par >> s) & 1u, nullptr, limit);
    }
  // ================================================================ MMA
  // Issues QK^T of tile nq and PV of tile np in whatever order their inputs
  // become ready (non-blocking tests), so neither product waits behind the
  // other.  QK^T(t): A = K codes, B = Q', D = S slot.  PV(t): A = V codes,
  // B = P', D = O slot.
    else if (warp == kWarpMma && lane == 0 && ntiles > 0) {
      bool ok = true;
      int nq = 0, np = 0;
      uint64_t idle_since = 0;
      uint32_t backoff = 32;
      while (np < ntiles) {
        bool progressed = false;
        if (np < nq) {
          const int a = np % C::kNAV, sl = np % C::kSlots;
          const uint32_t pa = (uint32_t)(np / C::kNAV) & 1u, ps4 = (uint32_t)(np / C::kSlots) & 1u;
          if (mbar_test3(&sh.av_full[a], pa, &sh.p_full[sl], ps4, &sh.o_empty[sl], ps4 ^ 1u)) {
            tc_fence_after();
            const uint32_t b0 = smem_u32(pop + sl * C::kBBytes);
#pragma unroll
            for (int k = 0; k < C::kKSteps; ++k) {
              uint64_t bd = make_smem_desc(b0 + k * C::kKStepBBytes, C::kLbo, C::kSbo);
              uint32_t d = tmem + C::kColO + 16 * sl, av = tmem + C::kColAV + a * C::kACols + 8 * k;
              if (C::kE2V)  // A = E2M1 tile in shared memory; K-step k = K-groups 2k, 2k + 1
                mma_f8f6f4_ss(d, make_smem_desc(smem_u32(asm_tiles + a * C::kASmBytes) + 2 * k * C::kALbo, C::kALbo,
                                                C::kASbo),
                              bd, C::kIdescV, k > 0);
              else mma_f8f6f4_ts(d, av, bd, C::kIdesc, k > 0);
            }
            if (!kLeanCommits) {
              tc_commit(&sh.av_empty[a]);
              tc_commit(&sh.p_empty[sl]);
            }
            tc_commit(&sh.o_full[sl]);
            KVQ_TR(17, np)
            ++np;
            progressed = true;
          }
        }
        if (nq < ntiles) {
          const int a = nq % C::kNAK, sl = nq % C::kSlots, q2 = nq & 1;
          const uint32_t pa = (uint32_t)(nq / C::kNAK) & 1u, ps4 = (uint32_t)(nq / C::kSlots) & 1u,
                         p2 = (uint32_t)(nq >> 1) & 1u;
          if (mbar_test3(&sh.ak_full[a], pa, &sh.q_full[q2], p2, &sh.s_empty[sl], ps4 ^ 1u)) {
            tc_fence_after();
            const uint32_t b0 = smem_u32(qop + q2 * C::kBBytes);
#pragma unroll
            for (int k = 0; k < C::kKSteps; ++k) {
              uint64_t bd = make_smem_desc(b0 + k * C::kKStepBBytes, C::kLbo, C::kSbo);
              uint32_t d = tmem + C::kColS + 16 * sl, ak = tmem + C::kColAK + a * C::kACols + 8 * k;
              mma_f8f6f4_ts(d, ak, bd, C::kIdesc, k > 0);
            }
            if (!kLeanCommits) {
              tc_commit(&sh.ak_empty[a]);
              tc_commit(&sh.q_empty[q2]);
            }
            tc_commit(&sh.s_full[sl]);
            KVQ_TR(16, nq)
            ++nq;
            progressed = true;
          }
        }
        if (progressed) {
          idle_since = 0;
          backoff = 32;
        } else {
          __nanosleep(backoff);  // back off: leave issue slots to the warps sharing this sub-partition
          backoff = backoff < 512 ? 2 * backoff : 512;
          const uint64_t now = globaltimer_ns();
          if (idle_since == 0) idle_since = now;
          if (*abort_flag || now - idle_since > limit) { ok = false; break; }
        }
      }
      if (!ok) set_abort(abort_flag, p.dev_status);
      // drain: all issued MMAs complete before tensor memory is released
      tc_commit(&sh.drain);
      mbar_wait_bounded<true>(&sh.drain, 0, nullptr, limit);
    }
    finish_cta();
    return;
  }
  // ========================================================== converters
  // Software-pipelined: Q' and K of tile t + 1 are produced before V of tile
  // t, so QK^T runs a tile ahead and never waits behind an earlier PV.
  else if (warp < kWarpSoftmax0) {
    setmaxnreg_inc<kRegsConvert>();
    const int r = tid;  // tensor-memory lane = A row; also this thread's channel of Q'
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int qrow = a_pos<BITS, false>(r);
    float qh[4] = {0.f, 0.f, 0.f, 0.f};  // q[b, 4h + i, r] times the head's prescale
    int seg = -1, slot_seg0 = -2, slot_seg1 = -2;  // Q' slot contents (token-wise K: constant per segment)
    TileIter it;
    if (ntiles > 0) it.init(prefix, B, Hkv, (int)g0);

    // codes of one packed row -> tensor-memory row (32 columns per store)
    auto convert_rows = [&](const unsigned char* blk, uint32_t col) {
      constexpr int kPasses = C::kACols / 32, kPerPass = C::kChunks / kPasses;
#pragma unroll
      for (int ps2 = 0; ps2 < kPasses; ++ps2) {
        uint32_t o[32];
#pragma unroll
        for (int c = 0; c < kPerPass; ++c) {
          uint4 v = *reinterpret_cast<const uint4*>(blk + ((size_t)(ps2 * kPerPass + c) * kBlockTokens + r) * 16);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            Convert<BITS, false>::run(w[i], &o[(4 * c + i) * Convert<BITS, false>::kOut], p.nibble_mul, p.minus_one);
        }
        tmem_st_32x32b_x32(col + 32 * ps2, o);
      }
    };
    // 2-bit codes of one packed row -> E2M1 (code / 2) nibbles in a shared-
    // memory tile: per 32-bit word (16 codes) the even codes (x & 0x33333333)
    // then the odd ones ((x >> 2) & 0x33333333), 3 operations per 16 codes
    // (rag-lover.com summary of arXiv 2611.09722, "解説": 2-bit codes in the
    // low bits of an E2M1 element read as q / 2).
    auto convert_rows_e2m1 = [&](const unsigned char* blk, unsigned char* tile) {
      unsigned char* row = tile + (r >> 3) * C::kASbo + (r & 7) * 16;
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(blk + ((size_t)c * kBlockTokens + r) * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)  // K-group 4c + i holds codes 16 (4c + i) ... + 15
          *reinterpret_cast<uint2*>(row + (4 * c + i) * C::kALbo) =
              make_uint2(w[i] & 0x33333333u, (w[i] >> 2) & 0x33333333u);
      }
    };

    // stage wait, Q' operand and K codes of tile t (it = tile t).  A_K[a] and
    // Q' slot t & 1 are free once QK^T(t - kNAK) has completed; with lean
    // commits that is the phase of its S slot (kNAK <= 2, and the products
    // complete in issue order).
    auto k_part = [&](int t) -> bool {
      const int s = t % C::kStages, a = t % C::kNAK, sl = t & 1;
      const uint32_t ps = (uint32_t)(t / C::kStages) & 1u, pa = (uint32_t)(t / C::kNAK) & 1u,
                     p2 = (uint32_t)(t >> 1) & 1u;
      const int tp = t - C::kNAK;
      KVQ_PT(c0)
      if (kLeanCommits ? (tp < 0 ? !warp_wait<true>(&sh.stg_full[s], ps, abort_flag, limit)
                                 : !warp_wait2<true>(&sh.stg_full[s], ps, &sh.s_full[tp % C::kSlots],
                                                     (uint32_t)(tp / C::kSlots) & 1u, abort_flag, limit))
                       : !warp_wait4<true>(&sh.stg_full[s], ps, &sh.q_empty[sl], p2 ^ 1u, &sh.ak_empty[a], pa ^ 1u,
                                           &sh.ak_empty[a], pa ^ 1u, abort_flag, limit))
        return false;
      KVQ_PA(1, c0)
      const unsigned char* st = stages + (size_t)s * C::kStageBytes;
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(st + 2 * C::kBlockBytes);
      if (t == 0 || it.j == 0) {  // new (sequence, kv head): its four query rows
        ++seg;
        const float4 q4 =
            converter_unit_q<KCW>(p.q + ((size_t)it.b * p.num_q_heads + (size_t)it.h * gq) * kHeadDim, gq, r);
        qh[0] = q4.x; qh[1] = q4.y; qh[2] = q4.z; qh[3] = q4.w;
      }
      // Q' operand: token-wise K uses q (written once per segment per slot);
      // channel-wise K folds this group's scales into q.
      KVQ_PT(c4)
      KVQ_PA(5, c4)
      KVQ_PT(c3)
      if (KCW || (sl ? slot_seg1 : slot_seg0) != seg) {
        float f = odd_quarter<BITS, false>(r);
        if (KCW) f *= h2f(ks[r]) * pow2_group(f16_exp_field(max_f16_bits_128(ks)));
        const float4 v = make_float4(qh[0] * f, qh[1] * f, qh[2] * f, qh[3] * f);
        *reinterpret_cast<uint4*>(qop + sl * C::kBBytes + b_row_off(qrow)) = split3_e4m3(v);
        fence_proxy_async_smem();
        if (sl) slot_seg1 = seg; else slot_seg0 = seg;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.q_full[sl]);
      KVQ_PA(4, c3)
      // K codes -> A_K[a] (row r = token r)
      KVQ_PT(c1)
      KVQ_PA(2, c1)
      KVQ_PT(c2)
      convert_rows(st, tmem + lane_off + C::kColAK + a * C::kACols);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.ak_full[a]);
      KVQ_PA(7, c2)
      KVQ_TR(0 + warp, t)
      return true;
    };

    // V codes of tile t -> A_V[a] (row r = channel r); releases the stage.
    // A_V[a] is free once PV(t - kNAV) has completed (lean commits: the phase
    // of its O slot).
    auto v_part = [&](int t) -> bool {
      const int s = t % C::kStages, a = t % C::kNAV;
      const uint32_t pa = (uint32_t)(t / C::kNAV) & 1u;
      const int tp = t - C::kNAV;
      KVQ_PT(c5)
      if (kLeanCommits ? (tp >= 0 && !warp_wait<true>(&sh.o_full[tp % C::kSlots], (uint32_t)(tp / C::kSlots) & 1u,
                                                      abort_flag, limit))
                       : !warp_wait<true>(&sh.av_empty[a], pa ^ 1u, abort_flag, limit))
        return false;
      KVQ_PA(6, c5)
      KVQ_PT(c6)
      if (C::kE2V) {
        convert_rows_e2m1(stages + (size_t)s * C::kStageBytes + C::kBlockBytes, asm_tiles + a * C::kASmBytes);
        fence_proxy_async_smem();  // visible to the tensor core
      } else {
        convert_rows(stages + (size_t)s * C::kStageBytes + C::kBlockBytes, tmem + lane_off + C::kColAV + a * C::kACols);
        tc_wait_st();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.av_full[a]);
        mbar_arrive(&sh.stg_empty[s]);
      }
      KVQ_PA(8, c6)
      KVQ_TR(4 + warp, t)
      return true;
    };

    bool ok = ntiles == 0 || k_part(0);
    if (ntiles > 0) it.next(prefix, B, Hkv);
    for (int t = 0; t < ntiles && ok; ++t) {
      if (t + 1 < ntiles) {
        ok = k_part(t + 1);
        it.next(prefix, B, Hkv);
        if (!ok) break;
      }
      ok = v_part(t);
    }
    if (!ok) set_abort(abort_flag, p.dev_status);
    finish_cta();
    return;
  }
  // ============================================================= softmax
  // Two tiles of one (sequence, kv head) per step: the fixed per-step costs
  // (waits, the cross-warp reduction round, bookkeeping) are paid once per
  // pair, and both tiles share one running-max update.
  else {
    setmaxnreg_inc<kRegsSoftmax>();
    const int i = tid - kWarpSoftmax0 * 32;  // tensor-memory lane: token (scores) / channel (output)
    const int sw = warp - kWarpSoftmax0;     // warp = lane quarter
    const uint32_t lane_off = (uint32_t)(sw * 32) << 16;
    const int prow = a_pos<BITS, false, C::kE2V>(i);
    uint32_t grp_phase = 0;
    const float kLn2 = 0.69314718055994530942f;
    const float kFix = 67108864.0f;  // 2^26: fixed-point scale of p for integer warp sums
    // reduction-round payload slots: [0,8) score maxima, per tile for
    // channel-wise K (value tile * 4 + head), per pair for token-wise K (value
    // head); [8,16) channel-wise K offsets q.z_g (tile * 4 + head); [16,24)
    // channel-wise V previous tiles' sum(p); 24: token-wise V largest scale
    // of the pair
    constexpr int kTM = 0, kCG = 8, kWS = 16, kVM = 24, kNV = 26;
    const bool lane_max = (lane < kCG) || (lane >= kVM);  // lane's value combines by max, else by sum

    // empty sequences: out = 0, lse = -inf
    for (int b = cta; b < B; b += (int)gridDim.x) {
      if (lens[b] != 0) continue;
      for (int hq = 0; hq < p.num_q_heads; ++hq) {
        p.out[((size_t)b * p.num_q_heads + hq) * kHeadDim + i] = 0.0f;
        if (i == 0) p.lse[(size_t)b * p.num_q_heads + hq] = -INFINITY;
      }
    }

    float m[4], lp[4], zp[4], O[4];  // running max (log2 units), partial sum p, partial sum p*z, output
    // deferred epilogue inputs of the previous step (up to two tiles)
    int pend = -1, pend_n = 0;
    float a_prev[4], ws_prev[8], sv_prev[2], zv_prev[2];
    uint32_t pexp_prev = 0u;  // P' prescale exponents E of the previous step, one signed byte per head
    constexpr int kCodeLog2 = C::kVCodeLog2;  // log2 of the V code scale
    float qi[4], qmax[4], mult[4], add[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) { qi[k] = 0.f; qmax[k] = 0.f; mult[k] = 0.f; add[k] = 0.f; a_prev[k] = 0.f; }
#pragma unroll
    for (int k = 0; k < 8; ++k) ws_prev[k] = 0.f;
    sv_prev[0] = sv_prev[1] = zv_prev[0] = zv_prev[1] = 0.f;
    auto reset = [&]() {
#pragma unroll
      for (int k = 0; k < 4; ++k) { m[k] = -INFINITY; lp[k] = 0.f; zp[k] = 0.f; O[k] = 0.f; }
    };
    reset();

    // One cross-warp round: lane 0 of every warp publishes `vals`, then lane
    // v merges value v over the four warps and the results are broadcast.
    // `used` (bit v = value v) selects the values published and broadcast;
    // callers pass compile-time masks.
    // Optionally also waits, in the same probe as the group barrier, for two
    // more phases (xa, xb; null: none).
    auto round = [&](const float (&vals)[kNV], float (&res)[kNV], uint32_t used, bool cg_dist = false,
                     float cg = 0.f, uint64_t* xa = nullptr, uint32_t pxa = 0u, uint64_t* xb = nullptr,
                     uint32_t pxb = 0u) -> bool {
      float* red = sh.sw_red[grp_phase][sw];
      if (cg_dist && (lane & 3) == 0) red[kCG + (lane >> 2)] = cg;
      const uint32_t used_all = used;
      if (cg_dist) used &= ~(0xffu << kCG);
      if (lane == 0) {
#pragma unroll
        for (int v = 0; v < kNV; v += 2) {
          const uint32_t two = (used >> v) & 3u;
          if (two == 3u) *reinterpret_cast<float2*>(red + v) = make_float2(vals[v], vals[v + 1]);
          else if (two == 1u) red[v] = vals[v];
          else if (two == 2u) red[v + 1] = vals[v + 1];
        }
      }
      const uint32_t use = grp_phase;
      if (xa != nullptr) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.sw_grp);
        const bool okw = warp_wait4<true>(&sh.sw_grp, grp_phase, xa, pxa, xb, pxb, xb, pxb, abort_flag, limit);
        grp_phase ^= 1u;
        if (!okw) return false;
      } else if (!group_sync<true>(&sh.sw_grp, grp_phase, abort_flag, limit)) {
        return false;
      }
      const int v = lane < kNV ? lane : 0;
      const float r0 = sh.sw_red[use][0][v], r1 = sh.sw_red[use][1][v];
      const float r2 = sh.sw_red[use][2][v], r3 = sh.sw_red[use][3][v];
      const float mine = lane_max ? fmaxf(fmaxf(r0, r1), fmaxf(r2, r3)) : (r0 + r1) + (r2 + r3);
#pragma unroll
      for (int k = 0; k < kNV; ++k) res[k] = ((used_all >> k) & 1u) ? __shfl_sync(FULL, mine, k) : 0.f;
      return true;
    };

    // PV epilogue of the previous step's tiles: O = O * alpha + folded partial products
    // Both partial products are awaited and loaded together (a lone tile is
    // loaded twice and its copy masked out).
    auto epilogue = [&](const float (&ts)[8]) -> bool {
      const int tA = pend, tB = pend_n > 1 ? pend + 1 : pend;
      const int oA = tA % C::kSlots, oB = tB % C::kSlots;
      KVQ_PT(e0)
      if (!warp_wait2<true>(&sh.o_full[oA], (uint32_t)(tA / C::kSlots) & 1u, &sh.o_full[oB], (uint32_t)(tB / C::kSlots) & 1u,
                      abort_flag, limit))
        return false;
      KVQ_PA(23, e0)

      tc_fence_after();
      uint32_t acc[2][12];
      tmem_ld_parts(tmem + lane_off + C::kColO + 16 * oA, acc[0]);
      tmem_ld_parts(tmem + lane_off + C::kColO + 16 * oB, acc[1]);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.o_empty[oA]);
        if (pend_n > 1) mbar_arrive(&sh.o_empty[oB]);
      }
      { KVQ_TR(12 + sw, tA) if (pend_n > 1) KVQ_TR(12 + sw, tB) }
#pragma unroll
      for (int k = 0; k < 4; k += 2) {  // heads k, k + 1
        const float2 pinv = make_float2(p_inverse(pexp_prev, k, kCodeLog2), p_inverse(pexp_prev, k + 1, kCodeLog2));
        float2 o[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          o[u] = add2(f2u(acc[u][k], acc[u][k + 1]), f2u(acc[u][4 + k], acc[u][5 + k]));
          o[u] = add2(o[u], f2u(acc[u][8 + k], acc[u][9 + k]));
          o[u] = mul2(o[u], pinv);
        }
        if (pend_n < 2) o[1] = f2s(0.f);
        const float2 o_add =
            VCW ? add2(fma2(f2s(sv_prev[0]), o[0], mul2(f2s(zv_prev[0]), make_float2(ts[k], ts[k + 1]))),
                       fma2(f2s(sv_prev[1]), o[1], mul2(f2s(zv_prev[1]), make_float2(ts[4 + k], ts[5 + k]))))
                : add2(o[0], o[1]);
        const float2 o2 = fma2(make_float2(O[k], O[k + 1]), make_float2(a_prev[k], a_prev[k + 1]), o_add);
        O[k] = o2.x;
        O[k + 1] = o2.y;
      }
      return true;
    };

    // Cross-warp sums of the previous step's per-warp p sums (channel-wise V),
    // for a drain that has no following step to carry them.
    auto combine_prev_sums = [&](float (&ts)[8]) -> bool {
      float vals[kNV], res[kNV];
#pragma unroll
      for (int k = 0; k < kNV; ++k) vals[k] = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) vals[kWS + k] = ws_prev[k];
      if (!round(vals, res, 0xffu << kWS)) return false;
#pragma unroll
      for (int k = 0; k < 8; ++k) ts[k] = res[kWS + k];
      return true;
    };

    // finish a (sequence, kv head) segment: normalise, store or merge
    auto finalize = [&](int b, int h, bool first_global, bool last_global, long long ustart, long long uend) -> bool {
      float vals[kNV], res[kNV];
#pragma unroll
      for (int k = 0; k < kNV; ++k) vals[k] = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) { vals[kCG + k] = warp_sum(lp[k]); vals[kCG + 4 + k] = VCW ? 0.f : warp_sum(zp[k]); }
      if (!round(vals, res, 0xffu << kCG)) return false;
      float out4[4], lse4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float l = res[kCG + k], z = res[kCG + 4 + k];
        out4[k] = (O[k] + z) / l;
        lse4[k] = (m[k] + __log2f(l)) * kLn2;
      }
      const size_t row0 = (size_t)b * p.num_q_heads + (size_t)h * gq;
      if (first_global && last_global) {  // whole (sequence, head) in this CTA
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (k >= gq) break;  // empty head slots
          p.out[(row0 + k) * kHeadDim + i] = out4[k];
          if (i == k) p.lse[row0 + k] = lse4[k];
        }
        return true;
      }
      // split: publish this part; the last part to arrive merges all parts
      const int c_first = cta_of_tile(ustart, T, Cn), c_last = cta_of_tile(uend - 1, T, Cn);
      const int slot = (ustart <= g0) ? 0 : 1;
      float* po = p.part_o + ((size_t)cta * 2 + slot) * kGroupQ * kHeadDim;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        po[k * kHeadDim + i] = out4[k];
        if (i == k) p.part_lse[((size_t)cta * 2 + slot) * kGroupQ + k] = lse4[k];
      }
      __threadfence();
      if (!group_sync<true>(&sh.sw_grp, grp_phase, abort_flag, limit)) return false;
      const int u = b * Hkv + h;
      if (i == 0) {
        int old = atomicAdd(&p.counters[u], 1);
        sh.flag = (old == c_last - c_first) ? 1 : 0;
      }
      if (!group_sync<true>(&sh.sw_grp, grp_phase, abort_flag, limit)) return false;
      if (!sh.flag) return true;
      __threadfence();
      float mx[4], den[4], acc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) { mx[k] = -INFINITY; den[k] = 0.f; acc[k] = 0.f; }
      for (int c = c_first; c <= c_last; ++c) {
        const int sl2 = (ustart <= range_start(c, T, Cn)) ? 0 : 1;
        const float* pl = p.part_lse + ((size_t)c * 2 + sl2) * kGroupQ;
        const float* pv = p.part_o + ((size_t)c * 2 + sl2) * kGroupQ * kHeadDim;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float l = __ldcg(pl + k), v = __ldcg(pv + k * kHeadDim + i);
          float nm = fmaxf(mx[k], l);
          float sc = __expf(mx[k] - nm), w = __expf(l - nm);
          den[k] = den[k] * sc + w;
          acc[k] = acc[k] * sc + w * v;
          mx[k] = nm;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (k >= gq) break;
        p.out[(row0 + k) * kHeadDim + i] = acc[k] / den[k];
        if (i == k) p.lse[row0 + k] = mx[k] + __logf(den[k]);
      }
      if (i == 0) p.counters[u] = 0;
      return true;
    };

    auto drain = [&](void) -> bool {
      float ts[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ts[k] = 0.f;
      return (!VCW || combine_prev_sums(ts)) && epilogue(ts);
    };

    TileIter it;
    if (ntiles > 0) it.init(prefix, B, Hkv, (int)g0);
    int pb = 0, ph = 0;
    bool pfirst = false;
    long long pus = 0, pue = 0;
    bool ok = true;
    for (int t = 0; t < ntiles && ok;) {
      const long long g = g0 + t;
      const long long ustart = g - it.j, uend = ustart + it.nblk;
      const bool seg_first = (t == 0) || it.j == 0;
      if (seg_first && pend_n > 0) {  // close the previous segment
        KVQ_PT(f0)
        ok = drain() && finalize(pb, ph, pfirst, pue <= g1, pus, pue);
        KVQ_PA(24, f0)
        if (!ok) break;
        reset();
        pend_n = 0;
      }
      if (seg_first) {
        pb = it.b; ph = it.h; pfirst = ustart >= g0; pus = ustart; pue = uend;
        const SegConsts sc4 = softmax_unit_consts<KCW>(
            p.q + ((size_t)it.b * p.num_q_heads + (size_t)it.h * gq) * kHeadDim, gq, i, p.sm_scale_log2,
            C::kCodeInv);
#pragma unroll
        for (int k = 0; k < 4; ++k) { qi[k] = sc4.qi[k]; mult[k] = sc4.mult[k]; add[k] = sc4.add[k]; }
      }
      // this step: tile t and, if it belongs to the same segment, tile t + 1
      const int n = (t + 1 < ntiles && it.j + 1 < it.nblk) ? 2 : 1;
      const int len = lens[it.b];

      KVQ_PT(s0)
      if (sw == 0) { KVQ_TR(19, t) if (n > 1) KVQ_TR(19, t + 1) }
      float sc[8], vs_t[2], vz_t[2];
      uint32_t pexp = 0u;
      float vals[kNV];
#pragma unroll
      for (int k = 0; k < kNV; ++k) vals[k] = 0.f;
      // Both tiles' scores are normally complete well before the step: wait
      // for both, then load them together so the two tiles' work interleaves
      // (a lone tile is loaded twice and its copy masked out).
      const int t1 = n > 1 ? t + 1 : t;
      const int st0 = t % C::kStages, st1 = t1 % C::kStages, q0 = t % C::kSlots, q1 = t1 % C::kSlots;
      if (!warp_wait4<true>(&sh.s_full[q0], (uint32_t)(t / C::kSlots) & 1u, &sh.s_full[q1], (uint32_t)(t1 / C::kSlots) & 1u,
                      &sh.stg_full[st0], (uint32_t)(t / C::kStages) & 1u, &sh.stg_full[st1],
                      (uint32_t)(t1 / C::kStages) & 1u, abort_flag, limit)) {
        ok = false;
        break;
      }
      if (sw == 0) { KVQ_TR(18, t) if (n > 1) KVQ_TR(18, t + 1) }
      tc_fence_after();
      uint32_t acc[2][12];
      tmem_ld_parts(tmem + lane_off + C::kColS + 16 * q0, acc[0]);
      tmem_ld_parts(tmem + lane_off + C::kColS + 16 * q1, acc[1]);
      float ks_t[2], kz_t[2], fs_t[2] = {1.f, 1.f};
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint16_t* szp = reinterpret_cast<const uint16_t*>(stages + (size_t)(u ? st1 : st0) * C::kStageBytes +
                                                                2 * C::kBlockBytes);
        ks_t[u] = h2f(szp[i]);
        kz_t[u] = h2f(szp[kBlockTokens + i]);
        vs_t[u] = h2f(szp[2 * kBlockTokens + i]);
        vz_t[u] = h2f(szp[3 * kBlockTokens + i]);
        // channel-wise K: undo this group's Q' prescale (the converters' factor)
        if (KCW) fs_t[u] = pow2_group_inv(f16_exp_field(max_f16_bits_128(szp)));
      }
      if (n < 2) { kz_t[1] = 0.f; vs_t[1] = 0.f; vz_t[1] = 0.f; }
      // what does not depend on the scores runs while their loads are in flight:
      // token-wise V: largest V scale of the pair (positive: ordered as integers);
      // channel-wise K: the offsets q . z_g, reduced over this warp's channels
      if (!VCW) vals[kVM] = __uint_as_float(__reduce_max_sync(FULL, __float_as_uint(fmaxf(vs_t[0], vs_t[1]))));
      float cgp = 0.f;
      if (KCW) {
        float za[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) { za[k] = qi[k] * kz_t[0]; za[4 + k] = qi[k] * kz_t[1]; }
        cgp = warp_sum8_transposed(za);
      }
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.s_empty[q0]);
        mbar_arrive(&sh.stg_empty[st0]);
        if (n > 1) { mbar_arrive(&sh.s_empty[q1]); mbar_arrive(&sh.stg_empty[st1]); }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const bool valid = u < n && i < len - (it.j + u) * kBlockTokens;
        const float2 ks2 = f2s(ks_t[u]), kz2 = f2s(kz_t[u]), fs2 = f2s(fs_t[u]);
#pragma unroll
        for (int k = 0; k < 4; k += 2) {  // heads k, k + 1
          float2 a = add2(f2u(acc[u][k], acc[u][k + 1]), f2u(acc[u][4 + k], acc[u][5 + k]));
          a = add2(a, f2u(acc[u][8 + k], acc[u][9 + k]));
          // channel-wise K adds q . z_g once reduced over channels
          const float2 addk = make_float2(add[k], add[k + 1]);
          const float2 v = KCW ? mul2(a, mul2(addk, fs2))
                               : fma2(mul2(a, make_float2(mult[k], mult[k + 1])), ks2, mul2(kz2, addk));
          sc[4 * u + k] = valid ? v.x : -INFINITY;
          sc[4 * u + k + 1] = valid ? v.y : -INFINITY;
          if (KCW) {  // the tile's offset q . z_g is still to come: per-tile maxima
            vals[kTM + 4 * u + k] = warp_max_redux(sc[4 * u + k]);
            vals[kTM + 4 * u + k + 1] = warp_max_redux(sc[4 * u + k + 1]);
          }
        }
      }
      if (!KCW) {  // one maximum per head over both tiles
#pragma unroll
        for (int k = 0; k < 4; ++k) vals[kTM + k] = warp_max_redux(fmaxf(sc[k], sc[4 + k]));
      }
      if (VCW) {
#pragma unroll
        for (int k = 0; k < 8; ++k) vals[kWS + k] = ws_prev[k];
      }
      KVQ_PA(16, s0)
      KVQ_PT(s2)
      float res[kNV];
      constexpr uint32_t kUsed = (KCW ? 0xffffu : 0xfu) | (VCW ? (0xffu << kWS) : (1u << kVM));
      // Channel-wise K with token-wise V: the pair's P' buffers are awaited
      // with the round's barrier (one barrier round trip less; measured +1%
      // there, -1% for the other scheme pairs, which wait after the update)
      // (with lean commits the P' slot of tile t is free at the previous
      // phase of its O slot: PV(t - kSlots) has completed; on a fresh barrier
      // that phase reads as complete)
      constexpr bool kPWaitInRound = KCW && !VCW;
      const uint32_t pe0 = ((uint32_t)(t / C::kSlots) & 1u) ^ 1u, pe1 = ((uint32_t)(t1 / C::kSlots) & 1u) ^ 1u;
      uint64_t* const pb0 = kLeanCommits ? &sh.o_full[q0] : &sh.p_empty[q0];
      uint64_t* const pb1 = kLeanCommits ? &sh.o_full[q1] : &sh.p_empty[q1];
      if (!(kPWaitInRound ? round(vals, res, kUsed, KCW, cgp, pb0, pe0, pb1, pe1)
                          : round(vals, res, kUsed, KCW, cgp))) {
        ok = false;
        break;
      }
      KVQ_PA(18, s2)
      if (sw == 0) { KVQ_TR(20, t) if (n > 1) KVQ_TR(20, t + 1) }
      KVQ_PT(s3)
      // one running-max update for the pair, and each head's P' prescale
      // exponent from the pair's own largest p (2^(mt - mn)) times the largest
      // V scale: far from the running max the p values would otherwise sit at
      // the bottom of the E4M3 range
      float pr[8], alpha[4];
      const int e_v = VCW ? 0 : (int)((__float_as_uint(res[kVM]) >> 23) & 0xffu) - 127;
#pragma unroll
      for (int k = 0; k < 4; k += 2) {  // heads k, k + 1
        const float2 cg0 = KCW ? mul2(make_float2(res[kCG + k], res[kCG + k + 1]), f2s(p.sm_scale_log2)) : f2s(0.f);
        const float2 cg1 =
            KCW ? mul2(make_float2(res[kCG + 4 + k], res[kCG + 5 + k]), f2s(p.sm_scale_log2)) : f2s(0.f);
        float2 mn;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float c0 = h ? cg0.y : cg0.x, c1 = h ? cg1.y : cg1.x;
          const float mt = KCW ? fmaxf(res[kTM + k + h] + c0, res[kTM + 4 + k + h] + c1) : res[kTM + k + h];
          const float mnh = fmaxf(m[k + h], mt);
          pexp |= ((uint32_t)p_exponent(mt - mnh, e_v) & 0xffu) << (8 * (k + h));
          alpha[k + h] = ex2(m[k + h] - mnh);
          m[k + h] = mnh;
          if (h) mn.y = mnh; else mn.x = mnh;
        }
        const float2 nmn = make_float2(-mn.x, -mn.y);
        const float2 x0 = KCW ? add2(add2(make_float2(sc[k], sc[k + 1]), cg0), nmn) : add2(make_float2(sc[k], sc[k + 1]), nmn);
        const float2 x1 =
            KCW ? add2(add2(make_float2(sc[4 + k], sc[5 + k]), cg1), nmn) : add2(make_float2(sc[4 + k], sc[5 + k]), nmn);
        pr[k] = ex2(x0.x);
        pr[k + 1] = ex2(x0.y);
        pr[4 + k] = ex2(x1.x);
        pr[5 + k] = ex2(x1.y);
        const float2 p0 = make_float2(pr[k], pr[k + 1]), p1 = make_float2(pr[4 + k], pr[5 + k]);
        const float2 al = make_float2(alpha[k], alpha[k + 1]);
        const float2 l2 = fma2(make_float2(lp[k], lp[k + 1]), al, add2(p0, p1));
        lp[k] = l2.x;
        lp[k + 1] = l2.y;
        if (!VCW) {
          const float2 z2 = fma2(make_float2(zp[k], zp[k + 1]), al, fma2(p0, f2s(vz_t[0]), mul2(p1, f2s(vz_t[1]))));
          zp[k] = z2.x;
          zp[k + 1] = z2.y;
        }
      }
      // P' operands (lane i = token i): token-wise V folds s into P; both
      // buffers are awaited first so the two rows are built together
      if (!kPWaitInRound && !warp_wait2<true>(pb0, pe0, pb1, pe1, abort_flag, limit)) {
        ok = false;
        break;
      }
      if (sw == 0) { KVQ_TR(23, t) if (n > 1) KVQ_TR(23, t + 1) }
      {
        float psc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) psc[k] = p_scale(pexp, k);
        uint4 bytes[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float2 f = f2s((VCW ? 1.0f : vs_t[u]) * odd_quarter<BITS, false, C::kE2V>(i));
          const float2 lo = mul2(make_float2(pr[4 * u], pr[4 * u + 1]), mul2(f, make_float2(psc[0], psc[1])));
          const float2 hi = mul2(make_float2(pr[4 * u + 2], pr[4 * u + 3]), mul2(f, make_float2(psc[2], psc[3])));
          const float4 pv = make_float4(lo.x, lo.y, hi.x, hi.y);
          bytes[u] = split3_e4m3_via_f16(pv);
        }
        *reinterpret_cast<uint4*>(pop + q0 * C::kBBytes + b_row_off(prow)) = bytes[0];
        if (n > 1) *reinterpret_cast<uint4*>(pop + q1 * C::kBBytes + b_row_off(prow)) = bytes[1];
      }
      fence_proxy_async_smem();  // both P' rows visible to the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.p_full[q0]);
        if (n > 1) mbar_arrive(&sh.p_full[q1]);
      }
      { KVQ_TR(8 + sw, t) if (n > 1) KVQ_TR(8 + sw, t + 1) }
      KVQ_PA(19, s3)

      // epilogue of the previous step (its sums of p arrived in this round)
      KVQ_PT(s6)
      if (pend_n > 0) {
        float ts[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ts[k] = VCW ? res[kWS + k] : 0.f;
        if (!epilogue(ts)) { ok = false; break; }
      }
      KVQ_PA(22, s6)
      if (sw == 0) { KVQ_TR(22, t) if (n > 1) KVQ_TR(22, t + 1) }
      pend = t;
      pend_n = n;
#pragma unroll
      for (int k = 0; k < 4; ++k) a_prev[k] = alpha[k];
      pexp_prev = pexp;  // per head, both tiles of the pair
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        sv_prev[u] = vs_t[u];  // channel-wise V: lane i = channel i
        zv_prev[u] = vz_t[u];
        // channel-wise V: this group's per-warp sum(p), in exact fixed point
#pragma unroll
        for (int k = 0; k < 4; ++k)
          ws_prev[4 * u + k] = VCW ? (float)__reduce_add_sync(FULL, __float2uint_rn(pr[4 * u + k] * kFix)) * (1.0f / kFix)
                                   : 0.f;
      }
      for (int u = 0; u < n; ++u) it.next<true>(prefix, B, Hkv);
      t += n;
    }
    if (ok && pend_n > 0) ok = drain() && finalize(pb, ph, pfirst, pue <= g1, pus, pue);
    if (!ok && ntiles > 0) set_abort(abort_flag, p.dev_status);
    finish_cta();
  }
}

template <int BITS, bool KCW, bool VCW, bool GQ4, bool E2V = false>
cudaError_t launch_decode_instance(const DecodeParams& p, cudaStream_t stream) {
  constexpr size_t smem = decode_smem_layout_bytes<BITS, E2V>();
  static_assert(smem <= 113 * 1024, "two CTAs per SM");
  auto kern = decode_kernel<BITS, KCW, VCW, GQ4, E2V>;
  // The register split inside the kernel assumes exactly kRegsLaunch
  // registers per thread at launch; with fewer, the softmax warpgroup's
  // increase could never be granted.  Refuse to launch such a build.
  static const bool regs_ok = [&] {
    cudaFuncAttributes a{};
    return cudaFuncGetAttributes(&a, kern) == cudaSuccess && a.numRegs == kRegsLaunch;
  }();
  if (!regs_ok) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.num_ctas, kDecodeThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
