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
// GB300 design (this library's; the pages' Blackwell pipeline is prior art):
//  * swap-AB MMAs: tokens (QK^T) or channels (PV) are the M = 128 rows, the
//    4 GQA query heads x operand splits are N = 16 columns;
//  * the KV operand (A) is written by converter warps straight into tensor
//    memory (tcgen05.st) and read by tcgen05.mma from there, so the hot
//    operand never passes through shared memory: packed codes are the only
//    KV bytes staged in shared memory (by cp.async.bulk);
//  * INT4 and INT2 codes both become E4M3 bytes (code * 2^-9): 3 integer ops
//    per 8 INT4 codes, 7 per 16 INT2 codes;
//  * Q' and P' are sums of three E4M3 parts (two BF16 parts in the BF16
//    correctness mode) stacked along N, so precision costs no extra MMA;
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

constexpr int kDecodeThreads = 320;  // 10 warps
constexpr int kMaxBatch = 1024;      // sequences per call (prefix table in shared memory)
constexpr uint32_t FULL = 0xffffffffu;

// Warp roles.
constexpr int kWarpConvert0 = 0;  // warps 0-3: KV codes -> tensor memory, Q' operand
constexpr int kWarpSoftmax0 = 4;  // warps 4-7: fold, online softmax, P' operand, epilogue
constexpr int kWarpLoad = 8;      // packed tiles HBM -> shared memory
constexpr int kWarpMma = 9;       // tcgen05.mma issue, tensor memory owner

template <int BITS, bool BF16>
struct DecodeCfg {
  static constexpr int kBlockBytes = kBlockTokens * kHeadDim * BITS / 8;  // 8192 / 4096
  static constexpr int kChunks = kHeadDim * BITS / 8 / 16;                // 16-byte chunks per row
  static constexpr int kStages = (BITS == 4) ? 4 : 6;
  static constexpr int kSzBytes = kBlockTokens * 2;                       // one fp16 [128] array
  static constexpr int kStageBytes = 2 * kBlockBytes + 4 * kSzBytes;
  static constexpr int kACols = BF16 ? 64 : 32;  // tensor-memory columns of one 128 x 128 A tile
  static constexpr int kNA = BF16 ? 1 : 2;       // A tile buffers per operand
  static constexpr int kSplits = BF16 ? 2 : 3;   // parts of Q' and P'
  static constexpr int kBBytes = BF16 ? 4096 : 2048;  // one B operand (128 K-rows x N=16)
  static constexpr int kKSteps = BF16 ? 8 : 4;
  static constexpr uint32_t kKStepBBytes = 512;
  static constexpr uint32_t kLbo = BF16 ? 256 : 128;  // K-direction core-matrix stride
  static constexpr uint32_t kSbo = 128;               // N-direction core-matrix stride
  static constexpr uint32_t kIdesc = BF16 ? make_idesc(1, 1, 0, 1, 128, 16) : make_idesc(0, 0, 0, 1, 128, 16);
  static constexpr int kColAK = 0;
  static constexpr int kColAV = kNA * kACols;
  static constexpr int kColS = 2 * kNA * kACols;
  static constexpr int kColO = kColS + 32;
  static constexpr int kTmemCols = 256;
  static constexpr float kCodeInv = BF16 ? 1.0f : 512.0f;  // code = operand value * kCodeInv
  static_assert(kColO + 32 <= kTmemCols, "tensor memory budget");
};

// Position of element e (channel of a K row, token of a V row) along the
// contraction dimension of the A operand, i.e. where the converter's masks
// put it.  The B operand rows (Q' channels, P' tokens) use the same order.
template <int BITS, bool BF16>
__device__ __forceinline__ int a_pos(int e) {
  if (!BF16) {
    if (BITS == 4) return (e & ~7) + ((e & 1) << 2) + ((e & 7) >> 1);
    return (e & ~15) + ((e & 3) << 2) + ((e & 15) >> 2);
  } else {
    if (BITS == 4) return (e & ~7) + ((e & 3) << 1) + ((e & 7) >> 2);
    return (e & ~15) + ((e & 7) << 1) + ((e & 15) >> 3);
  }
}

// Byte offset of B-operand row p (MN-major, no swizzle).
template <bool BF16>
__device__ __forceinline__ uint32_t b_row_off(int p) {
  return BF16 ? (uint32_t)((p >> 3) * 256 + (p & 7) * 16) : (uint32_t)(p * 16);
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

// Power of two 2^k with m * 2^k in [128, 256) (1 for m == 0 or non-normal).
__device__ __forceinline__ float pow2_prescale(float m) {
  int e = (int)((__float_as_uint(m) >> 23) & 0xffu);
  if (e == 0 || e == 0xff) return 1.0f;
  return __uint_as_float((uint32_t)(261 - e) << 23);  // 2^(7 - (e - 127))
}

// Converted code words of one packed 32-bit word.
template <int BITS, bool BF16>
struct Convert {
  static constexpr int kOut = BF16 ? (BITS == 4 ? 4 : 8) : (BITS == 4 ? 2 : 4);
  __device__ __forceinline__ static void run(uint32_t x, uint32_t* o) {
    if (!BF16) {
      if (BITS == 4) {  // codes e = 0,2,4,6 then 1,3,5,7 as E4M3 0x0q
        o[0] = x & 0x0F0F0F0Fu;
        o[1] = (x >> 4) & 0x0F0F0F0Fu;
      } else {  // word k holds codes e = k, k+4, k+8, k+12
#pragma unroll
        for (int k = 0; k < 4; ++k) o[k] = (x >> (2 * k)) & 0x03030303u;
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
template <int BITS, bool BF16>
struct alignas(16) DecodeBarriers {
  using C = DecodeCfg<BITS, BF16>;
  uint64_t stg_full[C::kStages], stg_empty[C::kStages];
  uint64_t ak_full[C::kNA], ak_empty[C::kNA], av_full[C::kNA], av_empty[C::kNA];
  uint64_t q_full[2], q_empty[2], sd_full[2], sd_empty[2];
  uint64_t s_full[2], s_empty[2], p_full[2], p_empty[2], o_full[2], o_empty[2];
  uint64_t cw_grp, sw_grp, drain;
  float side[2][8];         // per tile: score multiplier [4], score offset [4] (converter -> softmax)
  float cw_red[2][4][8];    // converter group reduction scratch [parity][warp][value]
  float sw_red[2][4][8];    // softmax group reduction scratch
  int flag[2];              // split-unit "last arriver" broadcast
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
};

template <int BITS, bool BF16>
constexpr size_t decode_smem_layout_bytes() {
  using C = DecodeCfg<BITS, BF16>;
  size_t b = (size_t)C::kStages * C::kStageBytes + 4 * (size_t)C::kBBytes + sizeof(DecodeBarriers<BITS, BF16>) +
             (2 * kMaxBatch + 1) * sizeof(int) + 1024;
  return b < 80 * 1024 ? 80 * 1024 : b;  // >= 80 KB keeps at most two CTAs per SM
}

// --------------------------------------------------------------- helpers
__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

// All lanes poll; the warp gives up together (after the time limit or when
// the CTA has been told to abort).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(FULL, ok)) return true;
    if ((it & 31u) == 31u) {
      int stop = 0;
      if (lane_id() == 0) {
        uint64_t now = globaltimer_ns();
        if (t0 == 0) t0 = now;
        stop = (*abort_flag != 0) || (now - t0 > limit_ns);
      }
      if (__shfl_sync(FULL, stop, 0)) return false;
    }
  }
}

__device__ __forceinline__ void set_abort(volatile int* abort_flag, uint32_t* dev_status) {
  *abort_flag = 1;
  report(dev_status, KVQ_DEV_TIMEOUT);
}

// A four-warp group barrier on an mbarrier (count 4), bounded.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, volatile int* abort_flag,
                                           uint64_t limit_ns) {
  __syncwarp();
  if (lane_id() == 0) mbar_arrive(bar);
  bool ok = warp_wait(bar, phase, abort_flag, limit_ns);
  phase ^= 1u;
  return ok;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ float warp_maxf(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

__device__ __forceinline__ float h2f(uint16_t bits) { return __half2float(__ushort_as_half(bits)); }

__device__ __forceinline__ float bf2f(uint16_t bits) { return __uint_as_float((uint32_t)bits << 16); }

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
  __device__ __forceinline__ void next(const int* prefix, int B, int Hkv) {
    if (++j < nblk) return;
    j = 0;
    if (++h < Hkv) return;
    h = 0;
    do { ++b; } while (b < B && prefix[b + 1] == prefix[b]);
    if (b < B) nblk = (prefix[b + 1] - prefix[b]) / Hkv;
  }
};

__device__ __forceinline__ int cta_of_tile(long long t, long long T, int C) {
  return (int)(((t + 1) * C - 1) / T);
}
__device__ __forceinline__ long long range_start(int c, long long T, int C) { return (long long)c * T / C; }

// ================================================================= kernel
template <int BITS, bool KCW, bool VCW, bool BF16>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_kernel(const DecodeParams p) {
  using C = DecodeCfg<BITS, BF16>;
  using Bars = DecodeBarriers<BITS, BF16>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* stages = smem_raw;
  unsigned char* qop = stages + (size_t)C::kStages * C::kStageBytes;  // [2][kBBytes]
  unsigned char* pop = qop + 2 * C::kBBytes;                          // [2][kBBytes]
  Bars& sh = *reinterpret_cast<Bars*>(pop + 2 * C::kBBytes);
  int* prefix = reinterpret_cast<int*>(&sh + 1);  // [B + 1] tile offsets
  int* lens = prefix + (kMaxBatch + 1);           // [B] validated sequence lengths

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.batch, Hkv = p.num_kv_heads;
  const int cta = blockIdx.x;
  volatile int* abort_flag = &sh.abort_flag;
  const uint64_t limit = p.wait_limit_ns;

  // ------------------------------------------------------------ set-up
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) { mbar_init(&sh.stg_full[s], 1); mbar_init(&sh.stg_empty[s], 8); }
    for (int a = 0; a < C::kNA; ++a) {
      mbar_init(&sh.ak_full[a], 4); mbar_init(&sh.ak_empty[a], 1);
      mbar_init(&sh.av_full[a], 4); mbar_init(&sh.av_empty[a], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.q_full[s], 4); mbar_init(&sh.q_empty[s], 1);
      mbar_init(&sh.sd_full[s], 4); mbar_init(&sh.sd_empty[s], 4);
      mbar_init(&sh.s_full[s], 1); mbar_init(&sh.s_empty[s], 4);
      mbar_init(&sh.p_full[s], 4); mbar_init(&sh.p_empty[s], 1);
      mbar_init(&sh.o_full[s], 1); mbar_init(&sh.o_empty[s], 4);
    }
    mbar_init(&sh.cw_grp, 4); mbar_init(&sh.sw_grp, 4); mbar_init(&sh.drain, 1);
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
  if (BF16) {  // N columns 8..15 of the BF16 operands stay zero
    for (int i = tid; i < 4 * C::kBBytes / 16; i += kDecodeThreads)
      reinterpret_cast<uint4*>(qop)[i] = make_uint4(0u, 0u, 0u, 0u);
  }
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

  // ============================================================= loader
  if (warp == kWarpLoad) {
    if (lane == 0 && ntiles > 0) {
      const uint64_t policy = l2_policy_evict_first();
      int issued_parity[C::kStages];
      for (int s = 0; s < C::kStages; ++s) issued_parity[s] = -1;
      TileIter it;
      it.init(prefix, B, Hkv, (int)g0);
      for (int t = 0; t < ntiles; ++t, it.next(prefix, B, Hkv)) {
        const int s = t % C::kStages;
        const uint32_t ph = (uint32_t)(t / C::kStages) & 1u;
        if (!mbar_wait_bounded(&sh.stg_empty[s], ph ^ 1u, abort_flag, limit)) {
          set_abort(abort_flag, p.dev_status);
          break;
        }
        if ((p.flags & KVQ_FLAG_TEST_STALL) && cta == 0 && t == 1) continue;  // withhold one tile
        int page = p.page_table ? p.page_table[(size_t)it.b * p.max_blocks + it.j] : it.b * p.max_blocks + it.j;
        if (page < 0 || page >= p.num_pages) {
          report(p.dev_status, KVQ_DEV_BAD_PAGE);
          page = 0;
        }
        const size_t blk = (size_t)page * Hkv + it.h;
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
        issued_parity[s] = (int)ph;
      }
      // never leave a copy in flight: wait for every issued stage to land
      for (int s = 0; s < C::kStages; ++s)
        if (issued_parity[s] >= 0) mbar_wait_bounded(&sh.stg_full[s], (uint32_t)issued_parity[s], nullptr, limit);
    }
  }
  // ================================================================ MMA
  else if (warp == kWarpMma) {
    if (lane == 0 && ntiles > 0) {
      bool ok = true;
      auto issue_pv = [&](int t) -> bool {
        const int a = t % C::kNA, sl = t & 1;
        const uint32_t pa = (uint32_t)(t / C::kNA) & 1u, p2 = (uint32_t)(t >> 1) & 1u;
        if (!mbar_wait_bounded(&sh.av_full[a], pa, abort_flag, limit)) return false;
        if (!mbar_wait_bounded(&sh.p_full[sl], p2, abort_flag, limit)) return false;
        if (!mbar_wait_bounded(&sh.o_empty[sl], p2 ^ 1u, abort_flag, limit)) return false;
        tc_fence_after();
        const uint32_t b0 = smem_u32(pop + sl * C::kBBytes);
#pragma unroll
        for (int k = 0; k < C::kKSteps; ++k) {
          uint64_t bd = make_smem_desc(b0 + k * C::kKStepBBytes, C::kLbo, C::kSbo);
          uint32_t d = tmem + C::kColO + 16 * sl, av = tmem + C::kColAV + a * C::kACols + 8 * k;
          if (BF16) mma_f16_ts(d, av, bd, C::kIdesc, k > 0); else mma_f8f6f4_ts(d, av, bd, C::kIdesc, k > 0);
        }
        tc_commit(&sh.av_empty[a]);
        tc_commit(&sh.p_empty[sl]);
        tc_commit(&sh.o_full[sl]);
        return true;
      };
      for (int t = 0; t < ntiles && ok; ++t) {
        const int a = t % C::kNA, sl = t & 1;
        const uint32_t pa = (uint32_t)(t / C::kNA) & 1u, p2 = (uint32_t)(t >> 1) & 1u;
        ok = mbar_wait_bounded(&sh.ak_full[a], pa, abort_flag, limit) &&
             mbar_wait_bounded(&sh.q_full[sl], p2, abort_flag, limit) &&
             mbar_wait_bounded(&sh.s_empty[sl], p2 ^ 1u, abort_flag, limit);
        if (!ok) break;
        tc_fence_after();
        const uint32_t b0 = smem_u32(qop + sl * C::kBBytes);
#pragma unroll
        for (int k = 0; k < C::kKSteps; ++k) {
          uint64_t bd = make_smem_desc(b0 + k * C::kKStepBBytes, C::kLbo, C::kSbo);
          uint32_t d = tmem + C::kColS + 16 * sl, ak = tmem + C::kColAK + a * C::kACols + 8 * k;
          if (BF16) mma_f16_ts(d, ak, bd, C::kIdesc, k > 0); else mma_f8f6f4_ts(d, ak, bd, C::kIdesc, k > 0);
        }
        tc_commit(&sh.ak_empty[a]);
        tc_commit(&sh.q_empty[sl]);
        tc_commit(&sh.s_full[sl]);
        if (t > 0) ok = issue_pv(t - 1);
      }
      if (ok) ok = issue_pv(ntiles - 1);
      if (!ok) set_abort(abort_flag, p.dev_status);
      // drain: all issued MMAs complete before tensor memory is released
      tc_commit(&sh.drain);
      mbar_wait_bounded(&sh.drain, 0, nullptr, limit);
    }
  }
  // ========================================================== converters
  else if (warp < kWarpSoftmax0) {
    const int r = tid;  // tensor-memory lane = A row = Q' channel
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t grp_phase = 0;
    float qv[4] = {0.f, 0.f, 0.f, 0.f};  // q[b, 4h + i, r]
    uint4 qtok = make_uint4(0u, 0u, 0u, 0u);  // token-wise K: this channel's Q' row
    float tok_mult[4], tok_add[4];
    const int qrow = a_pos<BITS, BF16>(r);
    TileIter it;
    if (ntiles > 0) it.init(prefix, B, Hkv, (int)g0);
    for (int t = 0; t < ntiles; ++t, it.next(prefix, B, Hkv)) {
      const int s = t % C::kStages, a = t % C::kNA, sl = t & 1;
      const uint32_t ps = (uint32_t)(t / C::kStages) & 1u, pa = (uint32_t)(t / C::kNA) & 1u,
                     p2 = (uint32_t)(t >> 1) & 1u;
      const bool seg_first = (t == 0) || it.j == 0;
      if (!warp_wait(&sh.stg_full[s], ps, abort_flag, limit)) { set_abort(abort_flag, p.dev_status); break; }
      const unsigned char* st = stages + (size_t)s * C::kStageBytes;
      const uint16_t* ks = reinterpret_cast<const uint16_t*>(st + 2 * C::kBlockBytes);
      const uint16_t* kz = ks + kBlockTokens;

      // ---- K codes -> A_K[a] (row r = token r)
      if (!warp_wait(&sh.ak_empty[a], pa ^ 1u, abort_flag, limit)) { set_abort(abort_flag, p.dev_status); break; }
      {
        uint32_t o[C::kACols];
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          uint4 v = *reinterpret_cast<const uint4*>(st + ((size_t)c * kBlockTokens + r) * 16);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) Convert<BITS, BF16>::run(w[i], &o[(4 * c + i) * Convert<BITS, BF16>::kOut]);
        }
        const uint32_t col = tmem + lane_off + C::kColAK + a * C::kACols;
#pragma unroll
        for (int c0 = 0; c0 < C::kACols; c0 += 32)
          tmem_st_32x32b_x32(col + c0, *reinterpret_cast<const uint32_t(*)[32]>(&o[c0]));
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.ak_full[a]);
      }

      // ---- Q' operand and score constants for this tile
      if (seg_first) {
        const uint16_t* qsrc = p.q + ((size_t)it.b * p.num_q_heads + (size_t)it.h * kGroupQ) * kHeadDim + r;
#pragma unroll
        for (int i = 0; i < 4; ++i) qv[i] = bf2f(qsrc[i * kHeadDim]);
        if (!KCW) {  // token-wise K: Q' = q (prescaled), constant over the segment
          float m[4], sm[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) { m[i] = warp_maxf(fabsf(qv[i])); sm[i] = warp_sum(qv[i]); }
          float* red = sh.cw_red[grp_phase][warp];
          if (lane == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i) { red[i] = m[i]; red[4 + i] = sm[i]; }
          }
          const uint32_t use = grp_phase;
          if (!group_sync(&sh.cw_grp, grp_phase, abort_flag, limit)) { set_abort(abort_flag, p.dev_status); break; }
          float qs[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float mx = 0.f, su = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) { mx = fmaxf(mx, sh.cw_red[use][w][i]); su += sh.cw_red[use][w][4 + i]; }
            qs[i] = BF16 ? 1.0f : pow2_prescale(mx);
            tok_mult[i] = C::kCodeInv / qs[i] * p.sm_scale_log2;
            tok_add[i] = su * p.sm_scale_log2;
          }
          float4 v = make_float4(qv[0] * qs[0], qv[1] * qs[1], qv[2] * qs[2], qv[3] * qs[3]);
          qtok = BF16 ? split2_bf16(v) : split3_e4m3(v);
        }
      }
      if (!warp_wait(&sh.q_empty[sl], p2 ^ 1u, abort_flag, limit) ||
          !warp_wait(&sh.sd_empty[sl], p2 ^ 1u, abort_flag, limit)) {
        set_abort(abort_flag, p.dev_status);
        break;
      }
      uint4 qrow_bytes;
      float mult[4], add[4];
      if (!KCW) {
        qrow_bytes = qtok;
#pragma unroll
        for (int i = 0; i < 4; ++i) { mult[i] = tok_mult[i]; add[i] = tok_add[i]; }
      } else {  // channel-wise K: Q' = q * s_g (operand fold), offset q . z_g
        const float sd = h2f(ks[r]), zd = h2f(kz[r]);
        float qf[4], m[4], sm[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          qf[i] = qv[i] * sd;
          m[i] = warp_maxf(fabsf(qf[i]));
          sm[i] = warp_sum(qv[i] * zd);
        }
        float* red = sh.cw_red[grp_phase][warp];
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) { red[i] = m[i]; red[4 + i] = sm[i]; }
        }
        const uint32_t use = grp_phase;
        if (!group_sync(&sh.cw_grp, grp_phase, abort_flag, limit)) { set_abort(abort_flag, p.dev_status); break; }
        float qs[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float mx = 0.f, su = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) { mx = fmaxf(mx, sh.cw_red[use][w][i]); su += sh.cw_red[use][w][4 + i]; }
          qs[i] = BF16 ? 1.0f : pow2_prescale(mx);
          mult[i] = C::kCodeInv / qs[i] * p.sm_scale_log2;
          add[i] = su * p.sm_scale_log2;
        }
        float4 v = make_float4(qf[0] * qs[0], qf[1] * qs[1], qf[2] * qs[2], qf[3] * qs[3]);
        qrow_bytes = BF16 ? split2_bf16(v) : split3_e4m3(v);
      }
      *reinterpret_cast<uint4*>(qop + sl * C::kBBytes + b_row_off<BF16>(qrow)) = qrow_bytes;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.q_full[sl]);
      if (tid == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) { sh.side[sl][i] = mult[i]; sh.side[sl][4 + i] = add[i]; }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.sd_full[sl]);

      // ---- V codes -> A_V[a] (row r = channel r)
      if (!warp_wait(&sh.av_empty[a], pa ^ 1u, abort_flag, limit)) { set_abort(abort_flag, p.dev_status); break; }
      {
        uint32_t o[C::kACols];
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c) {
          uint4 v = *reinterpret_cast<const uint4*>(st + C::kBlockBytes + ((size_t)c * kBlockTokens + r) * 16);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) Convert<BITS, BF16>::run(w[i], &o[(4 * c + i) * Convert<BITS, BF16>::kOut]);
        }
        const uint32_t col = tmem + lane_off + C::kColAV + a * C::kACols;
#pragma unroll
        for (int c0 = 0; c0 < C::kACols; c0 += 32)
          tmem_st_32x32b_x32(col + c0, *reinterpret_cast<const uint32_t(*)[32]>(&o[c0]));
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) { mbar_arrive(&sh.av_full[a]); mbar_arrive(&sh.stg_empty[s]); }
      }
    }
  }
  // ============================================================= softmax
  else {
    const int i = tid - kWarpSoftmax0 * 32;  // tensor-memory lane: token (scores) / channel (output)
    const int sw = warp - kWarpSoftmax0;
    const uint32_t lane_off = (uint32_t)(sw * 32) << 16;
    const int prow = a_pos<BITS, BF16>(i);
    uint32_t grp_phase = 0;
    const float kLn2 = 0.69314718055994530942f;

    // empty sequences: out = 0, lse = -inf
    for (int b = cta; b < B; b += (int)gridDim.x) {
      if (lens[b] != 0) continue;
      for (int hq = 0; hq < p.num_q_heads; ++hq) {
        p.out[((size_t)b * p.num_q_heads + hq) * kHeadDim + i] = 0.0f;
        if (i == 0) p.lse[(size_t)b * p.num_q_heads + hq] = -INFINITY;
      }
    }

    float m[4], lp[4], zp[4], O[4];          // running max (log2), partial sum, partial sum(p z), output
    float a_prev[4], ts_prev[4], pinv_prev = 0.f, sv_prev = 0.f, zv_prev = 0.f;  // deferred epilogue inputs
    auto reset = [&]() {
#pragma unroll
      for (int k = 0; k < 4; ++k) { m[k] = -INFINITY; lp[k] = 0.f; zp[k] = 0.f; O[k] = 0.f; }
    };
    reset();

    // PV epilogue of tile t: O = O * alpha + folded partial product
    auto epilogue = [&](int t) -> bool {
      const int sl = t & 1;
      const uint32_t p2 = (uint32_t)(t >> 1) & 1u;
      if (!warp_wait(&sh.o_full[sl], p2, abort_flag, limit)) return false;
      tc_fence_after();
      uint32_t acc[16];
      tmem_ld_32x32b_x16(tmem + lane_off + C::kColO + 16 * sl, acc);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.o_empty[sl]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float o = __uint_as_float(acc[k]) + __uint_as_float(acc[4 + k]);
        if (!BF16) o += __uint_as_float(acc[8 + k]);
        o *= pinv_prev;
        if (VCW) O[k] = fmaf(O[k], a_prev[k], fmaf(sv_prev, o, zv_prev * ts_prev[k]));
        else O[k] = fmaf(O[k], a_prev[k], o);
      }
      return true;
    };

    // finish a (sequence, kv head) segment: normalise, store or merge
    auto finalize = [&](int b, int h, bool first_global, bool last_global, long long ustart, long long uend) -> bool {
      float lsum[4], zsum[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) { lsum[k] = warp_sum(lp[k]); zsum[k] = VCW ? 0.f : warp_sum(zp[k]); }
      float* red = sh.sw_red[grp_phase][sw];
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) { red[k] = lsum[k]; red[4 + k] = zsum[k]; }
      }
      const uint32_t use = grp_phase;
      if (!group_sync(&sh.sw_grp, grp_phase, abort_flag, limit)) return false;
      float res[4], lse2[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float l = 0.f, z = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) { l += sh.sw_red[use][w][k]; z += sh.sw_red[use][w][4 + k]; }
        res[k] = (O[k] + z) / l;
        lse2[k] = m[k] + __log2f(l);
      }
      const size_t row0 = (size_t)b * p.num_q_heads + (size_t)h * kGroupQ;
      if (first_global && last_global) {  // whole (sequence, head) in this CTA
#pragma unroll
        for (int k = 0; k < 4; ++k) p.out[(row0 + k) * kHeadDim + i] = res[k];
        if (i < 4) p.lse[row0 + i] = lse2[i] * kLn2;
        return true;
      }
      // split: publish this part, the last part to arrive merges all parts
      const int c_first = cta_of_tile(ustart, T, Cn), c_last = cta_of_tile(uend - 1, T, Cn);
      const int slot = (ustart <= g0) ? 0 : 1;
      float* po = p.part_o + ((size_t)cta * 2 + slot) * kGroupQ * kHeadDim;
#pragma unroll
      for (int k = 0; k < 4; ++k) po[k * kHeadDim + i] = res[k];
      if (i < 4) p.part_lse[((size_t)cta * 2 + slot) * kGroupQ + i] = lse2[i] * kLn2;
      __threadfence();
      if (!group_sync(&sh.sw_grp, grp_phase, abort_flag, limit)) return false;
      const int u = b * Hkv + h;
      if (i == 0) {
        int old = atomicAdd(&p.counters[u], 1);
        sh.flag[use] = (old == c_last - c_first) ? 1 : 0;
      }
      const uint32_t use2 = grp_phase;
      if (!group_sync(&sh.sw_grp, grp_phase, abort_flag, limit)) return false;
      if (!sh.flag[use]) return true;
      (void)use2;
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
      for (int k = 0; k < 4; ++k) p.out[(row0 + k) * kHeadDim + i] = acc[k] / den[k];
      if (i < 4) p.lse[row0 + i] = mx[i] + __logf(den[i]);
      if (i == 0) p.counters[u] = 0;
      return true;
    };

    TileIter it;
    if (ntiles > 0) it.init(prefix, B, Hkv, (int)g0);
    int pend = -1;
    int pb = 0, ph = 0;
    bool pfirst = false;
    long long pus = 0, pue = 0;
    bool ok = true;
    for (int t = 0; t < ntiles && ok; ++t, it.next(prefix, B, Hkv)) {
      const int s = t % C::kStages, sl = t & 1;
      const uint32_t ps = (uint32_t)(t / C::kStages) & 1u, p2 = (uint32_t)(t >> 1) & 1u;
      const long long g = g0 + t;
      const long long ustart = g - it.j, uend = ustart + it.nblk;
      const bool seg_first = (t == 0) || it.j == 0;
      if (seg_first && pend >= 0) {  // close the previous segment
        ok = epilogue(pend) && finalize(pb, ph, pfirst, pue <= g1, pus, pue);
        if (!ok) break;
        reset();
        pend = -1;
      }
      if (seg_first) { pb = it.b; ph = it.h; pfirst = ustart >= g0; pus = ustart; pue = uend; }
      const int nvalid = min(kBlockTokens, lens[it.b] - it.j * kBlockTokens);

      // ---- scores of this tile (lane i = token i)
      if (!warp_wait(&sh.s_full[sl], p2, abort_flag, limit) || !warp_wait(&sh.stg_full[s], ps, abort_flag, limit) ||
          !warp_wait(&sh.sd_full[sl], p2, abort_flag, limit)) { ok = false; break; }
      tc_fence_after();
      uint32_t acc[16];
      tmem_ld_32x32b_x16(tmem + lane_off + C::kColS + 16 * sl, acc);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.s_empty[sl]);
      float mult[4], add[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) { mult[k] = sh.side[sl][k]; add[k] = sh.side[sl][4 + k]; }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.sd_empty[sl]);
      const unsigned char* st = stages + (size_t)s * C::kStageBytes;
      const uint16_t* szp = reinterpret_cast<const uint16_t*>(st + 2 * C::kBlockBytes);
      const float ks_i = h2f(szp[i]), kz_i = h2f(szp[kBlockTokens + i]);
      const float vs_i = h2f(szp[2 * kBlockTokens + i]), vz_i = h2f(szp[3 * kBlockTokens + i]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.stg_empty[s]);

      const bool valid = i < nvalid;
      float sc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float a = __uint_as_float(acc[k]) + __uint_as_float(acc[4 + k]);
        if (!BF16) a += __uint_as_float(acc[8 + k]);
        float v = KCW ? fmaf(a, mult[k], add[k]) : fmaf(a * mult[k], ks_i, kz_i * add[k]);
        sc[k] = valid ? v : -INFINITY;
      }
      // tile maxima (4 heads) and, for token-wise V, the largest scale
      float* red = sh.sw_red[grp_phase][sw];
      {
        float tm[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) tm[k] = warp_maxf(sc[k]);
        float smax = VCW ? 0.f : warp_maxf(valid ? vs_i : 0.f);
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) red[k] = tm[k];
          red[4] = smax;
        }
      }
      uint32_t use = grp_phase;
      if (!group_sync(&sh.sw_grp, grp_phase, abort_flag, limit)) { ok = false; break; }
      float alpha[4], pr[4], smax = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float tmx = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) tmx = fmaxf(tmx, sh.sw_red[use][w][k]);
        const float mn = fmaxf(m[k], tmx);
        alpha[k] = exp2f(m[k] - mn);
        m[k] = mn;
        pr[k] = exp2f(sc[k] - mn);
        lp[k] = fmaf(lp[k], alpha[k], pr[k]);
        if (!VCW) zp[k] = fmaf(zp[k], alpha[k], pr[k] * vz_i);
      }
      if (!VCW) {
#pragma unroll
        for (int w = 0; w < 4; ++w) smax = fmaxf(smax, sh.sw_red[use][w][4]);
      }
      // P' operand (lane i = token i): token-wise V folds s into P
      const float pscale = VCW ? 256.0f : (BF16 ? 1.0f : pow2_prescale(smax));
      const float pmul = VCW ? pscale : vs_i * pscale;
      float4 pv = make_float4(pr[0] * pmul, pr[1] * pmul, pr[2] * pmul, pr[3] * pmul);
      uint4 prow_bytes = BF16 ? split2_bf16(pv) : split3_e4m3(pv);
      if (!warp_wait(&sh.p_empty[sl], p2 ^ 1u, abort_flag, limit)) { ok = false; break; }
      *reinterpret_cast<uint4*>(pop + sl * C::kBBytes + b_row_off<BF16>(prow)) = prow_bytes;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.p_full[sl]);

      // channel-wise V needs this group's sum(p) for its offset term
      float tsum[4] = {0.f, 0.f, 0.f, 0.f};
      if (VCW) {
        float ws[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) ws[k] = warp_sum(pr[k]);
        red = sh.sw_red[grp_phase][sw];
        if (lane == 0) {
#pragma unroll
          for (int k = 0; k < 4; ++k) red[k] = ws[k];
        }
        use = grp_phase;
        if (!group_sync(&sh.sw_grp, grp_phase, abort_flag, limit)) { ok = false; break; }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
#pragma unroll
          for (int w = 0; w < 4; ++w) tsum[k] += sh.sw_red[use][w][k];
        }
      }

      // epilogue of the previous tile of this segment
      if (pend >= 0) { ok = epilogue(pend); if (!ok) break; }
      pend = t;
#pragma unroll
      for (int k = 0; k < 4; ++k) { a_prev[k] = alpha[k]; ts_prev[k] = tsum[k]; }
      pinv_prev = C::kCodeInv / pscale;
      sv_prev = vs_i;  // channel-wise V: lane i = channel i
      zv_prev = vz_i;
    }
    if (ok && pend >= 0) ok = epilogue(pend) && finalize(pb, ph, pfirst, pue <= g1, pus, pue);
    if (!ok && ntiles > 0) set_abort(abort_flag, p.dev_status);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int BITS, bool KCW, bool VCW, bool BF16>
cudaError_t launch_decode_instance(const DecodeParams& p, cudaStream_t stream) {
  constexpr size_t smem = decode_smem_layout_bytes<BITS, BF16>();
  auto kern = decode_kernel<BITS, KCW, VCW, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.num_ctas, kDecodeThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
