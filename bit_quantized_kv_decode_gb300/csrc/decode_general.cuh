// Decode attention for every cache geometry (head dims 64, 128 and 256,
// groups of 32, 64 or 128 elements) and both operand modes; the host sends
// it every call of real size (the specialised kernel of decode.cuh keeps
// small calls and the E2M1 V placement).  One warpgroup per CTA runs every
// step of a 128-token block in turn
// -- bulk copies into a ring of stages, codes to E4M3 operands in tensor
// memory, Q' and P' operands in shared memory, tcgen05 MMAs with the
// accumulators in tensor memory, the affine folds and an online softmax --
// over a contiguous range of one (sequence, unit)'s blocks; the ranges'
// partial results are merged by log-sum-exp afterwards.  Tensor memory is
// kept small (operand and accumulator regions reused within a block) so that
// several CTAs share an SM and hide one another's latencies.
//
// Folds per quantization group (rag-lover.com summary of arXiv 2611.09722,
// "限界と未検証の範囲": accumulator folds are applied one group at a time;
// "解説": which side each scheme folds on):
//   * token-wise K (groups of G channels): the K-steps of each channel group
//     accumulate into their own 16-column score block, and the softmax adds
//     s_(l,g) * partial_g + z_(l,g) * sum_(c in g) q_c;
//   * channel-wise K (groups of G tokens): Q'_g = q * s_g for each token
//     group g, stacked along N; token l reads the block of its group, plus
//     q . z_g;
//   * token-wise V: P'_g = p * s_(l,g) for each channel group, stacked along
//     N; channel c reads the block of its group, plus sum_l p_l z_(l,g);
//   * channel-wise V: the K-steps of each token group accumulate into their
//     own output block: O += s_g * partial_g + z_g * sum_(l in g) p_l.
#pragma once
#include "decode.cuh"
#include "decode_general.h"

namespace kvq {
namespace gen {

constexpr int kThreads = 128;

// Byte offset of row p, 16-column block nb of a B operand with nb16 blocks
// (MN-major, no swizzle: core matrices of 8 rows x 16 bytes, N-direction
// stride 128).  An E4M3 block is one core matrix wide (K-direction stride
// nb16 * 128); a BF16 block two (K-direction stride nb16 * 256), of which
// the parts use the first.
template <bool BF16>
__device__ __forceinline__ uint32_t b_off(int p, int nb, int nb16) {
  constexpr int kCm = BF16 ? 256 : 128;
  return (uint32_t)((p >> 3) * (nb16 * kCm) + nb * kCm + (p & 7) * 16);
}

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// The used columns of a 16-column block (4 heads x 3 E4M3 parts, or x 2
// BF16 parts).
template <bool BF16>
__device__ __forceinline__ void ld_block(uint32_t taddr, uint32_t (&v)[12]) {
  tmem_ld_32x32b_x8(taddr, v);
  if (!BF16) tmem_ld_32x32b_x4(taddr + 8, v + 8);
}
// Sum of the parts of head h.
template <bool BF16>
__device__ __forceinline__ float parts(const uint32_t (&v)[12], int h) {
  return BF16 ? __uint_as_float(v[h]) + __uint_as_float(v[4 + h])
              : (__uint_as_float(v[h]) + __uint_as_float(v[4 + h])) + __uint_as_float(v[8 + h]);
}

// Warp reduction of N values per lane at once (sum or max), halving the
// values held at each exchange: afterwards lane l holds the warp's result for
// value l >> (5 - log2 N).  N - 1 + (5 - log2 N) shuffles instead of 5 N.
template <int N, bool MAX>
__device__ __forceinline__ float warp_reduce_t(float (&v)[N]) {
  static_assert(N == 1 || N == 2 || N == 4 || N == 8 || N == 16 || N == 32, "N");
  const int lane = threadIdx.x & 31;
  int o = 16;
#pragma unroll
  for (int n = N; n > 1; n >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      const float got = __shfl_xor_sync(FULL, send, o);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  float r = v[0];
#pragma unroll
  for (; o > 0; o >>= 1) {
    const float got = __shfl_xor_sync(FULL, r, o);
    r = MAX ? fmaxf(r, got) : r + got;
  }
  return r;
}
// ... and the per-warp results into buf[N][4] (value-major: one 16-byte row
// of the 4 warps' results per value, read back with one vector load).
template <int N, bool MAX>
__device__ __forceinline__ void warp_reduce_store(float (&v)[N], float* buf) {
  constexpr int kLog = N == 1 ? 0 : N == 2 ? 1 : N == 4 ? 2 : N == 8 ? 3 : N == 16 ? 4 : 5;
  const float r = warp_reduce_t<N, MAX>(v);
  const int lane = threadIdx.x & 31;
  if ((lane & ((32 >> kLog) - 1)) == 0) buf[(lane >> (5 - kLog)) * 4 + (threadIdx.x >> 5)] = r;
  __syncwarp();
}
// The per-warp maxima of N values into buf[N][4]: one redux.sync.max.f32
// per value (independent instructions whose latencies overlap, where the
// butterfly above chains log2(32) exchanges), lane i storing value i.
template <int N>
__device__ __forceinline__ void warp_max_store(const float (&v)[N], float* buf) {
  static_assert(N <= 32, "N");
  const int lane = threadIdx.x & 31;
  float mine = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float r = warp_max_redux(v[i]);
    mine = lane == i ? r : mine;
  }
  if (lane < N) buf[lane * 4 + (threadIdx.x >> 5)] = mine;
  __syncwarp();
}
// Programmatic dependent launch (sm_90+): a kernel launched with the
// programmatic-serialization attribute may start while the kernel before it
// in the stream still runs; grid_dep_wait() blocks until that kernel has
// completed and its memory is visible (a no-op without the attribute), and
// grid_dep_launch() lets the next such kernel start launching.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Largest of D non-negative fp16 values in shared memory (bits; they order as
// integers), computed by each warp on its own: no cross-warp exchange.
template <int D>
__device__ __forceinline__ uint32_t max_f16_bits(const uint16_t* v) {
  const int lane = threadIdx.x & 31;
  uint32_t m;
  if (D == 64) {
    m = reinterpret_cast<const uint32_t*>(v)[lane];
  } else if (D == 128) {
    const uint2 w = reinterpret_cast<const uint2*>(v)[lane];
    m = __vmaxu2(w.x, w.y);
  } else {
    const uint4 w = reinterpret_cast<const uint4*>(v)[lane];
    m = __vmaxu2(__vmaxu2(w.x, w.y), __vmaxu2(w.z, w.w));
  }
  return __reduce_max_sync(FULL, max(m & 0xffffu, m >> 16));
}
// Block-wide result i from buf[N][4] (after a barrier): one 16-byte load.
template <int N>
__device__ __forceinline__ float sum4(const float* buf, int i) {
  const float4 v = reinterpret_cast<const float4*>(buf)[i];
  return (v.x + v.y) + (v.z + v.w);
}
template <int N>
__device__ __forceinline__ float max4(const float* buf, int i) {
  const float4 v = reinterpret_cast<const float4*>(buf)[i];
  return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
}

// A wait that runs out sets the CTA's sticky `fail` word in shared memory;
// every thread reads it after the next CTA barrier, so that all of them leave
// the block loop at the same barrier.  (A plain barrier and a shared word:
// the barrier-reduction form, __syncthreads_and, measured 2-5% slower.)
//
// Thread 0 waits (bounded) for the phase, then the CTA barrier.  Ends with
// the warp converged: the tcgen05.ld / st that follow are .sync.aligned
// (every lane of the warp must execute them together).
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, volatile int* fail, uint64_t limit) {
  if (threadIdx.x == 0 && !mbar_wait_bounded(bar, parity, nullptr, limit)) *fail = 1;
  __syncthreads();
  const bool ok = *fail == 0;
  if (ok) (void)mbar_try_wait(bar, parity);  // completed: observe it in every thread
  __syncwarp();
  return ok;
}
// Every lane of the warp waits (bounded) for the phase, without a CTA
// barrier (each warp then reads only its own lanes of the accumulator); a
// wait that runs out sets `fail`, read after the next CTA barrier.
__device__ __forceinline__ void warp_wait(uint64_t* bar, uint32_t parity, volatile int* fail, uint64_t limit) {
  const bool ok = mbar_wait_bounded(bar, parity, nullptr, limit);
  if (!__all_sync(FULL, ok)) *fail = 1;
}

// Codes of `CHUNKS` 16-byte chunks of row `row` (chunk-major block layout
// with `nrows` rows) -> operand words (E4M3 bytes or exact BF16 values) in
// tensor memory from column taddr: 4 * kOut columns per chunk.
template <int BITS, bool BF16, int CHUNKS>
__device__ __forceinline__ void convert_row(const unsigned char* blk, int nrows, int row, uint32_t taddr, uint32_t mul,
                                            uint32_t m1) {
  using Cv = Convert<BITS, BF16>;
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    const uint4 v = *reinterpret_cast<const uint4*>(blk + ((size_t)c * nrows + row) * 16);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4 * Cv::kOut];
#pragma unroll
    for (int i = 0; i < 4; ++i) Cv::run(w[i], &o[i * Cv::kOut], mul, m1);
#pragma unroll
    for (int q8 = 0; q8 < Cv::kOut / 2; ++q8) tmem_st_x8(taddr + c * 4 * Cv::kOut + 8 * q8, &o[8 * q8]);
  }
}

// ------------------------------------------------------------------ plan
// How the batch is cut into CTAs, computed once per call on the device (the
// plan kernel) from the sequence lengths, so that ragged batches balance
// without a host round trip.  With T the blocks of all units, the CTA count
// aimed at is N = min(N_host, R * max(1, ceil(T / kGenRangeBlocks / R))): the host's count
// (whole waves for max_blocks per unit), lowered when the actual lengths hold
// less work -- to ranges of about kGenRangeBlocks blocks, rounded up to whole
// waves of resident CTAs R (one at least).  Sequence b (nblk_b blocks per unit) gets S_b =
// clamp(floor(nblk_b * N / T), 1, nblk_b) block ranges per unit (none when
// empty); ps[b] = sum over b' < b of units * S_b', ps[B] = the CTAs with work
// (<= N + units of non-empty sequences).  CTA c (ps[b] <= c < ps[b + 1])
// takes unit (c - ps[b]) / S_b, range (c - ps[b]) % S_b, and writes its part
// to slot c.
__device__ __forceinline__ long long gen_aim(long long total, long long n_host, long long n_floor) {
  const long long w = n_floor > 0 ? n_floor : 1;
  const long long want = (total / kGenRangeBlocks + w - 1) / w * w;  // whole waves, at least one
  return want < w ? (w < n_host ? w : n_host) : (want < n_host ? want : n_host);
}
__device__ __forceinline__ int gen_ranges(int nblk, long long total, long long n_target) {
  if (nblk == 0) return 0;
  const long long s = (long long)nblk * n_target / (total > 0 ? total : 1);
  return (int)(s < 1 ? 1 : (s > nblk ? nblk : s));
}
// The plan of a batch with unequal lengths (lens already in shared memory):
// one 64-bit division per sequence and a block-wide scan.  Out of line: the
// common equal-length case keeps the kernel's own code compact.
template <int NT>
static __device__ __noinline__ void gen_plan_ragged(int B, int units, long long n_target, long long n_floor, int* ps,
                                                    const int* lens, long long* red, long long t) {
  constexpr int kWarps = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (B + NT - 1) / NT, b0 = tid * per, b1 = min(B, b0 + per);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(FULL, t, o);
  if (lane == 0) red[w] = t;
  __syncthreads();
  long long total = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) total += red[i];
  total *= units;
  n_target = gen_aim(total, n_target, n_floor);
  int cnt = 0;
  for (int b = b0; b < b1; ++b) {  // this sequence's CTAs, kept in ps[b] until the scan
    const int c = units * gen_ranges((lens[b] + kBlockTokens - 1) / kBlockTokens, total, n_target);
    ps[b] = c;
    cnt += c;
  }
  int incl = cnt;  // inclusive warp scan
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += v;
  }
  __syncthreads();  // red is reused
  if (lane == 31) red[w] = incl;
  __syncthreads();
  int run = incl - cnt;
  for (int i = 0; i < w; ++i) run += (int)red[i];
  for (int b = b0; b < b1; ++b) {
    const int c = ps[b];
    ps[b] = run;
    run += c;
  }
  if (tid == NT - 1) ps[B] = run;
}

// NT threads; ps: shared int[B + 1]; lens: shared int[B] (the validated
// lengths, 0 for a bad one); red: shared long long[NT / 32] scratch.  Each
// thread reads the lengths of a run of consecutive sequences once.
template <int NT>
__device__ __forceinline__ void gen_plan(const int32_t* seq_lens, int B, int max_blocks, int units,
                                         long long n_target, long long n_floor, int* ps, int* lens, long long* red) {
  const int tid = threadIdx.x;
  const int per = (B + NT - 1) / NT, b0 = tid * per, b1 = min(B, b0 + per);
  const int max_len = max_blocks * kBlockTokens;
  int len0 = seq_lens[0];
  if (len0 < 0 || len0 > max_len) len0 = 0;
  long long t = 0;
  bool same = true;
  for (int b = b0; b < b1; ++b) {
    int len = seq_lens[b];
    if (len < 0 || len > max_len) len = 0;
    lens[b] = len;
    same = same && len == len0;
    t += (len + kBlockTokens - 1) / kBlockTokens;
  }
  if (__syncthreads_and(same)) {  // equal lengths: S = min(N / units, nblk) ranges for every unit
    const int nb = (len0 + kBlockTokens - 1) / kBlockTokens;
    const long long all = (long long)B * units;
    n_target = gen_aim(all * nb, n_target, n_floor);
    const int sq = nb == 0 ? 0 : (int)(n_target / all < 1 ? 1 : (n_target / all > nb ? nb : n_target / all));
    for (int b = b0; b < b1; ++b) ps[b] = b * units * sq;
    if (tid == NT - 1) ps[B] = B * units * sq;
  } else {
    gen_plan_ragged<NT>(B, units, n_target, n_floor, ps, lens, red, t);
  }
  __syncthreads();
}
// Sequence of CTA (or slot) c: the b with ps[b] <= c < ps[b + 1] (c < ps[B]).
__device__ __forceinline__ int gen_find(const int* ps, int B, int c) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ps[mid] <= c) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// NH: query heads per unit (4, or 8 with every KV block read once); they
// come in quads of 4 -- one 16-column block (4 heads x 3 E4M3 or 2 BF16
// parts) per quad of Q', S, P' and O.
template <int BITS, bool KCW, bool VCW, int D, int G, bool BF16, int NH>
__global__ void __launch_bounds__(kThreads, gen_min_ctas(BITS, D, G, KCW, VCW, BF16, NH))
decode_general_kernel(const GenParams p, int stages) {
  constexpr int kKBytes = kBlockTokens * D * BITS / 8;  // K (and V) codes of a block
  constexpr int kElems = BF16 ? 16 : 32;                // contraction elements per MMA
  constexpr int kCm = BF16 ? 256 : 128;                 // bytes of one B block per 8 rows
  constexpr int kVCols = BF16 ? 64 : 32;                // operand columns of 128 V codes (one row)
  constexpr uint32_t kFmt = BF16 ? 1u : 0u;             // BF16 (kind::f16) or E4M3 (kind::f8f6f4)
  constexpr int kHalves = D > 128 ? 2 : 1;              // M = 128 halves of the channels
  constexpr int kQv = (D + 127) / 128;                  // channels per thread
  constexpr int HH = NH / 4;                            // head quads
  constexpr int NGC = D / G;                            // channel groups (token-wise)
  constexpr int NGT = kBlockTokens / G;                 // token groups (channel-wise)
  constexpr int NBQ = (KCW ? NGT : 1) * HH;             // 16-column blocks of Q' (and of S with channel-wise K)
  constexpr int NBP = (VCW ? 1 : NGC) * HH;             // of P'
  constexpr int NBO = (VCW ? NGT : NGC) * HH;           // of O per channel half
  constexpr int NSZ = kBlockTokens * D / G;
  constexpr int NM = VCW ? NH : 2 * NH;                 // block-max reduction: heads (+ largest V scale)
  constexpr int NZ = VCW ? NH : 4 * NGC;                // per-group p sums (token-wise V: one quad at a time)
  constexpr bool kQszSmem = NH > 4;                     // token-wise K's q sums in shared memory
  // token-wise V with up to 16 (group, head) pairs: each thread keeps its
  // token's running sum of p * z per channel group and head, reduced once per
  // range (else the per-group sums are reduced across the CTA at every block)
  constexpr bool kZp = !VCW && NGC * NH <= 16;
  extern __shared__ __align__(1024) unsigned char smem[];
  const GenLayout L = gen_layout(BITS, D, G, KCW, VCW, BF16, NH, stages);  // shared-memory offsets
  constexpr GenLayout LT = gen_layout(BITS, D, G, KCW, VCW, BF16, NH, 2);  // tensor-memory columns
  constexpr bool kSeq = LT.seq_halves;
  // Refills: the next copy into a stage goes out as PV starts (nothing reads
  // the stage after that barrier; with channel-wise V and one token group per
  // channel half, kVPre, the epilogue's V scales and offsets are read into
  // registers before it), and no CTA barrier ends the block (the next
  // block's copy wait is the one); the other channel-wise V instances refill
  // after a barrier at the end of the block.  A thread of the last warp
  // issues the refills: thread 0 issues the MMAs and waits for the copies,
  // and a refill on its path delays every warp (measured, refills moved off
  // thread 0: +4.7 points of the peak on INT4 K-cw/V-tw, +3.3 on INT2
  // K-/V-token-wise; early refills for channel-wise V: +2-5).
  constexpr bool kVPre = VCW && NGT * kHalves <= 2;
  constexpr bool kEarlyRefill = !VCW || kVPre;
  constexpr int kRefillTid = kThreads - 32;

  unsigned char* qop = smem + L.q_off;  // [D rows][NBQ blocks]
  unsigned char* pop = smem + L.p_off;  // [128 rows][NBP blocks]
  float* red_c = reinterpret_cast<float*>(smem + L.scratch_off);  // [32][4 warps] q . z_g (channel-wise K)
  float* red_m = red_c + 128;                                     // [16][4] block maxima
  float* red_z = red_m + 64;                                      // [2][32][4] per-group p (z) sums
  float* qsz_s = red_z + 256;  // [8][8] token-wise K q sums (NH = 8); channel-wise K, kMultSmem: the multipliers
  int* pend = reinterpret_cast<int*>(qsz_s + 64);                 // [4] block whose copy into stage s is in flight
  uint64_t* bars = reinterpret_cast<uint64_t*>(qsz_s + 64 + 16);  // (12 spare words) stages [4], mma, drain
  uint32_t* tbase = reinterpret_cast<uint32_t*>(bars + 6);
  volatile int* fail = reinterpret_cast<volatile int*>(tbase + 1);  // a wait ran out (see cta_wait)

  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const int cta = blockIdx.x;
  grid_dep_wait();    // the plan kernel's assignments (this kernel may start while it runs)
  grid_dep_launch();  // the merge kernel may launch (it waits for this grid to complete)
  const int4 asg = p.assign[cta];  // written by general_plan_kernel: {b | unit << 16, j0, j1, length}
  if (asg.x < 0) return;           // no work left for this CTA
  const int b = asg.x & 0xffff, uh = asg.x >> 16, kvh = uh >> p.kv_shift;
  const int j0 = asg.y, j1 = asg.z, len = asg.w;
  const size_t row0 = (size_t)b * p.num_q_heads + (size_t)uh * p.gq;  // first query head of the unit
  float* part_o = p.part_o + (size_t)cta * p.gq * D;  // this CTA's slot: [gq][D] and [gq]
  float* part_lse = p.part_lse + (size_t)cta * p.gq;

  const uint64_t limit = p.wait_limit_ns;
  auto load = [&](int j, int s) {  // one thread: block j of the unit into stage s
    int page = p.page_table ? p.page_table[(size_t)b * p.max_blocks + j] : b * p.max_blocks + j;
    if (page < 0 || page >= p.num_pages) {
      report(p.dev_status, KVQ_DEV_BAD_PAGE);
      page = 0;
    }
    const size_t blk = (size_t)page * p.num_kv_heads + kvh;
    unsigned char* st = smem + s * L.stage_bytes;
    constexpr uint32_t szb = (uint32_t)NSZ * 2;
    mbar_arrive_expect_tx(&bars[s], (uint32_t)L.stage_bytes);
    bulk_g2s(st, p.k_codes + blk * kKBytes, kKBytes, &bars[s]);
    bulk_g2s(st + kKBytes, p.v_codes + blk * kKBytes, kKBytes, &bars[s]);
    unsigned char* sz = st + 2 * kKBytes;
    bulk_g2s(sz, p.k_scale + blk * NSZ, szb, &bars[s]);
    bulk_g2s(sz + szb, p.k_zero + blk * NSZ, szb, &bars[s]);
    bulk_g2s(sz + 2 * szb, p.v_scale + blk * NSZ, szb, &bars[s]);
    bulk_g2s(sz + 3 * szb, p.v_zero + blk * NSZ, szb, &bars[s]);
    pend[s] = j;
  };
  if (tid == 0) {  // the first copies go out before the rest of the set-up
    for (int i = 0; i < 4; ++i) pend[i] = -1;
    *fail = 0;
    for (int i = 0; i < stages; ++i) mbar_init(&bars[i], 1);
    // test hook: this CTA's MMA barrier takes two signals a phase, so its first QK^T wait runs out
    mbar_init(&bars[stages], ((p.flags & KVQ_FLAG_TEST_STALL_MMA) && cta == 0) ? 2u : 1u);
    mbar_init(&bars[stages + 1], 1);
    fence_barrier_init();
    for (int i = 0; i < stages && j0 + i < j1; ++i) {
      if (i == 0 && (p.flags & KVQ_FLAG_TEST_STALL) && blockIdx.x == 0) continue;  // test hook: withhold one block
      load(j0 + i, i);
    }
  }

  for (int i = tid; i < (L.scratch_off - L.q_off) / 16; i += kThreads)
    reinterpret_cast<uint4*>(qop)[i] = make_uint4(0u, 0u, 0u, 0u);  // unused operand columns stay zero
  __syncwarp();  // converged for the .sync.aligned allocation
  if (warp == 0) {
    tmem_alloc(tbase, (uint32_t)LT.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tbase;
  const uint32_t t_a = tmem + lane_off + LT.col_a;    // this warp's lanes of the operand region
  const uint32_t t_so = tmem + lane_off + LT.col_so;  // ... of the S / O region
  uint64_t* mma_bar = &bars[stages];
  uint64_t* drain_bar = &bars[stages + 1];

  // ---- per-unit query statistics (all NH head slots; empty slots are 0)
  const uint16_t* qb = p.q + row0 * D;
  float qv[NH][kQv];  // q of this thread's channels c = tid + 128 i
  float qmax[NH];
#pragma unroll
  for (int k = 0; k < NH; ++k) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < kQv; ++i) {
      const int c = tid + 128 * i;
      qv[k][i] = (k < p.gq && c < D) ? bf2f(qb[k * D + c]) : 0.f;
      m = fmaxf(m, fabsf(qv[k][i]));
    }
    qmax[k] = m;
  }
  {
    float t[NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) t[k] = qmax[k];
    warp_max_store<NH>(t, red_m);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < NH; ++k) qmax[k] = max4<NH>(red_m, k);
  }
  float mult[NH];  // partial-score multiplier (log2 units)
#pragma unroll
  for (int k = 0; k < NH; ++k)
    mult[k] = BF16 ? p.sm_scale_log2  // exact BF16 codes, no prescale
                   : 512.0f * (KCW ? pow2_head_inv(qmax[k]) : pow2_prescale_inv(qmax[k])) * p.sm_scale_log2;
  // channel-wise K (E4M3) where registers are short (8 heads at 5 CTAs per
  // SM, 96 registers a thread; 2-bit codes at 8, 64 a thread): q . z_g is
  // taken against the prescaled q, so that q itself is not kept, and with 8
  // heads the multipliers wait in shared memory (the q sums' buffer, unused
  // by this scheme).  (Measured: 8 heads +2.5-3 points of the peak with 4-bit
  // codes, +1.3-2.5 with 2-bit; 4 heads 2-bit +1.1-1.5; 4-bit codes with 4
  // heads, whose registers suffice, lost 2-4 points, the BF16 mode 0-0.2.)
  constexpr bool kQkZ = KCW && !BF16 && (NH > 4 || BITS == 2);
  constexpr bool kMultSmem = kQkZ && NH > 4;
  if (kMultSmem && tid < NH) qsz_s[tid] = mult[tid];
  float qsz[kQszSmem ? 1 : NGC][NH];  // token-wise K: sum of q over channel group g, times the log2 scale
  if (!KCW) {
    // Q' = q * 2^k (k per head) in three E4M3 parts at row a_pos(c), one
    // block per head quad; and the per-channel-group sums of q for the offset
#pragma unroll
    for (int i = 0; i < kQv; ++i) {
      const int c = tid + 128 * i;
      if (c < D) {
        const float f = odd_quarter<BITS, BF16>(c);
#pragma unroll
        for (int hq = 0; hq < HH; ++hq) {
          float x[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) x[h] = qv[4 * hq + h][i] * (BF16 ? 1.0f : pow2_prescale(qmax[4 * hq + h])) * f;
          const float4 v = make_float4(x[0], x[1], x[2], x[3]);
          *reinterpret_cast<uint4*>(qop + b_off<BF16>(a_pos<BITS, BF16>(c), hq, HH)) = BF16 ? split2_bf16(v)
                                                                                           : split3_e4m3(v);
        }
      }
    }
#pragma unroll
    for (int hq = 0; hq < HH; ++hq) {
      float t[4 * NGC];
#pragma unroll
      for (int g = 0; g < NGC; ++g)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float s = 0.f;
#pragma unroll
          for (int i = 0; i < kQv; ++i)
            if ((tid + 128 * i) / G == g && tid + 128 * i < D) s += qv[4 * hq + h][i];
          t[g * 4 + h] = s;
        }
      warp_reduce_store<4 * NGC, false>(t, red_z + hq * 128);
    }
    fence_proxy_async_smem();
    __syncthreads();
#pragma unroll
    for (int g = 0; g < NGC; ++g)
#pragma unroll
      for (int k = 0; k < NH; ++k) {
        const float v = sum4<4 * NGC>(red_z + (k >> 2) * 128, g * 4 + (k & 3)) * p.sm_scale_log2;
        if (kQszSmem) {
          if (tid == 0) qsz_s[g * NH + k] = v;
        } else {
          qsz[kQszSmem ? 0 : g][k] = v;
        }
      }
    if (kQszSmem) __syncthreads();
  }
  float qk[NH][kQv];  // channel-wise K: q * 2^(6 - E_q)
#pragma unroll
  for (int k = 0; k < NH; ++k)
#pragma unroll
    for (int i = 0; i < kQv; ++i) qk[k][i] = BF16 ? qv[k][i] : qv[k][i] * pow2_head(qmax[k]);

  float m_run[NH], l_thr[NH], oacc[kHalves][NH], zacc[kHalves][NH];
  float zp[kZp ? NGC : 1][kZp ? NH : 1];  // kZp: this token's running sum of p * z
#pragma unroll
  for (int k = 0; k < NH; ++k) {
    m_run[k] = -INFINITY;
    l_thr[k] = 0.f;
#pragma unroll
    for (int hf = 0; hf < kHalves; ++hf) oacc[hf][k] = zacc[hf][k] = 0.f;
  }
#pragma unroll
  for (int g = 0; g < (kZp ? NGC : 1); ++g)
#pragma unroll
    for (int k = 0; k < (kZp ? NH : 1); ++k) zp[g][k] = 0.f;

  bool ok = true;
  uint32_t mma_phase = 0u;
  for (int j = j0; j < j1; ++j) {
    const int s = (j - j0) % stages;
    if (!cta_wait(&bars[s], (uint32_t)((j - j0) / stages) & 1u, fail, limit)) { ok = false; break; }
    const unsigned char* st = smem + s * L.stage_bytes;
    const uint16_t* ksz = reinterpret_cast<const uint16_t*>(st + 2 * kKBytes);
    const uint16_t* kzz = ksz + NSZ;
    const uint16_t* vsz = kzz + NSZ;
    const uint16_t* vzz = vsz + NSZ;
    const int nv = min(kBlockTokens, len - j * kBlockTokens);  // valid tokens of the block
    const int l = tid;
    const bool valid = l < nv;

    // ---- channel-wise K: the largest scale of each group (the E4M3 Q'
    //      prescale), found by every warp on its own; with one token group
    //      ahead of the K conversion, which hides its latency (with several,
    //      after it: the values held across it cost more than they hide)
    uint32_t e16[KCW && !BF16 ? NGT : 1];
    auto group_maxima = [&]() {
#pragma unroll
      for (int g = 0; g < (KCW && !BF16 ? NGT : 1); ++g) e16[g] = f16_exp_field(max_f16_bits<D>(ksz + g * D));
    };
    if (KCW && !BF16 && NGT == 1) group_maxima();

    // ---- K codes -> E4M3 operand (rows = tokens)
    __syncwarp();
    convert_row<BITS, BF16, D * BITS / 128>(st, kBlockTokens, tid, t_a, p.nibble_mul, p.minus_one);
    tc_wait_st();
    if (KCW && !BF16 && NGT > 1) group_maxima();

    // ---- channel-wise K: Q'_g = q * s_g per token group g, and q . z_g
    float t[KCW ? NH * NGT : 1];  // channel-wise K: q . z_g (this thread's channels), value g * NH + k
    if (KCW) {
#pragma unroll
      for (int k = 0; k < NH * NGT; ++k) t[k] = 0.f;
#pragma unroll
      for (int g = 0; g < NGT; ++g) {
        const float fg = BF16 ? 1.0f : pow2_group(e16[KCW && !BF16 ? g : 0]);
#pragma unroll
        for (int i = 0; i < kQv; ++i) {
          const int c = tid + 128 * i;
          if (c < D) {
            const float f = h2f(ksz[g * D + c]) * fg * odd_quarter<BITS, BF16>(c);
#pragma unroll
            for (int hq = 0; hq < HH; ++hq) {
              const float4 v = make_float4(qk[4 * hq][i] * f, qk[4 * hq + 1][i] * f, qk[4 * hq + 2][i] * f,
                                           qk[4 * hq + 3][i] * f);
              *reinterpret_cast<uint4*>(qop + b_off<BF16>(a_pos<BITS, BF16>(c), g * HH + hq, NBQ)) =
                  BF16 ? split2_bf16(v) : split3_e4m3(v);
            }
            // the offsets in log2 score units; or, kQkZ, times 2^-9 against the
            // prescaled q (the score multiplier holds 2^9 / prescale)
            const float zgc = h2f(kzz[g * D + c]) * (kQkZ ? 1.0f / 512.0f : p.sm_scale_log2);
#pragma unroll
            for (int k = 0; k < NH; ++k) t[g * NH + k] = fmaf(kQkZ ? qk[k][i] : qv[k][i], zgc, t[g * NH + k]);
          }
        }
      }
      fence_proxy_async_smem();
    }

    // ---- QK^T: S[token][column block] (swap-AB: tokens are the M = 128 rows)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      constexpr uint32_t idesc_q = make_idesc(kFmt, kFmt, 0, 1, 128, 16 * NBQ);
#pragma unroll
      for (int k = 0; k < D / kElems; ++k) {
        const uint64_t bd = make_smem_desc(smem_u32(qop) + k * 4 * NBQ * 128, NBQ * kCm, 128);
        const uint32_t a = tmem + LT.col_a + 8 * k;
        // channel-wise K: one accumulator; token-wise K: the K-steps of channel
        // group g accumulate into S blocks g * HH ... (both head quads)
        const uint32_t d = tmem + LT.col_so + (KCW ? 0 : 16 * HH * ((kElems * k) / G));
        const uint32_t acc = KCW ? (k > 0) : ((kElems * k) % G != 0);
        if (BF16) mma_f16_ts(d, a, bd, idesc_q, acc);
        else mma_f8f6f4_ts(d, a, bd, idesc_q, acc);
      }
      tc_commit(mma_bar);
    }
    // while QK^T runs: the warps' sums of q . z_g (channel-wise K; read after
    // the barrier that ends the wait for QK^T) and the largest V scale of
    // this token (token-wise V)
    if (KCW) warp_reduce_store<KCW ? NH * NGT : 1, false>(t, red_c);
    float vmax = 0.f;
    if (!VCW && valid) {
#pragma unroll
      for (int g = 0; g < NGC; ++g) vmax = fmaxf(vmax, h2f(vsz[l * NGC + g]));
    }
    // token-wise K: each warp waits for QK^T on its own and reads its lanes
    // of S (one CTA barrier less per block); channel-wise K waits as a CTA,
    // which also completes red_c.  (Channel-wise K with per-warp waits, q . z_g
    // then added after the block-maxima barrier, measured 1-4 points slower.)
    if (!KCW) {
      warp_wait(mma_bar, mma_phase, fail, limit);
    } else if (!cta_wait(mma_bar, mma_phase, fail, limit)) {
      ok = false;
      break;
    }
    mma_phase ^= 1u;
    tc_fence_after();

    // ---- scores of token l (log2 units), folded per group
    float sc[NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) sc[k] = 0.f;
    if (KCW) {
      const int g = l / G;  // warp-uniform (G >= 32)
      float fs = 1.0f;
      if (!BF16) {
#pragma unroll
        for (int gg = 0; gg < (KCW && !BF16 ? NGT : 1); ++gg)
          if (gg == g) fs = pow2_group_inv(e16[gg]);
      }
#pragma unroll
      for (int hq = 0; hq < HH; ++hq) {
        uint32_t v[12];
        ld_block<BF16>(t_so + 16 * (g * HH + hq), v);
        float cz[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) cz[h] = sum4<NH * NGT>(red_c, g * NH + 4 * hq + h);
        tc_wait_ld();
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int k = 4 * hq + h;
          sc[k] = kQkZ ? (kMultSmem ? qsz_s[k] : mult[k]) * fmaf(parts<BF16>(v, h), fs, cz[h])
                       : fmaf(parts<BF16>(v, h), mult[k] * fs, cz[h]);
        }
      }
    } else {
#pragma unroll
      for (int g = 0; g < NGC; ++g) {
        const float s_lg = h2f(ksz[l * NGC + g]), z_lg = h2f(kzz[l * NGC + g]);
#pragma unroll
        for (int hq = 0; hq < HH; ++hq) {
          uint32_t v[12];
          ld_block<BF16>(t_so + 16 * (g * HH + hq), v);
          tc_wait_ld();
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int k = 4 * hq + h;
            const float qs = kQszSmem ? qsz_s[g * NH + k] : qsz[kQszSmem ? 0 : g][k];
            sc[k] += fmaf(parts<BF16>(v, h) * mult[k], s_lg, z_lg * qs);
          }
        }
      }
    }
#pragma unroll
    for (int k = 0; k < NH; ++k) sc[k] = valid ? sc[k] : -INFINITY;

    // ---- V codes -> E4M3 operand (rows = channels), replacing the K codes
    //      (QK^T is complete).  A 64-dim head leaves rows 64..127 as they are:
    //      output row m depends on operand row m alone, and rows >= D are
    //      never read.
    __syncwarp();
#pragma unroll
    for (int hf = 0; hf < kHalves; ++hf)
      if (hf * 128 + tid < D)  // warp-uniform
        convert_row<BITS, BF16, BITS>(st + kKBytes, D, hf * 128 + tid, t_a + kVCols * hf, p.nibble_mul,
                                      p.minus_one);

    // ---- online softmax over the block: block maxima (and the largest V scale)
    {  // red_m[NM][warp]: value k < NH the head maxima, NM - 1 the largest V scale
      const int lane = tid & 31;
      float mine = 0.f;
#pragma unroll
      for (int k = 0; k < NH; ++k) {
        const float r = warp_max_redux(sc[k]);
        mine = lane == k ? r : mine;
      }
      if (!VCW) {
        const float r = warp_max_redux(vmax);
        mine = lane == NM - 1 ? r : mine;
      }
      if (lane < NM) red_m[lane * 4 + warp] = mine;
      __syncwarp();
    }
    tc_wait_st();
    __syncthreads();
    if (*fail) { ok = false; break; }  // a per-warp QK^T wait ran out
    float bmax[NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) bmax[k] = max4<NM>(red_m, k);
    const int e_v = VCW ? 0 : (int)((__float_as_uint(max4<NM>(red_m, NM - 1)) >> 23) & 0xffu) - 127;
    float alpha[NH], pr[NH];
    int pe[NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) {
      const float mn = fmaxf(m_run[k], bmax[k]);
      alpha[k] = ex2(m_run[k] - mn);
      m_run[k] = mn;
      pr[k] = valid ? ex2(sc[k] - mn) : 0.f;
      pe[k] = BF16 ? 6 : p_exponent(bmax[k] - mn, e_v);  // P' prescale 2^(6 - E) (1 for BF16)
      l_thr[k] = fmaf(l_thr[k], alpha[k], pr[k]);
    }

    // per-group sums: token-wise V: sum_l p_l z_(l,g) per channel group (one
    // head quad per buffer); channel-wise V: sum_(l in g) p_l per token group
    // (a warp's tokens lie in one group)
    if (kZp) {
#pragma unroll
      for (int g = 0; g < (kZp ? NGC : 1); ++g) {
        const float z_lg = valid ? h2f(vzz[l * NGC + g]) : 0.f;
#pragma unroll
        for (int k = 0; k < (kZp ? NH : 1); ++k) zp[g][k] = fmaf(zp[g][k], alpha[k], pr[k] * z_lg);
      }
    } else if (!VCW) {
#pragma unroll
      for (int hq = 0; hq < HH; ++hq) {
        float t[NZ];
#pragma unroll
        for (int g = 0; g < NGC; ++g) {
          const float z_lg = valid ? h2f(vzz[l * NGC + g]) : 0.f;
#pragma unroll
          for (int h = 0; h < 4; ++h) t[g * 4 + h] = pr[4 * hq + h] * z_lg;
        }
        warp_reduce_store<NZ, false>(t, red_z + hq * 128);
      }
    } else {
      float t[NZ];
#pragma unroll
      for (int k = 0; k < NH; ++k) t[k] = pr[k];
      warp_reduce_store<NZ, false>(t, red_z);
    }

    // ---- P' operand: row a_pos(l), one 16-column block per channel group
    //      (token-wise V) and head quad
    {
      const float oq = odd_quarter<BITS, BF16>(l);
      float ps[NH];
#pragma unroll
      for (int k = 0; k < NH; ++k) ps[k] = pr[k] * oq * __uint_as_float((uint32_t)(133 - pe[k]) << 23);
#pragma unroll
      for (int g = 0; g < NBP / HH; ++g) {
        const float sv = VCW ? 1.0f : (valid ? h2f(vsz[l * NGC + g]) : 0.f);
#pragma unroll
        for (int hq = 0; hq < HH; ++hq) {
          const float4 v = make_float4(ps[4 * hq] * sv, ps[4 * hq + 1] * sv, ps[4 * hq + 2] * sv, ps[4 * hq + 3] * sv);
          *reinterpret_cast<uint4*>(pop + b_off<BF16>(a_pos<BITS, BF16>(l), g * HH + hq, NBP)) =
              BF16 ? split2_bf16(v) : split3_e4m3_via_f16(v);
        }
      }
    }
    fence_proxy_async_smem();

    float pinv[NH];  // 2^(E - 6), times 2^9 for E4M3 codes (code * 2^-9)
#pragma unroll
    for (int k = 0; k < NH; ++k) pinv[k] = __uint_as_float((uint32_t)((BF16 ? 121 : 130) + pe[k]) << 23);

    float vpre_s[kVPre ? kHalves : 1][kVPre ? NGT : 1], vpre_z[kVPre ? kHalves : 1][kVPre ? NGT : 1];
    if (kVPre) {
#pragma unroll
      for (int hf = 0; hf < (kVPre ? kHalves : 1); ++hf)
#pragma unroll
        for (int g = 0; g < (kVPre ? NGT : 1); ++g) {
          const int c = hf * 128 + tid;
          vpre_s[hf][g] = c < D ? h2f(vsz[g * D + c]) : 0.f;
          vpre_z[hf][g] = c < D ? h2f(vzz[g * D + c]) : 0.f;
        }
    }

    // ---- PV: O[channel][column block] per M = 128 half of the channels, then
    //      the epilogue: channel c = 128 hf + tid; undo the P' prescale, fold V
#pragma unroll
    for (int pass = 0; pass < (kSeq ? kHalves : 1); ++pass) {
      tc_fence_before();
      __syncthreads();
      if (pass > 0 && *fail) { ok = false; break; }  // pass 0's PV wait
      tc_fence_after();
      if (tid == 0) {
#pragma unroll
        for (int hf = 0; hf < kHalves; ++hf) {
          if (kSeq && hf != pass) continue;
          const uint32_t o = tmem + LT.col_so + (kSeq ? 0 : hf * 16 * NBO);
#pragma unroll
          for (int k = 0; k < kBlockTokens / kElems; ++k) {
            const uint32_t a = tmem + LT.col_a + kVCols * hf + 8 * k;
            // channel-wise V: the K-steps of token group g accumulate into O
            // blocks g * HH ... (both head quads)
            const uint64_t bd = make_smem_desc(smem_u32(pop) + k * 4 * NBP * 128, NBP * kCm, 128);
            const uint32_t d = VCW ? o + 16 * HH * ((kElems * k) / G) : o;
            const uint32_t acc = VCW ? ((kElems * k) % G != 0) : (k > 0);
            constexpr uint32_t idesc_p = make_idesc(kFmt, kFmt, 0, 1, 128, 16 * NBP);
            if (BF16) mma_f16_ts(d, a, bd, idesc_p, acc);
            else mma_f8f6f4_ts(d, a, bd, idesc_p, acc);
          }
        }
        tc_commit(mma_bar);
      }
      if (kEarlyRefill && pass == 0 && tid == kRefillTid) {  // nothing reads the stage after this barrier
        pend[s] = -1;
        if (j + stages < j1) load(j + stages, s);
      }
      warp_wait(mma_bar, mma_phase, fail, limit);  // each warp reads its own lanes of O
      mma_phase ^= 1u;
      tc_fence_after();
#pragma unroll
      for (int hf = 0; hf < kHalves; ++hf) {
        if (kSeq && hf != pass) continue;
        const int c = hf * 128 + tid;
        const uint32_t o = t_so + (kSeq ? 0 : hf * 16 * NBO);
        float add[NH];
#pragma unroll
        for (int k = 0; k < NH; ++k) add[k] = 0.f;
        if (VCW) {
#pragma unroll
          for (int g = 0; g < NGT; ++g) {
#pragma unroll
            for (int hq = 0; hq < HH; ++hq) {
              uint32_t v[12];
              ld_block<BF16>(o + 16 * (g * HH + hq), v);
              tc_wait_ld();
              if (g * G >= nv || c >= D) continue;  // no valid token in this group / no such channel
              const float s_gc = kVPre ? vpre_s[kVPre ? hf : 0][kVPre ? g : 0] : h2f(vsz[g * D + c]);
              const float z_gc = kVPre ? vpre_z[kVPre ? hf : 0][kVPre ? g : 0] : h2f(vzz[g * D + c]);
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const int k = 4 * hq + h;
                float psum = 0.f;  // sum of p over the group's tokens (the warps covering them)
#pragma unroll
                for (int w = 0; w < 4; ++w)
                  if ((32 * w) / G == g) psum += red_z[k * 4 + w];
                add[k] = fmaf(s_gc, parts<BF16>(v, h) * pinv[k], fmaf(z_gc, psum, add[k]));
              }
            }
          }
        } else {
          const int g = (c < D ? c : 0) / G;  // warp-uniform (G >= 32)
#pragma unroll
          for (int hq = 0; hq < HH; ++hq) {
            uint32_t v[12];
            ld_block<BF16>(o + 16 * (g * HH + hq), v);
            tc_wait_ld();
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int k = 4 * hq + h;
              add[k] = parts<BF16>(v, h) * pinv[k];
              if (!kZp) zacc[hf][k] = fmaf(zacc[hf][k], alpha[k], sum4<NZ>(red_z + hq * 128, g * 4 + h));
            }
          }
        }
#pragma unroll
        for (int k = 0; k < NH; ++k) oacc[hf][k] = fmaf(oacc[hf][k], alpha[k], add[k]);
      }
    }
    if (!ok) break;
    if (!kEarlyRefill) {
      tc_fence_before();
      __syncthreads();  // stage s, Q', P', S / O and the reduction buffers are free again
      if (*fail) { ok = false; break; }
      if (tid == kRefillTid) {
        pend[s] = -1;
        if (j + stages < j1) load(j + stages, s);
      }
    }
  }

  // the last PV wait's outcome; every refill (and its pend entry) is issued
  __syncthreads();
  ok = ok && *fail == 0;

  // ---- this range's part: O / l and lse = m + ln l per head
  if (ok) {
    {
      float t[NH];
#pragma unroll
      for (int k = 0; k < NH; ++k) t[k] = l_thr[k];
      warp_reduce_store<NH, false>(t, red_m);
    }
    if (kZp) {  // the range's sum of p * z per channel group and head: red_z[g * NH + k][warp]
      constexpr int NP = kZp ? NGC * NH : 1;
      float t[NP];
#pragma unroll
      for (int g = 0; g < (kZp ? NGC : 1); ++g)
#pragma unroll
        for (int k = 0; k < (kZp ? NH : 1); ++k) t[g * NH + k] = zp[g][k];
      warp_reduce_store<NP, false>(t, red_z);
    }
    __syncthreads();
    float l_run[NH];
#pragma unroll
    for (int k = 0; k < NH; ++k) l_run[k] = sum4<NH>(red_m, k);
    if (kZp) {
#pragma unroll
      for (int hf = 0; hf < kHalves; ++hf) {
        const int g = (hf * 128 + tid < D ? hf * 128 + tid : 0) / G;
#pragma unroll
        for (int k = 0; k < NH; ++k) zacc[hf][k] = sum4<kZp ? NGC * NH : 1>(red_z, g * NH + k);
      }
    }
#pragma unroll
    for (int hf = 0; hf < kHalves; ++hf) {
      const int c = hf * 128 + tid;
      if (c < D) {
#pragma unroll
        for (int k = 0; k < NH; ++k)
          if (k < p.gq) part_o[k * D + c] = (oacc[hf][k] + zacc[hf][k]) / l_run[k];
      }
    }
#pragma unroll
    for (int k = 0; k < NH; ++k)
      if (tid == k && k < p.gq)
        part_lse[k] = (m_run[k] + __log2f(l_run[k])) * 0.69314718055994530942f;
  } else if (tid == 0) {
    report(p.dev_status, KVQ_DEV_TIMEOUT);
  }
  // leave no copy or MMA in flight: wait (bounded) for both, then release tensor memory
  if (tid == 0) {
    for (int s = 0; s < stages; ++s)
      if (pend[s] >= 0)
        (void)mbar_wait_bounded(&bars[s], (uint32_t)((pend[s] - j0) / stages) & 1u, nullptr, limit);
    tc_commit(drain_bar);
    (void)mbar_wait_bounded(drain_bar, 0u, nullptr, limit);
  }
  tc_fence_before();
  __syncthreads();
  __syncwarp();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)LT.tmem_cols);
  }
}

template <int BITS, bool KCW, bool VCW, int D, int G, bool BF16, int NH>
cudaError_t launch_instance(const GenParams& p, int grid, const GenLaunch& shape, cudaStream_t stream) {
  auto kern = decode_general_kernel<BITS, KCW, VCW, D, G, BF16, NH>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)shape.smem);
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the CTAs start while the plan kernel runs
  // and wait for it in the kernel (grid_dep_wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = shape.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, (int)shape.stages);
}

template <int BITS, int D, int G, bool BF16, int NH>
cudaError_t launch_schemes(bool kcw, bool vcw, const GenParams& p, int grid, const GenLaunch& shape, cudaStream_t s) {
  if (!kcw && !vcw) return launch_instance<BITS, false, false, D, G, BF16, NH>(p, grid, shape, s);
  if (!kcw && vcw) return launch_instance<BITS, false, true, D, G, BF16, NH>(p, grid, shape, s);
  if (kcw && !vcw) return launch_instance<BITS, true, false, D, G, BF16, NH>(p, grid, shape, s);
  return launch_instance<BITS, true, true, D, G, BF16, NH>(p, grid, shape, s);
}

}  // namespace gen
}  // namespace kvq
