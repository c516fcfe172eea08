// Decode attention for the cache geometries the specialised kernel does not
// take: head dims 64 and 256, groups of 32 or 64 elements (with any head
// dim).  One warpgroup per CTA runs every step of a 128-token block in turn
// -- bulk copies into a two-stage ring, codes to E4M3 operands in tensor
// memory, Q' and P' operands in shared memory, tcgen05 MMAs with the
// accumulators in tensor memory, the affine folds and an online softmax --
// over a contiguous range of one (sequence, unit)'s blocks; the ranges'
// partial results are merged by log-sum-exp afterwards.  Several CTAs share
// an SM (as many as their tensor-memory columns allow), so that one CTA's
// copies and MMAs overlap the others' arithmetic.
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
#include "decode.cuh"
#include "decode_general.h"

namespace kvq {

namespace {

constexpr int kGenThreads = 128;

// Byte offset of row p, 16-column block nb of a B operand with nb16 blocks
// (MN-major, no swizzle: core matrices of 8 rows x 16 bytes; K-direction
// stride nb16 * 128, N-direction stride 128).
__device__ __forceinline__ uint32_t b_off(int p, int nb, int nb16) {
  return (uint32_t)((p >> 3) * (nb16 * 128) + nb * 128 + (p & 7) * 16);
}

__device__ __forceinline__ void tmem_st_x8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// The 12 used columns of a 16-column block (4 heads x 3 parts).
__device__ __forceinline__ void ld_block(uint32_t taddr, uint32_t (&v)[12]) {
  tmem_ld_32x32b_x8(taddr, v);
  tmem_ld_32x32b_x4(taddr + 8, v + 8);
  tc_wait_ld();
}
// Sum of the three parts of head h.
__device__ __forceinline__ float parts3(const uint32_t (&v)[12], int h) {
  return (__uint_as_float(v[h]) + __uint_as_float(v[4 + h])) + __uint_as_float(v[8 + h]);
}

// Block-wide (128 threads) sum or max of 4 values per thread; every thread
// gets the results.  red: 16 floats of shared memory.
__device__ __forceinline__ void block_reduce4(float (&v)[4], float* red, bool is_max) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 0; h < 4; ++h) v[h] = is_max ? warp_maxf(v[h]) : warp_sum(v[h]);
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < 4; ++h) red[w * 4 + h] = v[h];
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float a = red[h], b = red[4 + h], c = red[8 + h], d = red[12 + h];
    v[h] = is_max ? fmaxf(fmaxf(a, b), fmaxf(c, d)) : (a + b) + (c + d);
  }
}

// Thread 0 waits (bounded) for the phase; the whole CTA learns the outcome,
// so that a wait that runs out leaves every thread on the same path.
__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, int* ok_flag, uint64_t limit) {
  if (threadIdx.x == 0) *ok_flag = mbar_wait_bounded(bar, parity, nullptr, limit) ? 1 : 0;
  __syncthreads();
  const bool ok = *ok_flag != 0;
  if (ok && threadIdx.x != 0) (void)mbar_try_wait(bar, parity);  // completed: observe it in every thread
  return ok;
}

template <int BITS, bool KCW, bool VCW, int D>
__global__ void __launch_bounds__(kGenThreads, 4) decode_general_kernel(const GenParams p) {
  constexpr int kKBytes = kBlockTokens * D * BITS / 8;  // K (and V) codes of a block
  constexpr int kKChunks = D * BITS / 128;              // 16-byte chunks of a K row (one token)
  constexpr int kVChunks = BITS;                        // of a V row (one channel: 128 tokens)
  constexpr int kHalves = D > 128 ? 2 : 1;              // M = 128 halves of the channels
  constexpr int kQv = (D + 127) / 128;                  // channels per thread
  extern __shared__ __align__(1024) unsigned char smem[];
  const int G = p.group;
  const int ngc = D / G;            // channel groups (token-wise)
  const int ngt = kBlockTokens / G;  // token groups (channel-wise)
  const GenLayout L = gen_layout(BITS, D, G, KCW, VCW);
  const int nsz = L.nsz;

  unsigned char* qop = smem + L.q_off;  // [D rows][nbq blocks]
  unsigned char* pop = smem + L.p_off;  // [128 rows][nbp blocks]
  float* red = reinterpret_cast<float*>(smem + L.scratch_off);  // 16
  float* gsum = red + 16;   // [8 groups][4 heads] per-group sums of this block
  float* zrun = gsum + 32;  // [8][4] token-wise V: running sum of p * z
  float* cgs = zrun + 32;   // [4][4] channel-wise K: q . z_g
  uint32_t* eg = reinterpret_cast<uint32_t*>(cgs + 16);  // [4] channel-wise K: largest scale of group g
  uint64_t* bars = reinterpret_cast<uint64_t*>(eg + 4);  // stage full [2], mma, drain
  uint32_t* tbase = reinterpret_cast<uint32_t*>(bars + 4);
  int* ok_flag = reinterpret_cast<int*>(tbase + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const int unit = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  const int b = unit / p.units_per_seq, uh = unit % p.units_per_seq, kvh = uh >> p.kv_shift;
  int len = p.seq_lens[b];
  if (len < 0 || len > p.max_blocks * kBlockTokens) {
    if (split == 0 && uh == 0 && tid == 0) report(p.dev_status, KVQ_DEV_BAD_SEQ_LEN);
    len = 0;
  }
  const int nblk = (len + kBlockTokens - 1) / kBlockTokens;
  const int j0 = (int)((long long)split * nblk / p.splits), j1 = (int)((long long)(split + 1) * nblk / p.splits);
  const size_t row0 = (size_t)b * p.num_q_heads + (size_t)uh * p.gq;  // first query head of the unit

  if (j1 <= j0) {  // no block in this range: an empty part (weight 0 in the merge)
    for (int k = 0; k < p.gq; ++k) {
      for (int c = tid; c < D; c += kGenThreads) p.part_o[((row0 + k) * p.splits + split) * D + c] = 0.f;
      if (tid == 0) p.part_lse[(row0 + k) * p.splits + split] = -INFINITY;
    }
    return;
  }

  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
    fence_barrier_init();
  }
  for (int i = tid; i < (L.scratch_off - L.q_off) / 16; i += kGenThreads)
    reinterpret_cast<uint4*>(qop)[i] = make_uint4(0u, 0u, 0u, 0u);  // unused operand columns stay zero
  if (tid < 32) zrun[tid] = 0.f;
  if (warp == 0) {
    tmem_alloc(tbase, (uint32_t)L.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tbase;
  if (D < 128) {  // channel rows 64..127 of the V operand stay zero (M = 128 with 64 channels)
    const uint32_t z8[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int c = 0; c < 32; c += 8) tmem_st_x8(tmem + lane_off + L.col_av + c, z8);
    tc_wait_st();
  }

  const uint64_t limit = p.wait_limit_ns;
  int pend[2] = {-1, -1};  // thread 0: block whose copy into stage s is in flight
  auto load = [&](int j, int s) {  // thread 0: block j of the unit into stage s
    int page = p.page_table ? p.page_table[(size_t)b * p.max_blocks + j] : b * p.max_blocks + j;
    if (page < 0 || page >= p.num_pages) {
      report(p.dev_status, KVQ_DEV_BAD_PAGE);
      page = 0;
    }
    const size_t blk = (size_t)page * p.num_kv_heads + kvh;
    unsigned char* st = smem + s * L.stage_bytes;
    const uint32_t szb = (uint32_t)nsz * 2;
    mbar_arrive_expect_tx(&bars[s], (uint32_t)L.stage_bytes);
    bulk_g2s(st, p.k_codes + blk * kKBytes, kKBytes, &bars[s]);
    bulk_g2s(st + kKBytes, p.v_codes + blk * kKBytes, kKBytes, &bars[s]);
    unsigned char* sz = st + 2 * kKBytes;
    bulk_g2s(sz, p.k_scale + blk * nsz, szb, &bars[s]);
    bulk_g2s(sz + szb, p.k_zero + blk * nsz, szb, &bars[s]);
    bulk_g2s(sz + 2 * szb, p.v_scale + blk * nsz, szb, &bars[s]);
    bulk_g2s(sz + 3 * szb, p.v_zero + blk * nsz, szb, &bars[s]);
    pend[s] = j;
  };
  if (tid == 0) {
    // test hook: the first CTA withholds its first block, so its wait runs out
    if (!((p.flags & KVQ_FLAG_TEST_STALL) && blockIdx.x == 0)) load(j0, 0);
    if (j0 + 1 < j1) load(j0 + 1, 1);
  }

  // ---- per-unit query statistics (all 4 head slots; empty slots are 0)
  const uint16_t* qb = p.q + row0 * D;
  float qmax[4], qv[4][kQv];  // q of this thread's channels c = tid + 128 i
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < kQv; ++i) {
      const int c = tid + 128 * i;
      qv[h][i] = (h < p.gq && c < D) ? bf2f(qb[h * D + c]) : 0.f;
      m = fmaxf(m, fabsf(qv[h][i]));
    }
    qmax[h] = m;
  }
  block_reduce4(qmax, red, true);
  float mult[4];  // partial-score multiplier (log2 units)
#pragma unroll
  for (int h = 0; h < 4; ++h)
    mult[h] = 512.0f * (KCW ? pow2_head_inv(qmax[h]) : pow2_prescale_inv(qmax[h])) * p.sm_scale_log2;
  float qsz[8][4];  // token-wise K: sum of q over channel group g, times the log2 softmax scale
  if (!KCW) {
    // Q' = q * 2^k (k per head) in three E4M3 parts at row a_pos(c); and the
    // per-channel-group sums of q for the offset term
#pragma unroll
    for (int i = 0; i < kQv; ++i) {
      const int c = tid + 128 * i;
      if (c < D) {
        const float f = odd_quarter<BITS, false>(c);
        const float4 v = make_float4(qv[0][i] * pow2_prescale(qmax[0]) * f, qv[1][i] * pow2_prescale(qmax[1]) * f,
                                     qv[2][i] * pow2_prescale(qmax[2]) * f, qv[3][i] * pow2_prescale(qmax[3]) * f);
        *reinterpret_cast<uint4*>(qop + b_off(a_pos<BITS, false>(c), 0, 1)) = split3_e4m3(v);
      }
    }
    if (tid < 32) gsum[tid] = 0.f;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kQv; ++i) {
      const int c = tid + 128 * i;  // a warp's 32 channels lie in one group (G >= 32)
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float s = warp_sum(qv[h][i]);
        if (lane == 0 && c < D) atomicAdd(&gsum[(c / G) * 4 + h], s);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
#pragma unroll
    for (int g = 0; g < 8; ++g)
#pragma unroll
      for (int h = 0; h < 4; ++h) qsz[g][h] = g < ngc ? gsum[g * 4 + h] * p.sm_scale_log2 : 0.f;
  }

  float m_run[4], l_run[4], oacc[kHalves][4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int hf = 0; hf < kHalves; ++hf) oacc[hf][h] = 0.f;
  }

  bool ok = true;
  uint32_t mma_phase = 0u;
  for (int j = j0; j < j1; ++j) {
    const int s = (j - j0) & 1;
    if (!cta_wait(&bars[s], (uint32_t)((j - j0) >> 1) & 1u, ok_flag, limit)) { ok = false; break; }
    const unsigned char* st = smem + s * L.stage_bytes;
    const uint16_t* ksz = reinterpret_cast<const uint16_t*>(st + 2 * kKBytes);
    const uint16_t* kzz = ksz + nsz;
    const uint16_t* vsz = kzz + nsz;
    const uint16_t* vzz = vsz + nsz;
    const int nv = min(kBlockTokens, len - j * kBlockTokens);  // valid tokens of the block
    const int l = tid;
    const bool valid = l < nv;

    // ---- codes -> E4M3 operands in tensor memory (K rows = tokens, V rows = channels)
    {
#pragma unroll
      for (int c = 0; c < kKChunks; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(st + ((size_t)c * kBlockTokens + tid) * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[16];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          Convert<BITS, false>::run(w[i], &o[i * Convert<BITS, false>::kOut], p.nibble_mul, p.minus_one);
#pragma unroll
        for (int q8 = 0; q8 < Convert<BITS, false>::kOut / 2; ++q8)  // a chunk gives 32 / BITS columns
          tmem_st_x8(tmem + lane_off + L.col_ak + c * (32 / BITS) + 8 * q8, &o[8 * q8]);
      }
      const unsigned char* vb = st + kKBytes;
#pragma unroll
      for (int hf = 0; hf < kHalves; ++hf) {
        const int r = hf * 128 + tid;  // channel row (warp-uniform test)
        if (r < D) {
#pragma unroll
          for (int c = 0; c < kVChunks; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(vb + ((size_t)c * D + r) * 16);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              Convert<BITS, false>::run(w[i], &o[i * Convert<BITS, false>::kOut], p.nibble_mul, p.minus_one);
#pragma unroll
            for (int q8 = 0; q8 < Convert<BITS, false>::kOut / 2; ++q8)
              tmem_st_x8(tmem + lane_off + L.col_av + 32 * hf + c * (32 / BITS) + 8 * q8, &o[8 * q8]);
          }
        }
      }
      tc_wait_st();
    }

    // ---- channel-wise K: Q'_g = q * s_g per token group g, and q . z_g
    if (KCW) {
      if (tid < 16) cgs[tid] = 0.f;
      if (tid < 4) eg[tid] = 0u;
      __syncthreads();
      for (int g = 0; g < ngt; ++g) {  // largest scale (fp16 bits of non-negative values order as integers)
        uint32_t mx = 0u;
        for (int c = tid; c < D; c += kGenThreads) mx = max(mx, (uint32_t)ksz[g * D + c]);
        mx = __reduce_max_sync(FULL, mx);
        if (lane == 0) atomicMax(&eg[g], mx);
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < kQv; ++i) {
        const int c = tid + 128 * i;  // warp-uniform test
        if (c < D) {
          for (int g = 0; g < ngt; ++g) {
            const float f = h2f(ksz[g * D + c]) * pow2_group(f16_exp_field(eg[g])) * odd_quarter<BITS, false>(c);
            const float4 v = make_float4(qv[0][i] * pow2_head(qmax[0]) * f, qv[1][i] * pow2_head(qmax[1]) * f,
                                         qv[2][i] * pow2_head(qmax[2]) * f, qv[3][i] * pow2_head(qmax[3]) * f);
            *reinterpret_cast<uint4*>(qop + b_off(a_pos<BITS, false>(c), g, ngt)) = split3_e4m3(v);
            const float zgc = h2f(kzz[g * D + c]);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float t = warp_sum(qv[h][i] * zgc);
              if (lane == 0) atomicAdd(&cgs[g * 4 + h], t);
            }
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
      const int nbq = KCW ? ngt : 1;
      const uint32_t idesc_q = make_idesc(0, 0, 0, 1, 128, 16 * nbq);
#pragma unroll
      for (int k = 0; k < D / 32; ++k) {
        const uint64_t bd = make_smem_desc(smem_u32(qop) + k * 4 * nbq * 128, nbq * 128, 128);
        const uint32_t a = tmem + L.col_ak + 8 * k;
        if (KCW) {
          mma_f8f6f4_ts(tmem + L.col_s, a, bd, idesc_q, k > 0);
        } else {  // the K-steps of channel group g accumulate into S block g
          mma_f8f6f4_ts(tmem + L.col_s + 16 * ((32 * k) / G), a, bd, idesc_q, (32 * k) % G != 0);
        }
      }
      tc_commit(&bars[2]);
    }
    if (!cta_wait(&bars[2], mma_phase, ok_flag, limit)) { ok = false; break; }
    mma_phase ^= 1u;
    tc_fence_after();

    // ---- scores of token l (log2 units), folded per group
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    if (KCW) {
      const int g = l / G;  // warp-uniform (G >= 32)
      uint32_t v[12];
      ld_block(tmem + lane_off + L.col_s + 16 * g, v);
      const float fs = pow2_group_inv(f16_exp_field(eg[g]));
#pragma unroll
      for (int h = 0; h < 4; ++h) sc[h] = fmaf(parts3(v, h), mult[h] * fs, cgs[g * 4 + h] * p.sm_scale_log2);
    } else {
      for (int g = 0; g < ngc; ++g) {
        uint32_t v[12];
        ld_block(tmem + lane_off + L.col_s + 16 * g, v);
        const float s_lg = h2f(ksz[l * ngc + g]), z_lg = h2f(kzz[l * ngc + g]);
#pragma unroll
        for (int h = 0; h < 4; ++h) sc[h] += fmaf(parts3(v, h) * mult[h], s_lg, z_lg * qsz[g][h]);
      }
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) sc[h] = valid ? sc[h] : -INFINITY;

    // ---- online softmax over the block (every thread holds the per-head state)
    float bmax[4] = {sc[0], sc[1], sc[2], sc[3]};
    block_reduce4(bmax, red, true);
    int e_v = 0;  // exponent of the block's largest V scale (token-wise V)
    if (!VCW) {
      float vmax = 0.f;
      if (valid)
        for (int g = 0; g < ngc; ++g) vmax = fmaxf(vmax, h2f(vsz[l * ngc + g]));
      float t4[4] = {vmax, 0.f, 0.f, 0.f};
      block_reduce4(t4, red, true);
      e_v = (int)((__float_as_uint(t4[0]) >> 23) & 0xffu) - 127;
    }
    float alpha[4], pr[4];
    int pe[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float mn = fmaxf(m_run[h], bmax[h]);
      alpha[h] = ex2(m_run[h] - mn);
      m_run[h] = mn;
      pr[h] = valid ? ex2(sc[h] - mn) : 0.f;
      pe[h] = p_exponent(bmax[h] - mn, e_v);  // P' prescale 2^(6 - E)
    }
    float psum[4] = {pr[0], pr[1], pr[2], pr[3]};
    block_reduce4(psum, red, false);
#pragma unroll
    for (int h = 0; h < 4; ++h) l_run[h] = fmaf(l_run[h], alpha[h], psum[h]);

    // per-group sums: token-wise V: sum_l p_l z_(l,g) per channel group;
    // channel-wise V: sum_(l in g) p_l per token group
    if (tid < 32) gsum[tid] = 0.f;
    __syncthreads();
    if (!VCW) {
      for (int g = 0; g < ngc; ++g) {
        const float z_lg = valid ? h2f(vzz[l * ngc + g]) : 0.f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float t = warp_sum(pr[h] * z_lg);
          if (lane == 0) atomicAdd(&gsum[g * 4 + h], t);
        }
      }
    } else {
      const int g = l / G;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float t = warp_sum(pr[h]);
        if (lane == 0) atomicAdd(&gsum[g * 4 + h], t);
      }
    }

    // ---- P' operand: row a_pos(l), one 16-column block per channel group (token-wise V)
    {
      const int nbp = VCW ? 1 : ngc;
      const float oq = odd_quarter<BITS, false>(l);
      float ps[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) ps[h] = pr[h] * oq * __uint_as_float((uint32_t)(133 - pe[h]) << 23);
      for (int g = 0; g < nbp; ++g) {
        const float sv = VCW ? 1.0f : (valid ? h2f(vsz[l * ngc + g]) : 0.f);
        const float4 v = make_float4(ps[0] * sv, ps[1] * sv, ps[2] * sv, ps[3] * sv);
        *reinterpret_cast<uint4*>(pop + b_off(a_pos<BITS, false>(l), g, nbp)) = split3_e4m3_via_f16(v);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!VCW && tid < 32 && (tid >> 2) < ngc) zrun[tid] = fmaf(zrun[tid], alpha[tid & 3], gsum[tid]);

    // ---- PV: O[channel][column block] for each M = 128 half of the channels
    if (tid == 0) {
#pragma unroll
      for (int hf = 0; hf < kHalves; ++hf) {
        const uint32_t o = tmem + L.col_o + hf * 16 * (VCW ? ngt : ngc);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t a = tmem + L.col_av + 32 * hf + 8 * k;
          if (VCW) {  // the K-steps of token group g accumulate into O block g
            const uint64_t bd = make_smem_desc(smem_u32(pop) + k * 4 * 128, 128, 128);
            mma_f8f6f4_ts(o + 16 * ((32 * k) / G), a, bd, make_idesc(0, 0, 0, 1, 128, 16), (32 * k) % G != 0);
          } else {
            const uint64_t bd = make_smem_desc(smem_u32(pop) + k * 4 * ngc * 128, ngc * 128, 128);
            mma_f8f6f4_ts(o, a, bd, make_idesc(0, 0, 0, 1, 128, 16 * ngc), k > 0);
          }
        }
      }
      tc_commit(&bars[2]);
    }
    if (!cta_wait(&bars[2], mma_phase, ok_flag, limit)) { ok = false; break; }
    mma_phase ^= 1u;
    tc_fence_after();

    // ---- epilogue: channel c = 128 hf + tid; undo the P' prescale, fold V, accumulate
    float pinv[4];  // 2^(E - 6) * 2^9 (the codes' E4M3 scale)
#pragma unroll
    for (int h = 0; h < 4; ++h) pinv[h] = __uint_as_float((uint32_t)(130 + pe[h]) << 23);
#pragma unroll
    for (int hf = 0; hf < kHalves; ++hf) {
      const int c = hf * 128 + tid;
      const uint32_t o = tmem + lane_off + L.col_o + hf * 16 * (VCW ? ngt : ngc);
      float add[4] = {0.f, 0.f, 0.f, 0.f};
      if (VCW) {
        for (int g = 0; g < ngt; ++g) {
          uint32_t v[12];
          ld_block(o + 16 * g, v);
          if (g * G >= nv || c >= D) continue;  // no valid token in this group / no such channel
          const float s_gc = h2f(vsz[g * D + c]), z_gc = h2f(vzz[g * D + c]);
#pragma unroll
          for (int h = 0; h < 4; ++h) add[h] += fmaf(s_gc, parts3(v, h) * pinv[h], z_gc * gsum[g * 4 + h]);
        }
      } else {
        uint32_t v[12];
        ld_block(o + 16 * ((c < D ? c : 0) / G), v);  // warp-uniform group (G >= 32)
#pragma unroll
        for (int h = 0; h < 4; ++h) add[h] = parts3(v, h) * pinv[h];
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) oacc[hf][h] = fmaf(oacc[hf][h], alpha[h], add[h]);
    }
    tc_fence_before();
    __syncthreads();  // stage s, Q', P', S and O are free again
    if (tid == 0) {
      pend[s] = -1;
      if (j + 2 < j1) load(j + 2, s);
    }
  }

  // ---- this range's part: O / l and lse = m + ln l per head
  if (ok) {
#pragma unroll
    for (int hf = 0; hf < kHalves; ++hf) {
      const int c = hf * 128 + tid;
      if (c < D) {
        for (int k = 0; k < p.gq; ++k) {
          const float z = VCW ? 0.f : zrun[(c / G) * 4 + k];
          p.part_o[((row0 + k) * p.splits + split) * D + c] = (oacc[hf][k] + z) / l_run[k];
        }
      }
    }
    if (tid < p.gq)
      p.part_lse[(row0 + tid) * p.splits + split] = (m_run[tid] + __log2f(l_run[tid])) * 0.69314718055994530942f;
  } else if (tid == 0) {
    report(p.dev_status, KVQ_DEV_TIMEOUT);
  }
  // leave no copy or MMA in flight: wait (bounded) for both, then release tensor memory
  if (tid == 0) {
    for (int s = 0; s < 2; ++s)
      if (pend[s] >= 0) (void)mbar_wait_bounded(&bars[s], (uint32_t)((pend[s] - j0) >> 1) & 1u, nullptr, limit);
    tc_commit(&bars[3]);
    (void)mbar_wait_bounded(&bars[3], 0u, nullptr, limit);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)L.tmem_cols);
  }
}

template <int BITS, bool KCW, bool VCW, int D>
cudaError_t launch_instance(const GenParams& p, int grid, size_t smem, cudaStream_t stream) {
  auto kern = decode_general_kernel<BITS, KCW, VCW, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kGenThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int BITS, int D>
cudaError_t launch_d(bool kcw, bool vcw, const GenParams& p, int grid, size_t smem, cudaStream_t s) {
  if (!kcw && !vcw) return launch_instance<BITS, false, false, D>(p, grid, smem, s);
  if (!kcw && vcw) return launch_instance<BITS, false, true, D>(p, grid, smem, s);
  if (kcw && !vcw) return launch_instance<BITS, true, false, D>(p, grid, smem, s);
  return launch_instance<BITS, true, true, D>(p, grid, smem, s);
}

}  // namespace

GenLaunch general_launch_shape(int bits, int k_scheme, int v_scheme, int head_dim, int group, int smem_per_sm,
                               int smem_reserved_per_cta) {
  const GenLayout L = gen_layout(bits, head_dim, group, k_scheme == KVQ_CHANNELWISE, v_scheme == KVQ_CHANNELWISE);
  GenLaunch r;
  r.ctas_per_sm = 512 / L.tmem_cols;
  if (r.ctas_per_sm > 4) r.ctas_per_sm = 4;
  // pad shared memory so that no more CTAs fit on an SM than tensor memory holds
  const long long cap = (long long)smem_per_sm / (r.ctas_per_sm + 1) - smem_reserved_per_cta + 16;
  r.smem = (size_t)((long long)L.total_bytes > cap ? (long long)L.total_bytes : cap);
  while (r.ctas_per_sm > 1 && (long long)r.ctas_per_sm * ((long long)r.smem + smem_reserved_per_cta) > smem_per_sm)
    --r.ctas_per_sm;
  return r;
}

cudaError_t launch_decode_general(int bits, int k_scheme, int v_scheme, int head_dim, const GenParams& p,
                                  int grid, size_t smem, cudaStream_t s) {
  const bool kcw = k_scheme == KVQ_CHANNELWISE, vcw = v_scheme == KVQ_CHANNELWISE;
  if (bits == 4) {
    if (head_dim == 64) return launch_d<4, 64>(kcw, vcw, p, grid, smem, s);
    if (head_dim == 128) return launch_d<4, 128>(kcw, vcw, p, grid, smem, s);
    return launch_d<4, 256>(kcw, vcw, p, grid, smem, s);
  }
  if (head_dim == 64) return launch_d<2, 64>(kcw, vcw, p, grid, smem, s);
  if (head_dim == 128) return launch_d<2, 128>(kcw, vcw, p, grid, smem, s);
  return launch_d<2, 256>(kcw, vcw, p, grid, smem, s);
}

}  // namespace kvq
