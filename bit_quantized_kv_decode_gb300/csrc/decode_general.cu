// Launch shape and dispatch of the general-geometry decode kernel
// (decode_general.cuh); its instances are compiled per head dim, operand
// type and heads per unit in decode_general_d{64,128,256}[_bf16][_h8].cu.
#include "decode_general.cuh"

namespace kvq {

namespace {

// The plan of a call: every CTA of 1024 threads (a thread per sequence)
// computes gen_plan in its own shared memory -- a few microseconds, no
// exchange between CTAs -- and writes the assignments of its own 1024 decode
// CTAs; the first CTA also writes the prefix and reports bad lengths.
constexpr int kPlanThreads = 1024;
constexpr int kPlanMaxCtas = 64;  // more decode CTAs than 64 x 1024: the CTAs loop

__global__ void __launch_bounds__(kPlanThreads) general_plan_kernel(const GenParams p, long long grid, int4* assign,
                                                                    int* plan_ps) {
  __shared__ int ps[kGenPlanInts];
  __shared__ long long red[kPlanThreads / 32];
  int* lens = ps + p.batch + 1;
  gen::grid_dep_launch();  // the decode kernel may launch now; it waits for this grid before reading the plan
  gen::gen_plan<kPlanThreads>(p.seq_lens, p.batch, p.max_blocks, p.units_per_seq, p.n_target, p.n_floor, ps, lens,
                              red);
  const int tid = threadIdx.x;
  if (blockIdx.x == 0) {
    for (int b = tid; b < p.batch; b += kPlanThreads) {
      const int len = p.seq_lens[b];
      if (len < 0 || len > p.max_blocks * kBlockTokens) report(p.dev_status, KVQ_DEV_BAD_SEQ_LEN);
    }
    for (int b = tid; b <= p.batch; b += kPlanThreads) plan_ps[b] = ps[b];
  }
  const long long step = (long long)gridDim.x * kPlanThreads;
  for (long long c = (long long)blockIdx.x * kPlanThreads + tid; c < grid; c += step) {
    int4 a = make_int4(-1, 0, 0, 0);
    if (c < ps[p.batch]) {
      const int b = gen::gen_find(ps, p.batch, (int)c);
      const int nr = (ps[b + 1] - ps[b]) / p.units_per_seq;  // ranges per unit of sequence b
      const int uh = ((int)c - ps[b]) / nr, split = ((int)c - ps[b]) % nr;
      const int nblk = (lens[b] + kBlockTokens - 1) / kBlockTokens;
      a = make_int4(b | (uh << 16), (int)((long long)split * nblk / nr), (int)((long long)(split + 1) * nblk / nr),
                    lens[b]);
    }
    assign[c] = a;
  }
}

// Log-sum-exp merge of the general kernel's parts: one warp per (sequence,
// query head) row; the row's parts are the slots of its unit's ranges, from
// the plan's prefix.
constexpr int kMergeThreads = 256;

__global__ void __launch_bounds__(kMergeThreads) general_merge_kernel(const GenParams p, int head_dim, float* out,
                                                                      float* lse) {
  gen::grid_dep_wait();  // the decode kernel's parts (this kernel may start while it finishes)
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
  if (row >= p.batch * p.num_q_heads) return;
  const int b = row / p.num_q_heads, head = row % p.num_q_heads;
  const int uh = head / p.gq, k = head % p.gq;
  const int p0 = p.plan_ps[b], p1 = p.plan_ps[b + 1];
  const int nr = (p1 - p0) / p.units_per_seq;  // ranges (parts) of the row's unit
  const int c0 = p0 + uh * nr;
  float* dst = out + (size_t)row * head_dim;
  if (nr <= 32) {  // one part per lane: its weight computed once, broadcast by shuffles
    const float ls = lane < nr ? p.part_lse[(size_t)(c0 + lane) * p.gq + k] : -INFINITY;
    float m = ls;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
    const float e = lane < nr ? expf(ls - m) : 0.f;
    float tot = e;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
    const float w = nr > 0 ? e / tot : 0.f;
    for (int d = lane * 4; d < head_dim; d += 128) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int s = 0; s < nr; ++s) {
        const float ws = __shfl_sync(FULL, w, s);
        const float4 v = *reinterpret_cast<const float4*>(p.part_o + ((size_t)(c0 + s) * p.gq + k) * head_dim + d);
        acc.x = fmaf(ws, v.x, acc.x);
        acc.y = fmaf(ws, v.y, acc.y);
        acc.z = fmaf(ws, v.z, acc.z);
        acc.w = fmaf(ws, v.w, acc.w);
      }
      *reinterpret_cast<float4*>(dst + d) = acc;
    }
    if (lane == 0) lse[row] = nr > 0 ? m + logf(tot) : -INFINITY;
    return;
  }
  float m = -INFINITY;
  for (int s = lane; s < nr; s += 32) m = fmaxf(m, p.part_lse[(size_t)(c0 + s) * p.gq + k]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
  float tot = 0.f;
  for (int s = lane; s < nr; s += 32) tot += expf(p.part_lse[(size_t)(c0 + s) * p.gq + k] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(FULL, tot, o);
  const float inv = 1.0f / tot;
  for (int d = lane * 4; d < head_dim; d += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < nr; ++s) {
      const float w = expf(p.part_lse[(size_t)(c0 + s) * p.gq + k] - m) * inv;
      const float4 v = *reinterpret_cast<const float4*>(p.part_o + ((size_t)(c0 + s) * p.gq + k) * head_dim + d);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    *reinterpret_cast<float4*>(dst + d) = acc;
  }
  if (lane == 0) lse[row] = nr > 0 ? m + logf(tot) : -INFINITY;
}

}  // namespace

cudaError_t launch_general_plan(const GenParams& p, long long grid, int4* assign, int* plan_ps, cudaStream_t stream) {
  const long long ctas = (grid + kPlanThreads - 1) / kPlanThreads;
  general_plan_kernel<<<(int)(ctas < 1 ? 1 : (ctas > kPlanMaxCtas ? kPlanMaxCtas : ctas)), kPlanThreads, 0, stream>>>(
      p, grid, assign, plan_ps);
  return cudaGetLastError();
}

cudaError_t launch_general_merge(const GenParams& p, int head_dim, float* out, float* lse, cudaStream_t stream) {
  const int rows = p.batch * p.num_q_heads;
  if (rows == 0) return cudaSuccess;
  constexpr int kRows = kMergeThreads / 32;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + kRows - 1) / kRows));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_instance
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, general_merge_kernel, p, head_dim, out, lse);
}

cudaError_t launch_general_d64(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                               const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d64_h8(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                  const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d64_bf16(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                    const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d64_bf16_h8(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                       const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d128(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d128_h8(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                   const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d128_bf16(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                     const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d128_bf16_h8(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                        const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d256(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d256_h8(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                   const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d256_bf16(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                     const GenLaunch& shape, cudaStream_t s);
cudaError_t launch_general_d256_bf16_h8(int bits, bool kcw, bool vcw, int group, const GenParams& p, int grid,
                                        const GenLaunch& shape, cudaStream_t s);

GenLaunch general_launch_shape(int bits, int k_scheme, int v_scheme, int head_dim, int group, bool bf16, int nh,
                               int smem_per_sm, int smem_reserved_per_cta) {
  const bool kcw = k_scheme == KVQ_CHANNELWISE, vcw = v_scheme == KVQ_CHANNELWISE;
  GenLaunch r;
  r.ctas_per_sm = gen_ctas_per_sm(bits, head_dim, group, kcw, vcw, bf16, nh);
  auto fits = [&](int ctas, int stages) {
    const long long need =
        gen_layout(bits, head_dim, group, kcw, vcw, bf16, nh, stages).total_bytes + smem_reserved_per_cta;
    return (long long)ctas * need <= smem_per_sm && need <= 227 * 1024;
  };
  // deepest copy ring (4 stages at most) that keeps the CTAs tensor memory allows
  for (;;) {
    r.stages = 0;
    for (int st = 4; st >= (gen_single_stage(bits, head_dim, group, kcw, vcw, bf16, nh) ? 1 : 2); --st)
      if (fits(r.ctas_per_sm, st)) { r.stages = st; break; }
    if (r.stages != 0 || r.ctas_per_sm == 1) break;
    --r.ctas_per_sm;
  }
  if (r.stages == 0) r.stages = 2;
  const long long total = gen_layout(bits, head_dim, group, kcw, vcw, bf16, nh, r.stages).total_bytes;
  // pad shared memory so that no more CTAs fit on an SM than tensor memory holds
  const long long cap = (long long)smem_per_sm / (r.ctas_per_sm + 1) - smem_reserved_per_cta + 16;
  r.smem = (size_t)(total > cap ? total : cap);
  return r;
}

cudaError_t launch_decode_general(int bits, int k_scheme, int v_scheme, int head_dim, int group, bool bf16, int nh,
                                  const GenParams& p, int grid, const GenLaunch& shape, cudaStream_t s) {
  const bool kcw = k_scheme == KVQ_CHANNELWISE, vcw = v_scheme == KVQ_CHANNELWISE;
  if (head_dim == 64) {
    if (!bf16 && nh <= 4) return launch_general_d64(bits, kcw, vcw, group, p, grid, shape, s);
    if (!bf16 && nh > 4) return launch_general_d64_h8(bits, kcw, vcw, group, p, grid, shape, s);
    if (bf16 && nh <= 4) return launch_general_d64_bf16(bits, kcw, vcw, group, p, grid, shape, s);
    if (bf16 && nh > 4) return launch_general_d64_bf16_h8(bits, kcw, vcw, group, p, grid, shape, s);
  }
  if (head_dim == 128) {
    if (!bf16 && nh <= 4) return launch_general_d128(bits, kcw, vcw, group, p, grid, shape, s);
    if (!bf16 && nh > 4) return launch_general_d128_h8(bits, kcw, vcw, group, p, grid, shape, s);
    if (bf16 && nh <= 4) return launch_general_d128_bf16(bits, kcw, vcw, group, p, grid, shape, s);
    if (bf16 && nh > 4) return launch_general_d128_bf16_h8(bits, kcw, vcw, group, p, grid, shape, s);
  }
  if (head_dim == 256) {
    if (!bf16 && nh <= 4) return launch_general_d256(bits, kcw, vcw, group, p, grid, shape, s);
    if (!bf16 && nh > 4) return launch_general_d256_h8(bits, kcw, vcw, group, p, grid, shape, s);
    if (bf16 && nh <= 4) return launch_general_d256_bf16(bits, kcw, vcw, group, p, grid, shape, s);
    if (bf16 && nh > 4) return launch_general_d256_bf16_h8(bits, kcw, vcw, group, p, grid, shape, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
