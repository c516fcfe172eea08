// Split-KV log-sum-exp merge of partial attention results.
//
// Partial results over disjoint token ranges, each normalised over its own
// range, combine exactly: lse = ln sum_s exp(lse_s) and
// out = sum_s exp(lse_s - lse) * o_s.  An empty part carries lse = -inf and
// weight 0; a row whose parts are all empty yields out = 0, lse = -inf.
// One warp per row, float4 accesses along head_dim.
#include <cstdint>

#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) merge_kernel(const float* __restrict__ o_parts,
                                                            const float* __restrict__ lse_parts, int rows,
                                                            int splits, int head_dim, float* __restrict__ out,
                                                            float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const float* lp = lse_parts + (size_t)row * splits;
  float m = -INFINITY;
  for (int s = lane; s < splits; s += 32) m = fmaxf(m, lp[s]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float tot = 0.0f;
  for (int s = lane; s < splits; s += 32) tot += (m == -INFINITY) ? 0.0f : expf(lp[s] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  const float inv = (m == -INFINITY) ? 0.0f : 1.0f / tot;
  const float* op = o_parts + (size_t)row * splits * head_dim;
  float* dst = out + (size_t)row * head_dim;
  for (int d = lane * 4; d < head_dim; d += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < splits; ++s) {
      float l = lp[s];
      if (l == -INFINITY) continue;
      float w = expf(l - m) * inv;
      float4 v = *reinterpret_cast<const float4*>(op + (size_t)s * head_dim + d);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    *reinterpret_cast<float4*>(dst + d) = acc;
  }
  if (lane == 0) lse[row] = (m == -INFINITY) ? -INFINITY : m + logf(tot);
}

}  // namespace

cudaError_t launch_merge(const float* o_parts, const float* lse_parts, int rows, int splits, int head_dim, float* out,
                         float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  merge_kernel<<<(rows + kWarps - 1) / kWarps, kWarps * 32, 0, stream>>>(o_parts, lse_parts, rows, splits, head_dim,
                                                                         out, lse);
  return cudaGetLastError();
}

}  // namespace kvq
