// Quantize + pack (and the inverse, dequantize) of one K or V cache.
//
// One CTA per (block j, KV head h, sequence b).  The block's 128 x D fp32
// tile (D = head dim: 64, 128 or 256) is staged in shared memory; groups are
// G consecutive channels of a token (token-wise) or G consecutive tokens of
// a channel (channel-wise), G = 32, 64 or 128.  Each group's min/max gives its scale s and
// offset z (asymmetric quantization, rag-lover.com summary of arXiv
// 2611.09722, section "使える条件"), codes are computed with IEEE fp32
// subtract/divide and round-half-even, and the block is written in the packed
// chunk-major layout described in kvq.h.  The arithmetic is bit-for-bit the
// library's quantizer rule: z = fp16 round-down of the minimum,
// s = fp16 round-up of fp32((max - z) / (2^b - 1)),
// code = clamp(rint(fp32(fp32(x - z) / s)), 0, 2^b - 1).
#include <cuda_fp16.h>

#include <cstdint>

#include "kvq_internal.h"

namespace kvq {

namespace {

constexpr int kThreads = 256;

struct GroupQ {
  float s, z;
  uint16_t s_bits, z_bits;
  bool ok;
};

// Scale and offset of a group with minimum mn and maximum mx (finite).
__device__ __forceinline__ GroupQ group_params(float mn, float mx, int qmax) {
  GroupQ g;
  __half zh = __float2half_rd(mn);
  float z = __half2float(zh);
  float rng = __fsub_rn(mx, z);
  __half sh = __float2half_rn(0.0f);
  if (rng != 0.0f) sh = __float2half_ru(__fdiv_rn(rng, (float)qmax));
  g.ok = !__hisinf(zh) && !__hisinf(sh);
  g.s = __half2float(sh);
  g.z = z;
  g.s_bits = __half_as_ushort(sh);
  g.z_bits = __half_as_ushort(zh);
  return g;
}

__device__ __forceinline__ uint32_t quantize_one(float x, const GroupQ& g, int qmax) {
  if (g.s == 0.0f) return 0u;
  float t = __fdiv_rn(__fsub_rn(x, g.z), g.s);
  t = rintf(t);
  t = fminf(fmaxf(t, 0.0f), (float)qmax);
  return (uint32_t)t;
}

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Resolve the block's page and valid token count; false = nothing to do.
__device__ __forceinline__ bool block_geometry(const PackParams& p, int b, int j, int* page, int* nv) {
  int len = p.seq_lens ? p.seq_lens[b] : p.max_seq_len;
  if (len < 0 || len > p.max_seq_len) {
    if (j == 0 && blockIdx.y == 0 && threadIdx.x == 0) report(p.dev_status, KVQ_DEV_BAD_SEQ_LEN);
    return false;
  }
  if (j * kBlockTokens >= len) return false;
  int pg = p.page_table ? p.page_table[(size_t)b * p.max_blocks + j] : b * p.max_blocks + j;
  if (pg < 0 || pg >= p.num_pages) {
    if (blockIdx.y == 0 && threadIdx.x == 0) report(p.dev_status, KVQ_DEV_BAD_PAGE);
    return false;
  }
  *page = pg;
  *nv = min(kBlockTokens, len - j * kBlockTokens);
  return true;
}

// Quantize and pack one block of KV head h: the nv valid token rows at src
// (fp32, D channels each) into page `page`.  s / z of a block: token-wise,
// entry t * (D / G) + g for channels [gG, gG + G) of token t; channel-wise,
// entry k * D + c for channel c over block tokens [kG, kG + G).
__device__ void pack_block(const PackParams& p, const float* src, int page, int nv, int h, unsigned char* smem_raw) {
  const int D = p.head_dim, G = p.group, pitch = D + 1;
  float* xs = reinterpret_cast<float*>(smem_raw);                                    // [128][D + 1]
  uint8_t* cs = reinterpret_cast<uint8_t*>(xs + kBlockTokens * pitch);              // [128 tok][D ch]
  uint16_t* s_out = reinterpret_cast<uint16_t*>(cs + kBlockTokens * D);             // [128 * D / G]
  uint16_t* z_out = s_out + kBlockTokens * D / G;                                   // [128 * D / G]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qmax = (1 << p.bits) - 1;
  const int nsz = kBlockTokens * D / G;

  // Stage the valid tokens of the tile (rows t < nv).
  for (int i = tid; i < nv * (D / 4); i += kThreads) {
    int t = i / (D / 4), c4 = (i % (D / 4)) * 4;
    float4 v = *reinterpret_cast<const float4*>(src + (size_t)t * D + c4);
    float* row = xs + t * pitch + c4;
    row[0] = v.x; row[1] = v.y; row[2] = v.z; row[3] = v.w;
  }
  for (int i = tid; i < kBlockTokens * D / 4; i += kThreads) reinterpret_cast<uint32_t*>(cs)[i] = 0u;
  for (int i = tid; i < nsz; i += kThreads) { s_out[i] = 0; z_out[i] = 0; }  // groups without valid values
  __syncthreads();

  const bool tokenwise = (p.which == 0 ? p.k_scheme : p.v_scheme) == KVQ_TOKENWISE;
  if (tokenwise) {
    // groups of G channels of token t; one warp per token, lane holds channels lane + 32 k
    const int gpt = D / G, kpg = G / 32;  // groups per token, 32-channel slices per group
    for (int t = warp; t < nv; t += kThreads / 32) {
      for (int g = 0; g < gpt; ++g) {
        float v[4];
        bool fin = true;
        float mn = INFINITY, mx = -INFINITY;
        for (int k = 0; k < kpg; ++k) {
          v[k] = xs[t * pitch + g * G + lane + 32 * k];
          fin &= isfinite(v[k]);
          mn = fminf(mn, v[k]);
          mx = fmaxf(mx, v[k]);
        }
        fin = __all_sync(0xffffffffu, fin);
        mn = warp_min(mn);
        mx = warp_max(mx);
        GroupQ q = fin ? group_params(mn, mx, qmax) : GroupQ{0.f, 0.f, 0, 0, false};
        if (!q.ok) {
          if (lane == 0) report(p.dev_status, KVQ_DEV_NONFINITE);  // group left as zeros
          continue;
        }
        for (int k = 0; k < kpg; ++k) cs[t * D + g * G + lane + 32 * k] = (uint8_t)quantize_one(v[k], q, qmax);
        if (lane == 0) { s_out[t * gpt + g] = q.s_bits; z_out[t * gpt + g] = q.z_bits; }
      }
    }
  } else {
    // groups of G tokens of channel c (aligned to the block); one warp per channel
    const int gpb = kBlockTokens / G;
    for (int c = warp; c < D; c += kThreads / 32) {
      for (int g = 0; g < gpb; ++g) {
        const int t0 = g * G, t1 = min(nv, t0 + G);
        if (t1 <= t0) break;  // no valid token in this group or the later ones: s = z = 0
        float mn = INFINITY, mx = -INFINITY;
        bool fin = true;
        for (int t = t0 + lane; t < t1; t += 32) {
          float v = xs[t * pitch + c];
          fin &= isfinite(v);
          mn = fminf(mn, v);
          mx = fmaxf(mx, v);
        }
        fin = __all_sync(0xffffffffu, fin);
        mn = warp_min(mn);
        mx = warp_max(mx);
        GroupQ q = fin ? group_params(mn, mx, qmax) : GroupQ{0.f, 0.f, 0, 0, false};
        if (!q.ok) {
          if (lane == 0) report(p.dev_status, KVQ_DEV_NONFINITE);
          continue;
        }
        for (int t = t0 + lane; t < t1; t += 32) cs[t * D + c] = (uint8_t)quantize_one(xs[t * pitch + c], q, qmax);
        if (lane == 0) { s_out[g * D + c] = q.s_bits; z_out[g * D + c] = q.z_bits; }
      }
    }
  }
  __syncthreads();

  // Pack: K rows are tokens (D columns), V rows are channels (128 columns);
  // row r, chunk k holds columns [k*per_chunk, (k+1)*per_chunk).
  const int bits = p.bits;
  const int per_chunk = 128 / bits;  // columns per 16-byte chunk: 32 (INT4) or 64 (INT2)
  const int nrows = p.which == 0 ? kBlockTokens : D, ncols = p.which == 0 ? D : kBlockTokens;
  const int nchunk = ncols / per_chunk;
  const size_t blk = (size_t)page * p.num_kv_heads + h;
  uint8_t* dst = p.codes + blk * (size_t)(kBlockTokens * D * bits / 8);
  for (int i = tid; i < nchunk * nrows; i += kThreads) {
    int k = i / nrows, r = i % nrows;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int e = 0; e < per_chunk; ++e) {
      int col = k * per_chunk + e;
      // K: row = token, column = channel.  V: row = channel, column = token.
      uint32_t code = (p.which == 0) ? cs[r * D + col] : cs[col * D + r];
      int bitpos = e * bits;
      w[bitpos >> 5] |= code << (bitpos & 31);
    }
    *reinterpret_cast<uint4*>(dst + (size_t)i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  for (int i = tid; i < nsz; i += kThreads) {
    p.scale[blk * nsz + i] = s_out[i];
    p.zero[blk * nsz + i] = z_out[i];
  }
}

__global__ void __launch_bounds__(kThreads) pack_kernel(PackParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  int page, nv;
  if (!block_geometry(p, b, j, &page, &nv)) return;
  const float* src = p.x + (((size_t)b * p.num_kv_heads + h) * p.max_seq_len + (size_t)j * kBlockTokens) * p.head_dim;
  pack_block(p, src, page, nv, h, smem_raw);
}

// Append one token per sequence: the token at position len = seq_lens[b]
// goes into row len % 128 of the caller's window of the current block, and
// the block is quantized and packed again from the window's len % 128 + 1
// valid rows (the same rule as a partial last block of kvq_pack).  One CTA
// per (KV head h, sequence b).
__global__ void __launch_bounds__(kThreads) append_kernel(PackParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int h = blockIdx.x, b = blockIdx.y;
  const int len = p.seq_lens[b];
  if (len < 0 || len >= p.max_blocks * kBlockTokens) {
    if (h == 0 && threadIdx.x == 0) report(p.dev_status, KVQ_DEV_BAD_SEQ_LEN);
    return;
  }
  const int j = len / kBlockTokens, r = len % kBlockTokens;
  const int page = p.page_table ? p.page_table[(size_t)b * p.max_blocks + j] : b * p.max_blocks + j;
  if (page < 0 || page >= p.num_pages) {
    if (h == 0 && threadIdx.x == 0) report(p.dev_status, KVQ_DEV_BAD_PAGE);
    return;
  }
  const int D = p.head_dim;
  float* win = p.window + ((size_t)b * p.num_kv_heads + h) * kBlockTokens * D;
  const float* xn = p.x + ((size_t)b * p.num_kv_heads + h) * D;
  for (int c = threadIdx.x; c < D; c += kThreads) win[(size_t)r * D + c] = xn[c];
  __syncthreads();  // the new row is visible to the whole CTA
  pack_block(p, win, page, r + 1, h, smem_raw);
}

__global__ void __launch_bounds__(kThreads) dequant_kernel(DequantParams p) {
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int D = p.head_dim, G = p.group, nsz = kBlockTokens * D / G;
  float* dst = p.x_hat + (((size_t)b * p.num_kv_heads + h) * p.max_seq_len + (size_t)j * kBlockTokens) * D;
  const int ntok = min(kBlockTokens, p.max_seq_len - j * kBlockTokens);
  int len = p.seq_lens ? p.seq_lens[b] : p.max_seq_len;
  bool bad_len = len < 0 || len > p.max_seq_len;
  if (bad_len && j == 0 && h == 0 && tid == 0) report(p.dev_status, KVQ_DEV_BAD_SEQ_LEN);
  int nv = bad_len ? 0 : max(0, min(ntok, len - j * kBlockTokens));
  int page = 0;
  if (nv > 0) {
    page = p.page_table ? p.page_table[(size_t)b * p.max_blocks + j] : b * p.max_blocks + j;
    if (page < 0 || page >= p.num_pages) {
      if (h == 0 && tid == 0) report(p.dev_status, KVQ_DEV_BAD_PAGE);
      nv = 0;
    }
  }
  const bool tokenwise = (p.which == 0 ? p.k_scheme : p.v_scheme) == KVQ_TOKENWISE;
  const size_t blk = (size_t)page * p.num_kv_heads + h;
  const int bits = p.bits;
  const uint8_t* src = p.codes + blk * (size_t)(kBlockTokens * D * bits / 8);
  const uint16_t* sp = p.scale + blk * nsz;
  const uint16_t* zp = p.zero + blk * nsz;
  const int per_chunk = 128 / bits;
  const int nrows = p.which == 0 ? kBlockTokens : D;
  for (int i = tid; i < ntok * D; i += kThreads) {
    int t = i / D, c = i % D;
    float v = 0.0f;
    if (t < nv) {
      int r = (p.which == 0) ? t : c;    // row in the block
      int col = (p.which == 0) ? c : t;  // column in the row
      int k = col / per_chunk, e = col % per_chunk;
      const uint32_t* chunk = reinterpret_cast<const uint32_t*>(src + ((size_t)k * nrows + r) * 16);
      int bitpos = e * bits;
      uint32_t code = (chunk[bitpos >> 5] >> (bitpos & 31)) & ((1u << bits) - 1u);
      int g = tokenwise ? t * (D / G) + c / G : (t / G) * D + c;
      float s = __half2float(__ushort_as_half(sp[g]));
      float z = __half2float(__ushort_as_half(zp[g]));
      v = fmaf(s, (float)code, z);
    }
    dst[(size_t)t * D + c] = v;
  }
}

}  // namespace

size_t pack_smem_bytes(int head_dim, int group) {
  return (size_t)kBlockTokens * (head_dim + 1) * sizeof(float) + (size_t)kBlockTokens * head_dim +
         2 * (size_t)kBlockTokens * head_dim / group * sizeof(uint16_t);
}

cudaError_t launch_pack(const PackParams& p, cudaStream_t stream) {
  const size_t smem = pack_smem_bytes(p.head_dim, p.group);
  cudaError_t e = cudaFuncSetAttribute(pack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.max_blocks_needed, p.num_kv_heads, p.batch);
  pack_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append(const PackParams& p, cudaStream_t stream) {
  const size_t smem = pack_smem_bytes(p.head_dim, p.group);
  cudaError_t e = cudaFuncSetAttribute(append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_kv_heads, p.batch);
  append_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantParams& p, cudaStream_t stream) {
  dim3 grid((p.max_seq_len + kBlockTokens - 1) / kBlockTokens, p.num_kv_heads, p.batch);
  dequant_kernel<<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
