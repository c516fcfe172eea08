// Launch shape and dispatch of the general-geometry decode kernel
// (decode_general.cuh); its instances are compiled per head dim, operand
// type and heads per unit in decode_general_d{64,128,256}[_bf16][_h8].cu.
#include "decode_general.h"

namespace kvq {

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
  const int tmem_cols = gen_layout(bits, head_dim, group, kcw, vcw, bf16, nh, 2).tmem_cols;
  GenLaunch r;
  r.ctas_per_sm = 512 / tmem_cols < 4 ? 512 / tmem_cols : 4;
  if (nh > 4 && r.ctas_per_sm > 2) r.ctas_per_sm = 2;  // the 8-head instances take up to 255 registers
  auto fits = [&](int ctas, int stages) {
    const long long need =
        gen_layout(bits, head_dim, group, kcw, vcw, bf16, nh, stages).total_bytes + smem_reserved_per_cta;
    return (long long)ctas * need <= smem_per_sm && need <= 227 * 1024;
  };
  // deepest copy ring (4 stages at most) that keeps the CTAs tensor memory allows
  for (;;) {
    r.stages = 0;
    for (int st = 4; st >= 2; --st)
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
