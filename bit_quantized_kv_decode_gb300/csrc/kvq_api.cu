// C-ABI entry points: argument validation, workspace layout and dispatch.
// Nothing here allocates memory; every launch goes to the caller's stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "decode_general.h"
#include "kvq_entry.h"

namespace kvq {
#ifdef KVQ_PROFILE
static unsigned long long* g_prof_counters = nullptr;
#endif
namespace {

constexpr int kMaxBatchDecode = 1024;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int group_of(const kvq_cache_desc* c) { return c->group_size == 0 ? 128 : c->group_size; }
int block_bytes(const kvq_cache_desc* c) { return kBlockTokens * c->head_dim * c->bits / 8; }
int sz_per_block(const kvq_cache_desc* c) { return kBlockTokens * c->head_dim / group_of(c); }

kvq_status check_cache(const kvq_cache_desc* c) {
  if (c == nullptr) return KVQ_ERR_INVALID_ARG;
  if (c->bits != 2 && c->bits != 4) return KVQ_ERR_UNSUPPORTED;
  if ((c->k_scheme != KVQ_TOKENWISE && c->k_scheme != KVQ_CHANNELWISE) ||
      (c->v_scheme != KVQ_TOKENWISE && c->v_scheme != KVQ_CHANNELWISE))
    return KVQ_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  const int g = group_of(c);
  if ((g != 32 && g != 64 && g != 128) || g > c->head_dim) return KVQ_ERR_UNSUPPORTED;
  if (c->num_kv_heads < 1 || c->num_pages < 1) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

// The specialised decode kernel's geometry; others take the general kernel.
bool default_geometry(const kvq_cache_desc* c) { return c->head_dim == kHeadDim && group_of(c) == 128; }

}  // namespace

// Checks the current device without launching anything.
kvq_status check_device(int* sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return KVQ_ERR_DEVICE; }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_DEVICE;
  }
  if (major != 10 || minor != 3) return KVQ_ERR_DEVICE;
  if (sm_count != nullptr &&
      cudaDeviceGetAttribute(sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ERR_DEVICE;
  }
  return KVQ_OK;
}

namespace {

struct WorkspaceLayout {
  size_t counters, part_lse, part_o, total;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Query heads per KV head the kernel takes (1, 2, 4 or 8; 0 otherwise) and
// the work units per sequence: a unit holds up to 4 query heads of one KV
// head, so 8 query heads per KV head make two units per KV head.
int heads_per_kv(const kvq_attn_desc* d) {
  const int hkv = d->cache.num_kv_heads;
  if (hkv < 1 || d->num_q_heads % hkv != 0) return 0;
  const int g = d->num_q_heads / hkv;
  return (g == 1 || g == 2 || g == 4 || g == 8) ? g : 0;
}
int units_per_seq(const kvq_attn_desc* d) {
  const int g = heads_per_kv(d);
  return g > kGroupQ ? d->cache.num_kv_heads * (g / kGroupQ) : d->cache.num_kv_heads;
}

// Calls the specialised kernel takes (any query heads per KV head it builds).
bool specialised_ok(const kvq_attn_desc* d) {
  return default_geometry(&d->cache) && d->operand_mode == KVQ_OPERANDS_FP8;
}
// Decode calls the block-range (general) kernel takes: every geometry but
// the default and every BF16-operand call (the specialised kernel is built
// for E4M3 operands at head dim 128, groups of 128), and on that geometry
// every call of real size -- measured faster there for every scheme pair and
// query-head count on GB300 at B = 128, L = 32K (INT4 K-cw/V-tw 74.5% of the
// HBM peak against 71.6%, INT2 K-/V-token-wise 51% against 44%, 8 query
// heads per KV head 54% against 35%) and at B = 32, L = 4K (8 heads: 15-17%
// against 13-15%).  Small calls stay in the specialised kernel, whose
// persistent CTAs start faster (10% against 7% at B = 8, L = 4K), and so do
// calls with the E2M1 V placement, which only it builds.
constexpr long long kGeneralMinBlocks = 8192;  // (sequence, unit, block) triples of max_blocks per unit
bool use_general(const kvq_attn_desc* d) {
  if (!specialised_ok(d)) return true;
  if (d->flags & KVQ_FLAG_E2M1_V) return false;
  return (long long)d->batch * units_per_seq(d) * d->max_blocks >= kGeneralMinBlocks;
}

WorkspaceLayout workspace_layout(int batch, int units, int num_ctas) {
  WorkspaceLayout w;
  w.counters = 0;
  w.part_lse = round_up((size_t)batch * units * kCounterGroups * sizeof(int), 256);
  w.part_o = w.part_lse + round_up((size_t)num_ctas * 2 * kGroupQ * sizeof(float), 256);
  w.total = w.part_o + round_up((size_t)num_ctas * 2 * kGroupQ * kHeadDim * sizeof(float), 256);
  return w;
}

kvq_status check_attn(const kvq_attn_desc* d) {
  if (d == nullptr) return KVQ_ERR_INVALID_ARG;
  kvq_status s = check_cache(&d->cache);
  if (s != KVQ_OK) return s;
  if (d->batch < 1 || d->max_blocks < 1 || d->num_q_heads < 1) return KVQ_ERR_INVALID_ARG;
  if (d->batch > kMaxBatchDecode) return KVQ_ERR_UNSUPPORTED;
  if (heads_per_kv(d) == 0) return KVQ_ERR_UNSUPPORTED;  // 1, 2, 4 or 8 query heads per KV head
  if (d->operand_mode != KVQ_OPERANDS_FP8 && d->operand_mode != KVQ_OPERANDS_BF16) return KVQ_ERR_INVALID_ARG;
  if (d->num_ctas < 0 || (d->flags & ~(KVQ_FLAG_TEST_STALL | KVQ_FLAG_TEST_STALL_MMA | KVQ_FLAG_E2M1_V)) != 0)
    return KVQ_ERR_INVALID_ARG;
  if ((d->flags & KVQ_FLAG_E2M1_V) &&
      (d->cache.bits != 2 || d->operand_mode != KVQ_OPERANDS_FP8 || heads_per_kv(d) != kGroupQ))
    return KVQ_ERR_UNSUPPORTED;  // the E2M1 placement is built for these only
  if (!default_geometry(&d->cache) && (d->flags & KVQ_FLAG_E2M1_V))
    return KVQ_ERR_UNSUPPORTED;  // the E2M1 placement is built for head dim 128, groups of 128
  if (!(std::isfinite(d->sm_scale))) return KVQ_ERR_INVALID_ARG;
  if ((long long)d->batch * units_per_seq(d) * d->max_blocks > (1LL << 30)) return KVQ_ERR_UNSUPPORTED;
  if (units_per_seq(d) >= (1 << 15)) return KVQ_ERR_UNSUPPORTED;  // the general kernel's CTA assignment packs the unit
  return KVQ_OK;
}

// General geometry: the CTA count the device-side plan aims at (gen_plan in
// decode_general.cuh cuts each sequence's units into ranges in proportion
// to its length), the launch shape and the workspace.  The target is
// units * S: with num_ctas = 0, S is chosen between one and eight waves of
// resident CTAs so that a batch of max_blocks per unit fills its last wave
// best (fewest idle CTA slots), then the fewest ranges, and the plan may aim
// lower (down to one wave) when the actual lengths hold less work; with
// num_ctas > 0, S = ceil(num_ctas / units), kept as given.  At most
// max_blocks ranges per unit.
struct GeneralPlan {
  GenLaunch launch;
  int nh;            // query heads per unit: 8 (each KV block read once) or 4
  int units;         // units per sequence
  int gq;            // query heads a unit holds
  long long n_target;
  long long n_floor;  // the fewest CTAs the plan may aim at (one wave; n_target with num_ctas > 0)
  long long slots;    // grid = part slots: n_target + every unit (one range each at least)
  size_t plan_ps, assign, part_lse, part_o, total;  // workspace offsets and size
};

kvq_status general_plan(const kvq_attn_desc* d, GeneralPlan* plan) {
  int sm = 0, smem_sm = 228 * 1024, reserved = 1024;
  if (d->num_ctas == 0) {
    kvq_status s = check_device(&sm);
    if (s != KVQ_OK) return s;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
      cudaGetLastError();
      return KVQ_ERR_DEVICE;
    }
  }
  plan->nh = heads_per_kv(d) == 8 ? 8 : 4;
  plan->units = plan->nh == 8 ? d->cache.num_kv_heads : units_per_seq(d);
  plan->launch = general_launch_shape(d->cache.bits, d->cache.k_scheme, d->cache.v_scheme, d->cache.head_dim,
                                      group_of(&d->cache), d->operand_mode == KVQ_OPERANDS_BF16, plan->nh, smem_sm,
                                      reserved);
  const long long units = (long long)d->batch * plan->units;
  const long long resident = (long long)plan->launch.ctas_per_sm * sm;
  long long splits;
  if (d->num_ctas > 0) {
    splits = (d->num_ctas + units - 1) / units;
  } else {
    const long long lo = (resident + units - 1) / units, hi = (8 * resident + units - 1) / units;
    splits = lo;
    double best = -1.0;
    for (long long s = lo; s <= hi && s <= d->max_blocks; ++s) {
      const long long ctas = units * s, waves = (ctas + resident - 1) / resident;
      const double fill = (double)ctas / (double)(waves * resident);
      if (fill > best + 1e-9) { best = fill; splits = s; }
    }
  }
  if (splits > d->max_blocks) splits = d->max_blocks;
  if (splits < 1) splits = 1;
  const int g = heads_per_kv(d);
  plan->gq = plan->nh == 8 ? 8 : (g < kGroupQ ? g : kGroupQ);
  plan->n_target = units * splits;
  plan->n_floor = d->num_ctas > 0 ? plan->n_target : resident;
  plan->slots = plan->n_target + units;
  plan->plan_ps = 0;
  plan->assign = round_up((size_t)(d->batch + 1) * sizeof(int), 256);
  plan->part_lse = plan->assign + round_up((size_t)plan->slots * 4 * sizeof(int), 256);
  plan->part_o = plan->part_lse + round_up((size_t)plan->slots * plan->gq * sizeof(float), 256);
  plan->total = plan->part_o + round_up((size_t)plan->slots * plan->gq * d->cache.head_dim * sizeof(float), 256);
  return KVQ_OK;
}

int resolve_ctas(const kvq_attn_desc* d, int sm_count) {
  long long want = d->num_ctas > 0 ? d->num_ctas : (long long)decode_ctas_per_sm() * sm_count;
  long long tiles_bound = (long long)d->batch * units_per_seq(d) * d->max_blocks;
  if (want > tiles_bound) want = tiles_bound;
  return (int)(want < 1 ? 1 : want);
}

// The general-geometry path of kvq_decode_attn (arguments already checked):
// the block-range kernel, then the log-sum-exp merge of the ranges.
kvq_status decode_general(const kvq_attn_desc* desc, const uint16_t* q, const uint8_t* k_codes,
                          const uint16_t* k_scale, const uint16_t* k_zero, const uint8_t* v_codes,
                          const uint16_t* v_scale, const uint16_t* v_zero, const int32_t* seq_lens,
                          const int32_t* page_table, float* out, float* lse, void* workspace, size_t workspace_bytes,
                          uint32_t* dev_status, float sm_scale, cudaStream_t st) {
  GeneralPlan plan;
  kvq_status s = general_plan(desc, &plan);
  if (s != KVQ_OK) return s;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KVQ_ERR_WORKSPACE;
  if (workspace_bytes < plan.total) return KVQ_ERR_WORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  GenParams p{};
  p.q = q; p.k_codes = k_codes; p.k_scale = k_scale; p.k_zero = k_zero;
  p.v_codes = v_codes; p.v_scale = v_scale; p.v_zero = v_zero;
  p.seq_lens = seq_lens; p.page_table = page_table; p.dev_status = dev_status;
  p.part_lse = reinterpret_cast<float*>(ws + plan.part_lse);
  p.part_o = reinterpret_cast<float*>(ws + plan.part_o);
  p.assign = reinterpret_cast<const int4*>(ws + plan.assign);
  p.plan_ps = reinterpret_cast<const int*>(ws + plan.plan_ps);
  p.batch = desc->batch; p.num_kv_heads = desc->cache.num_kv_heads; p.num_q_heads = desc->num_q_heads;
  p.max_blocks = desc->max_blocks; p.num_pages = desc->cache.num_pages;
  p.gq = plan.gq;
  p.units_per_seq = plan.units;
  p.kv_shift = 0;  // a unit is one KV head (up to 8 query heads)
  p.n_target = plan.n_target;
  p.n_floor = plan.n_floor;
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.flags = desc->flags;
  p.wait_limit_ns =
      (desc->flags & (KVQ_FLAG_TEST_STALL | KVQ_FLAG_TEST_STALL_MMA)) ? 50ull * 1000 * 1000 : 2ull * 1000 * 1000 * 1000;
  p.nibble_mul = 1u << 28;
  p.minus_one = 0xffffffffu;
  const int grid = (int)plan.slots;
  cudaError_t e = launch_general_plan(p, plan.slots, reinterpret_cast<int4*>(ws + plan.assign),
                                      reinterpret_cast<int*>(ws + plan.plan_ps), st);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  e = launch_decode_general(desc->cache.bits, desc->cache.k_scheme, desc->cache.v_scheme,
                                        desc->cache.head_dim, group_of(&desc->cache),
                                        desc->operand_mode == KVQ_OPERANDS_BF16, plan.nh, p, grid, plan.launch, st);
  if (e != cudaSuccess) return KVQ_ERR_CUDA;
  e = launch_general_merge(p, desc->cache.head_dim, out, lse, st);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// The kernel a checked call takes and its workspace: the general one where
// use_general says so, unless its workspace would exceed `limit` bytes and
// the specialised kernel takes the call (E4M3 operands, head dim 128, groups
// of 128), whose workspace is then the one returned.
kvq_status decode_route(const kvq_attn_desc* desc, size_t limit, bool* general, size_t* bytes) {
  kvq_status s;
  *general = use_general(desc);
  if (*general) {
    GeneralPlan plan;
    s = general_plan(desc, &plan);
    if (s != KVQ_OK) return s;
    *bytes = plan.total;
    if (plan.total <= limit || !specialised_ok(desc)) return KVQ_OK;
    *general = false;
  }
  int sm = 0;
  if (desc->num_ctas == 0) {
    s = check_device(&sm);
    if (s != KVQ_OK) return s;
  }
  const int ctas = resolve_ctas(desc, sm);
  *bytes = workspace_layout(desc->batch, units_per_seq(desc), ctas).total;
  return KVQ_OK;
}

}  // namespace

kvq_status decode_workspace_bounded(const kvq_attn_desc* desc, size_t limit, size_t* bytes) {
  kvq_status s = check_attn(desc);
  if (s != KVQ_OK) return s;
  if (bytes == nullptr) return KVQ_ERR_INVALID_ARG;
  bool general = false;
  return decode_route(desc, limit, &general, bytes);
}

kvq_status decode_attn_bounded(const kvq_attn_desc* desc, const uint16_t* q, const uint8_t* k_codes,
                               const uint16_t* k_scale, const uint16_t* k_zero, const uint8_t* v_codes,
                               const uint16_t* v_scale, const uint16_t* v_zero, const int32_t* seq_lens,
                               const int32_t* page_table, float* out, float* lse, void* workspace,
                               size_t workspace_bytes, size_t limit, uint32_t* dev_status, void* stream) {
  kvq_status s = check_attn(desc);
  if (s != KVQ_OK) return s;
  // cache arrays are read with 16-byte bulk copies; the rest with scalar accesses
  const void* bulk[] = {k_codes, k_scale, k_zero, v_codes, v_scale, v_zero};
  for (const void* ptr : bulk)
    if (ptr == nullptr || !aligned16(ptr)) return KVQ_ERR_INVALID_ARG;
  if (q == nullptr || seq_lens == nullptr || out == nullptr || lse == nullptr) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(out) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return KVQ_ERR_INVALID_ARG;
  if (page_table != nullptr && (reinterpret_cast<uintptr_t>(page_table) & 3u)) return KVQ_ERR_INVALID_ARG;
  if (page_table == nullptr && (long long)desc->batch * desc->max_blocks > desc->cache.num_pages)
    return KVQ_ERR_INVALID_ARG;
  int sm = 0;
  s = check_device(&sm);
  if (s != KVQ_OK) return s;
  bool general = false;
  size_t need = 0;
  s = decode_route(desc, limit, &general, &need);
  if (s != KVQ_OK) return s;
  const float sm_scale = desc->sm_scale > 0.0f ? desc->sm_scale : 1.0f / std::sqrt((float)desc->cache.head_dim);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (general) return decode_general(desc, q, k_codes, k_scale, k_zero, v_codes, v_scale, v_zero, seq_lens,
                                     page_table, out, lse, workspace, workspace_bytes, dev_status, sm_scale, st);
  const int ctas = resolve_ctas(desc, sm);
  const WorkspaceLayout w = workspace_layout(desc->batch, units_per_seq(desc), ctas);
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KVQ_ERR_WORKSPACE;
  if (workspace_bytes < w.total) return KVQ_ERR_WORKSPACE;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  if (cudaMemsetAsync(ws + w.counters, 0, (size_t)desc->batch * units_per_seq(desc) * kCounterGroups * sizeof(int),
                      st) !=
      cudaSuccess)
    return KVQ_ERR_CUDA;
  DecodeParams p{};
  p.q = q; p.k_codes = k_codes; p.k_scale = k_scale; p.k_zero = k_zero;
  p.v_codes = v_codes; p.v_scale = v_scale; p.v_zero = v_zero;
  p.seq_lens = seq_lens; p.page_table = page_table; p.out = out; p.lse = lse; p.dev_status = dev_status;
  p.counters = reinterpret_cast<int*>(ws + w.counters);
  p.part_lse = reinterpret_cast<float*>(ws + w.part_lse);
  p.part_o = reinterpret_cast<float*>(ws + w.part_o);
  p.batch = desc->batch; p.num_kv_heads = desc->cache.num_kv_heads; p.num_q_heads = desc->num_q_heads;
  p.max_blocks = desc->max_blocks; p.num_pages = desc->cache.num_pages; p.num_ctas = ctas;
  {
    const int g = heads_per_kv(desc);
    p.gq = g < kGroupQ ? g : kGroupQ;
    p.units_per_seq = units_per_seq(desc);
    p.kv_shift = g > kGroupQ ? 1 : 0;
  }
  p.sm_scale_log2 = sm_scale * 1.4426950408889634f;
  p.flags = desc->flags;
  p.nibble_mul = 1u << 28;
  p.minus_one = 0xffffffffu;
  p.wait_limit_ns =
      (desc->flags & (KVQ_FLAG_TEST_STALL | KVQ_FLAG_TEST_STALL_MMA)) ? 50ull * 1000 * 1000 : 2ull * 1000 * 1000 * 1000;
#ifdef KVQ_PROFILE
  p.prof = g_prof_counters;
#endif
  cudaError_t e = launch_decode(desc->cache.bits, desc->cache.k_scheme, desc->cache.v_scheme, p, st);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace kvq

using namespace kvq;

#ifdef KVQ_PROFILE
extern "C" KVQ_API void kvq_prof_set(unsigned long long* counters) { kvq::g_prof_counters = counters; }
#endif

extern "C" {

KVQ_API const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_DEVICE: return "no sm_103 device";
  }
  return "unknown status";
}

KVQ_API int32_t kvq_version(void) { return 100; }

KVQ_API kvq_status kvq_cache_bytes(const kvq_cache_desc* cache, size_t* codes_bytes, size_t* scale_bytes) {
  kvq_status s = check_cache(cache);
  if (s != KVQ_OK) return s;
  if (codes_bytes == nullptr || scale_bytes == nullptr) return KVQ_ERR_INVALID_ARG;
  const size_t blocks = (size_t)cache->num_pages * cache->num_kv_heads;
  *codes_bytes = blocks * block_bytes(cache);
  *scale_bytes = blocks * sz_per_block(cache) * sizeof(uint16_t);
  return KVQ_OK;
}

KVQ_API kvq_status kvq_pack(const kvq_cache_desc* cache, int32_t which, const float* x, int32_t batch,
                            int32_t max_seq_len, const int32_t* seq_lens, const int32_t* page_table,
                            int32_t max_blocks, uint8_t* codes, uint16_t* scale, uint16_t* zero,
                            uint32_t* dev_status, void* stream) {
  kvq_status s = check_cache(cache);
  if (s != KVQ_OK) return s;
  if (which != 0 && which != 1) return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || max_seq_len < 1 || batch > 65535) return KVQ_ERR_INVALID_ARG;
  const int need_blocks = (max_seq_len + kBlockTokens - 1) / kBlockTokens;
  if (max_blocks < need_blocks) return KVQ_ERR_INVALID_ARG;
  if (page_table == nullptr && (long long)batch * max_blocks > cache->num_pages) return KVQ_ERR_INVALID_ARG;
  if (!x || !codes || !scale || !zero || !aligned16(x) || !aligned16(codes) || !aligned16(scale) || !aligned16(zero))
    return KVQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seq_lens) & 3u) || (reinterpret_cast<uintptr_t>(page_table) & 3u))
    return KVQ_ERR_INVALID_ARG;
  s = check_device(nullptr);
  if (s != KVQ_OK) return s;
  PackParams p{};
  p.x = x; p.seq_lens = seq_lens; p.page_table = page_table;
  p.codes = codes; p.scale = scale; p.zero = zero; p.dev_status = dev_status;
  p.bits = cache->bits; p.k_scheme = cache->k_scheme; p.v_scheme = cache->v_scheme; p.which = which;
  p.head_dim = cache->head_dim; p.group = group_of(cache);
  p.num_kv_heads = cache->num_kv_heads; p.num_pages = cache->num_pages;
  p.batch = batch; p.max_seq_len = max_seq_len; p.max_blocks = max_blocks; p.max_blocks_needed = need_blocks;
  return launch_pack(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

KVQ_API kvq_status kvq_append(const kvq_cache_desc* cache, int32_t which, const float* x_new, int32_t batch,
                              const int32_t* seq_lens, const int32_t* page_table, int32_t max_blocks,
                              float* window, uint8_t* codes, uint16_t* scale, uint16_t* zero,
                              uint32_t* dev_status, void* stream) {
  kvq_status s = check_cache(cache);
  if (s != KVQ_OK) return s;
  if (which != 0 && which != 1) return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || batch > 65535 || max_blocks < 1 || cache->num_kv_heads > 65535) return KVQ_ERR_INVALID_ARG;
  if (page_table == nullptr && (long long)batch * max_blocks > cache->num_pages) return KVQ_ERR_INVALID_ARG;
  if (!x_new || !window || !seq_lens || !codes || !scale || !zero || !aligned16(x_new) || !aligned16(window) ||
      !aligned16(codes) || !aligned16(scale) || !aligned16(zero))
    return KVQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seq_lens) & 3u) || (reinterpret_cast<uintptr_t>(page_table) & 3u))
    return KVQ_ERR_INVALID_ARG;
  s = check_device(nullptr);
  if (s != KVQ_OK) return s;
  PackParams p{};
  p.x = x_new; p.window = window; p.seq_lens = seq_lens; p.page_table = page_table;
  p.codes = codes; p.scale = scale; p.zero = zero; p.dev_status = dev_status;
  p.bits = cache->bits; p.k_scheme = cache->k_scheme; p.v_scheme = cache->v_scheme; p.which = which;
  p.head_dim = cache->head_dim; p.group = group_of(cache);
  p.num_kv_heads = cache->num_kv_heads; p.num_pages = cache->num_pages;
  p.batch = batch; p.max_seq_len = max_blocks * kBlockTokens; p.max_blocks = max_blocks; p.max_blocks_needed = 1;
  return launch_append(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

KVQ_API kvq_status kvq_dequant(const kvq_cache_desc* cache, int32_t which, const uint8_t* codes,
                               const uint16_t* scale, const uint16_t* zero, int32_t batch, int32_t max_seq_len,
                               const int32_t* seq_lens, const int32_t* page_table, int32_t max_blocks,
                               float* x_hat, uint32_t* dev_status, void* stream) {
  kvq_status s = check_cache(cache);
  if (s != KVQ_OK) return s;
  if (which != 0 && which != 1) return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || max_seq_len < 1 || batch > 65535) return KVQ_ERR_INVALID_ARG;
  const int need_blocks = (max_seq_len + kBlockTokens - 1) / kBlockTokens;
  if (max_blocks < need_blocks) return KVQ_ERR_INVALID_ARG;
  if (page_table == nullptr && (long long)batch * max_blocks > cache->num_pages) return KVQ_ERR_INVALID_ARG;
  if (!x_hat || !codes || !scale || !zero || !aligned16(x_hat) || !aligned16(codes)) return KVQ_ERR_INVALID_ARG;
  s = check_device(nullptr);
  if (s != KVQ_OK) return s;
  DequantParams p{};
  p.codes = codes; p.scale = scale; p.zero = zero; p.seq_lens = seq_lens; p.page_table = page_table;
  p.x_hat = x_hat; p.dev_status = dev_status;
  p.bits = cache->bits; p.k_scheme = cache->k_scheme; p.v_scheme = cache->v_scheme; p.which = which;
  p.head_dim = cache->head_dim; p.group = group_of(cache);
  p.num_kv_heads = cache->num_kv_heads; p.num_pages = cache->num_pages;
  p.batch = batch; p.max_seq_len = max_seq_len; p.max_blocks = max_blocks;
  return launch_dequant(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

KVQ_API kvq_status kvq_decode_workspace_size(const kvq_attn_desc* desc, size_t* bytes) {
  return kvq::decode_workspace_bounded(desc, SIZE_MAX, bytes);
}

KVQ_API kvq_status kvq_decode_path(const kvq_attn_desc* desc, int32_t* path) {
  kvq_status s = check_attn(desc);
  if (s != KVQ_OK) return s;
  if (path == nullptr) return KVQ_ERR_INVALID_ARG;
  *path = use_general(desc) ? KVQ_PATH_GENERAL : KVQ_PATH_SPECIALISED;
  return KVQ_OK;
}

KVQ_API kvq_status kvq_decode_attn(const kvq_attn_desc* desc, const uint16_t* q, const uint8_t* k_codes,
                                   const uint16_t* k_scale, const uint16_t* k_zero, const uint8_t* v_codes,
                                   const uint16_t* v_scale, const uint16_t* v_zero, const int32_t* seq_lens,
                                   const int32_t* page_table, float* out, float* lse, void* workspace,
                                   size_t workspace_bytes, uint32_t* dev_status, void* stream) {
  return kvq::decode_attn_bounded(desc, q, k_codes, k_scale, k_zero, v_codes, v_scale, v_zero, seq_lens, page_table,
                                  out, lse, workspace, workspace_bytes, SIZE_MAX, dev_status, stream);
}

KVQ_API kvq_status kvq_merge(const float* o_parts, const float* lse_parts, int32_t rows, int32_t splits,
                             int32_t head_dim, float* out, float* lse, void* stream) {
  if (rows < 0 || splits < 1 || head_dim < 4 || head_dim > 1024 || (head_dim & 3) != 0) return KVQ_ERR_INVALID_ARG;
  if (rows == 0) return KVQ_OK;
  if (!o_parts || !lse_parts || !out || !lse || !aligned16(o_parts) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  kvq_status s = check_device(nullptr);
  if (s != KVQ_OK) return s;
  return launch_merge(o_parts, lse_parts, rows, splits, head_dim, out, lse, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

}  // extern "C"
