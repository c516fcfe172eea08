/*
 * kvq -- decode attention over an asymmetric INT2/INT4 group-quantized KV
 * cache, for one NVIDIA GB300 (sm_103a).
 *
 * The operation (cited by page title and section of the sources):
 *   - "FOSCAR: Accelerating Decode Attention over 2- and 4-Bit KV Caches
 *     through Affine Folding" (papers.pytorch.kr), abstract: decode attention
 *     streams a KV cache packed as 2- or 4-bit integers; scale and offset are
 *     applied to the other operand or to the output of the two attention
 *     matrix products ("affine folding"), exactly equal to dequantizing first.
 *   - rag-lover.com summary of arXiv 2611.09722, section "使える条件"
 *     (conditions of use): asymmetric quantization, each group shares a scale
 *     s and an offset z; K and V each choose token-wise or channel-wise groups
 *     independently; group size 128; 4 query heads per KV head.
 *   - same page, section "解説" (commentary): which side each scheme folds on,
 *     and code bits placed in the low bits of a tensor-core element.
 *
 * out[b, h, :] = softmax(S) V_hat[b, h/G_q],  S_l = sm_scale * q[b,h] . K_hat[b, h/G_q, l],
 * lse[b, h] = ln sum_l exp(S_l), with x_hat = s * code + z and code unsigned.
 *
 * Cache format (this library's; the pages leave it open)
 * -------------------------------------------------------
 * head_dim D (64, 128 or 256); a block (= page) holds 128 consecutive tokens
 * of one KV head.  Codes of one block form a matrix: K rows are the 128
 * tokens (D channels along the row), V rows are the D channels (128 tokens
 * along the row).  A row is packed little-endian (column i at bits
 * [b*(i mod 8/b), +b) of row byte i*b/8), cut into 16-byte chunks, and the
 * block is stored chunk-major: byte offset (chunk*nrows + row)*16 + byte,
 * nrows = 128 (K) or D (V).  Block bytes: 128 * D * b / 8 (8192 for INT4,
 * 4096 for INT2 at D = 128).  codes array: [num_pages][num_kv_heads][block
 * bytes].  Quantization groups of G elements: token-wise, G consecutive
 * channels of a token; channel-wise, G consecutive tokens of a channel
 * (aligned to the block).  scale / zero arrays (fp16 bit patterns):
 * [num_pages][num_kv_heads][128 * D / G]; token-wise, entry t * (D / G) + g
 * is channel group g of block token t; channel-wise, entry k * D + c is
 * channel c over block tokens [k G, (k + 1) G).  (D = G = 128: one entry per
 * token, resp. per channel.)  Tokens at or past a sequence's length have code
 * 0 (token-wise: s = z = 0; a channel-wise group without valid tokens:
 * s = z = 0).
 * Sequence b's block j lives in page page_table[b*max_blocks + j], or in page
 * b*max_blocks + j when page_table is NULL ("contiguous" cache).
 *
 * Conventions
 * -----------
 *  - All pointers except descriptors, out-params and the stream are device
 *    pointers on the current CUDA device, 16-byte aligned, owned by the
 *    caller.  The library allocates no memory; apart from the fixed scratch
 *    array behind kvq_decode_attn_static it keeps no state.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream); every call is
 *    asynchronous on it.
 *  - A non-KVQ_OK return means nothing was launched.  Errors found on the
 *    device are OR-ed into *dev_status (KVQ_DEV_* bits; the caller zeroes it
 *    and reads it after synchronizing; it may be NULL).  Device checks turn
 *    bad lengths and page ids into empty/zero work, never into out-of-range
 *    memory accesses.
 *  - No C++ exception crosses this interface.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_API __attribute__((visibility("default")))

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1, /* NULL/misaligned pointer, bad size or enum value */
  KVQ_ERR_UNSUPPORTED = 2, /* well-formed but not built (e.g. head_dim 96) */
  KVQ_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  KVQ_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  KVQ_ERR_DEVICE = 5       /* current device is not an sm_103 GPU */
} kvq_status;

/* Bits of *dev_status. */
#define KVQ_DEV_BAD_SEQ_LEN 0x1u /* seq_len < 0 or > max_blocks*128 (or > max_seq_len for pack) */
#define KVQ_DEV_BAD_PAGE 0x2u    /* page id outside [0, num_pages) */
#define KVQ_DEV_NONFINITE 0x4u   /* pack: NaN/Inf input, or s / z overflow fp16 */
#define KVQ_DEV_TIMEOUT 0x8u     /* a pipeline wait ran out; outputs are not valid */

typedef enum kvq_scheme { KVQ_TOKENWISE = 0, KVQ_CHANNELWISE = 1 } kvq_scheme;

/* Tensor-core operand precision of decode attention.
 * FP8: KV codes as exact E4M3 values (code * 2^-9); Q' and P' as sums of
 *      three E4M3 parts.  The production path.
 * BF16: KV codes as exact BF16 integers; Q' and P' as sums of two BF16
 *      parts.  A correctness mode with tighter error. */
typedef enum kvq_operand_mode { KVQ_OPERANDS_FP8 = 0, KVQ_OPERANDS_BF16 = 1 } kvq_operand_mode;

typedef struct kvq_cache_desc {
  int32_t bits;         /* 2 or 4 */
  int32_t k_scheme;     /* kvq_scheme used by K */
  int32_t v_scheme;     /* kvq_scheme used by V */
  int32_t head_dim;     /* D: 64, 128 or 256 */
  int32_t num_kv_heads; /* >= 1 */
  int32_t num_pages;    /* 128-token pages the cache arrays hold */
  int32_t group_size;   /* G: 32, 64 or 128 elements per quantization group
                           (0 = 128), at most head_dim; the same for K and V */
} kvq_cache_desc;

typedef struct kvq_attn_desc {
  kvq_cache_desc cache;
  int32_t batch;        /* sequences (>= 1) */
  int32_t num_q_heads;  /* 1, 2, 4 or 8 times num_kv_heads (query head h reads
                           KV head h / (num_q_heads / num_kv_heads)) */
  int32_t max_blocks;   /* page_table row length; contiguous: blocks per sequence */
  int32_t operand_mode; /* kvq_operand_mode */
  float sm_scale;       /* <= 0 selects 1/sqrt(head_dim) */
  int32_t num_ctas;     /* persistent CTAs; 0 = two per SM */
  uint32_t flags;       /* 0 or KVQ_FLAG_* bits */
} kvq_attn_desc;

/* Test hook: the loader withholds one tile so that every waiting stage runs
 * into its time limit; the call must end with KVQ_DEV_TIMEOUT set. */
#define KVQ_FLAG_TEST_STALL 0x1u
/* Test hook (general kernel; the specialised kernel ignores it): the first
 * CTA's MMA completion barrier waits for two signals a phase, so the wait
 * for its first QK^T product (per warp with token-wise K, CTA-wide with
 * channel-wise K) runs into its time limit; the call must end with
 * KVQ_DEV_TIMEOUT set. */
#define KVQ_FLAG_TEST_STALL_MMA 0x4u
/* 2-bit caches: feed the V codes to the tensor cores as E2M1 values
 * (code / 2, two 2-bit fields per nibble taken with one mask each) staged in
 * shared memory -- the placement of the rag-lover.com summary of arXiv
 * 2611.09722, section "解説" -- instead of the default E4M3 bytes
 * (code * 2^-9) written to tensor memory.  Same results within the FP8
 * tolerance; slower on GB300 (more shared-memory stores, fewer load stages).
 * Requires bits = 2, KVQ_OPERANDS_FP8 and 4 query heads per KV head, else
 * KVQ_ERR_UNSUPPORTED. */
#define KVQ_FLAG_E2M1_V 0x2u

/* Human-readable name of a status code (static storage). */
KVQ_API const char* kvq_status_string(kvq_status status);

/* Library version, major*10000 + minor*100 + patch. */
KVQ_API int32_t kvq_version(void);

/* Bytes of one K or V cache: *codes_bytes for the codes array,
 * *scale_bytes for each of the scale and zero arrays.  Host only. */
KVQ_API kvq_status kvq_cache_bytes(const kvq_cache_desc* cache, size_t* codes_bytes, size_t* scale_bytes);

/*
 * Quantize and pack K (which = 0) or V (which = 1) into the cache format
 * above.  Group rule ([SUM] 使える条件, asymmetric min/max; rounding is this
 * library's reading): z = fp16 round-down of the group minimum,
 * s = fp16 round-up of fp32((max - z) / (2^bits - 1)),
 * code = clamp(rint(fp32(fp32(x - z) / s)), 0, 2^bits - 1), all IEEE fp32;
 * max == z gives s = 0, code = 0.
 *   x          fp32 [batch][num_kv_heads][max_seq_len][head_dim]
 *   seq_lens   int32 [batch] in [0, max_seq_len], or NULL (all max_seq_len)
 *   page_table int32 [batch][max_blocks], or NULL (contiguous; then
 *              batch*max_blocks <= num_pages)
 *   max_blocks >= ceil(max_seq_len / 128)
 *   codes, scale, zero: the cache arrays (only pages the batch covers are
 *              written)
 * Device errors: KVQ_DEV_NONFINITE (that group is written as zeros),
 * KVQ_DEV_BAD_SEQ_LEN, KVQ_DEV_BAD_PAGE (that block is skipped).
 */
KVQ_API kvq_status kvq_pack(const kvq_cache_desc* cache, int32_t which, const float* x, int32_t batch,
                            int32_t max_seq_len, const int32_t* seq_lens, const int32_t* page_table,
                            int32_t max_blocks, uint8_t* codes, uint16_t* scale, uint16_t* zero,
                            uint32_t* dev_status, void* stream);

/*
 * Append one token per sequence to a packed K (which = 0) or V (which = 1)
 * cache, for a decode loop that grows the cache step by step.  The new token
 * of sequence b sits at position seq_lens[b] (the tokens already cached); it
 * is stored in row seq_lens[b] % 128 of the caller's window of that
 * sequence's current 128-token block, and the block is quantized and packed
 * again from the window's valid rows (seq_lens[b] % 128 + 1 of them), so the
 * cache equals what kvq_pack makes of the whole sequence: a channel-wise
 * group spans the block's valid tokens, as for a partial last block.  The
 * caller then advances seq_lens[b] by one; when a block fills, the next
 * block's rows overwrite the window from row 0 (no reset needed).  A cache
 * that starts from kvq_pack of a prefix needs the prefix's partial last block
 * copied into the window first.
 *   x_new      fp32 [batch][num_kv_heads][head_dim], 16-byte aligned
 *   seq_lens   int32 [batch], each in [0, max_blocks * 128)
 *   page_table int32 [batch][max_blocks] or NULL (contiguous; then
 *              batch * max_blocks <= num_pages)
 *   window     fp32 [batch][num_kv_heads][128][head_dim], caller-owned (one for
 *              K, one for V), 16-byte aligned
 *   codes, scale, zero: the cache arrays (only the current block's page is
 *              written)
 * Device errors as kvq_pack (KVQ_DEV_BAD_SEQ_LEN when seq_lens[b] is out of
 * range: that sequence is skipped).
 */
KVQ_API kvq_status kvq_append(const kvq_cache_desc* cache, int32_t which, const float* x_new, int32_t batch,
                              const int32_t* seq_lens, const int32_t* page_table, int32_t max_blocks,
                              float* window, uint8_t* codes, uint16_t* scale, uint16_t* zero,
                              uint32_t* dev_status, void* stream);

/*
 * Read a packed K or V cache back as fp32 x_hat = s * code + z (exact, one
 * rounding).  x_hat: fp32 [batch][num_kv_heads][max_seq_len][head_dim]; positions
 * at or past seq_lens[b] are written as 0.  Other arguments as kvq_pack.
 */
KVQ_API kvq_status kvq_dequant(const kvq_cache_desc* cache, int32_t which, const uint8_t* codes,
                               const uint16_t* scale, const uint16_t* zero, int32_t batch, int32_t max_seq_len,
                               const int32_t* seq_lens, const int32_t* page_table, int32_t max_blocks,
                               float* x_hat, uint32_t* dev_status, void* stream);

/* Workspace bytes kvq_decode_attn needs for `desc` (queries the current
 * device when desc->num_ctas == 0). */
KVQ_API kvq_status kvq_decode_workspace_size(const kvq_attn_desc* desc, size_t* bytes);

/* Which decode kernel kvq_decode_attn runs for `desc` (host only, no device
 * needed): *path = KVQ_PATH_SPECIALISED (persistent tile-range kernel, head
 * dim 128, groups of 128, E4M3 operands) or KVQ_PATH_GENERAL (plan, block-
 * range and merge kernels).  The rule is the one kvq_decode_attn describes. */
#define KVQ_PATH_SPECIALISED 0
#define KVQ_PATH_GENERAL 1
KVQ_API kvq_status kvq_decode_path(const kvq_attn_desc* desc, int32_t* path);

/*
 * Decode attention over the packed cache, affine-folded (abstract; [SUM] 解説):
 * token-wise K scales the partial q.code by s and adds z * sum(q); channel-
 * wise K multiplies q by s before the product and adds q . z; token-wise V
 * multiplies the probabilities by s and adds sum(p * z); channel-wise V scales
 * each G-token group's partial product by s and adds z * sum(p) of that
 * group ([SUM] 限界と未検証の範囲: per-group application); with groups
 * smaller than the head dim, token-wise K and V fold per G-channel group.
 * Two kernels (kvq_decode_path tells which one a call takes).  The
 * specialised one (head dim 128, groups of 128, E4M3 operands) splits the
 * work over persistent CTAs in equal tile ranges; a sequence/head cut
 * between CTAs is merged on the device by log-sum-exp; its units take up to
 * 4 query heads, so with 8 query heads per KV head it reads each KV block
 * twice.  The general one runs three launches -- a plan kernel cuts each
 * (sequence, unit)'s blocks into ranges in proportion to the sequence's
 * length, a second kernel decodes one range per CTA (units of 4 or 8 query
 * heads: each KV block is read once), and a log-sum-exp merge combines the
 * ranges.  The general kernel takes every other geometry (head dim 64 / 256,
 * groups of 32 / 64) and the BF16 mode, and on the specialised kernel's
 * geometry (E4M3) every call with batch x units x max_blocks >= 8192 (units
 * per sequence: the KV heads, twice that with 8 query heads per KV head),
 * where it was measured faster for every scheme pair and head count; smaller
 * calls and KVQ_FLAG_E2M1_V stay in the specialised kernel.  KVQ_FLAG_E2M1_V on
 * another geometry or in the BF16 mode: KVQ_ERR_UNSUPPORTED.  Query heads
 * per KV head: 1, 2, 4 or 8.  sm_scale <= 0 means 1 / sqrt(head_dim).
 *   q        bf16 [batch][num_q_heads][head_dim]
 *   k_codes, v_codes, k_scale, k_zero, v_scale, v_zero: cache arrays
 *   seq_lens int32 [batch], each in [0, max_blocks*128]
 *   page_table int32 [batch][max_blocks] or NULL (contiguous)
 *   out      fp32 [batch][num_q_heads][head_dim];  lse fp32 [batch][num_q_heads]
 *            (natural log; empty sequence: out = 0, lse = -inf)
 *   workspace >= kvq_decode_workspace_size bytes, 256-byte aligned; its
 *            contents need no initialisation; concurrent calls need separate
 *            workspaces
 */
KVQ_API kvq_status kvq_decode_attn(const kvq_attn_desc* desc, const uint16_t* q, const uint8_t* k_codes,
                                   const uint16_t* k_scale, const uint16_t* k_zero, const uint8_t* v_codes,
                                   const uint16_t* v_scale, const uint16_t* v_zero, const int32_t* seq_lens,
                                   const int32_t* page_table, float* out, float* lse, void* workspace,
                                   size_t workspace_bytes, uint32_t* dev_status, void* stream);

/*
 * Decode attention without a caller workspace, for callers that cannot
 * allocate device memory: a runtime whose device memory plan is frozen after
 * start-up, a plugin interface that hands over only input and output
 * buffers, or a latency-critical path where an allocation would synchronise
 * the device.  (No counterpart on the pages describing the method; this call
 * exists for such integrations.)  Same arguments, semantics and errors as
 * kvq_decode_attn minus the workspace: the split-merge scratch lives in a
 * fixed 4 MiB device array owned by the library, held on every device that
 * loads the library until the process exits.  Returns KVQ_ERR_WORKSPACE when
 * a call needs more scratch than that (the specialised kernel: batch *
 * num_kv_heads * 4 bytes of counters, twice that with 8 query heads per KV
 * head, plus 4 KiB per CTA; the general kernel: the plan (4 bytes per
 * sequence, 16 per CTA) and head_dim + 1 floats per query head and block
 * range).  A call kvq_decode_attn would run in the general kernel on the
 * specialised kernel's geometry (E4M3 operands) runs in the specialised
 * kernel here when the general kernel's scratch would not fit.
 * kvq_decode_attn with a caller workspace remains available.  Every call on a stream that is not being captured
 * looks up the array's address on the current device (the first such call
 * loads the module); a call inside a stream capture reuses the address of
 * the last uncaptured call on that device, so make one ordinary call on each
 * device before any capture, and again after a device reset.  Every call on a
 * device shares the array and the counters are cleared on the stream at each
 * call, so calls whose kernels may overlap on the GPU (unordered streams)
 * race.  Allocates nothing.
 */
KVQ_API kvq_status kvq_decode_attn_static(const kvq_attn_desc* desc, const uint16_t* q, const uint8_t* k_codes,
                                          const uint16_t* k_scale, const uint16_t* k_zero, const uint8_t* v_codes,
                                          const uint16_t* v_scale, const uint16_t* v_zero, const int32_t* seq_lens,
                                          const int32_t* page_table, float* out, float* lse, uint32_t* dev_status,
                                          void* stream);

/*
 * Log-sum-exp merge of partial attention results over disjoint token ranges
 * (split-KV): lse[r] = ln sum_s exp(lse_parts[r][s]),
 * out[r] = sum_s exp(lse_parts[r][s] - lse[r]) * o_parts[r][s].
 *   o_parts fp32 [rows][splits][head_dim] (each part normalised over its own
 *           range), lse_parts fp32 [rows][splits] (-inf = empty part)
 *   out fp32 [rows][head_dim], lse fp32 [rows]; all parts empty -> 0, -inf
 *   head_dim: a multiple of 4, at most 1024
 */
KVQ_API kvq_status kvq_merge(const float* o_parts, const float* lse_parts, int32_t rows, int32_t splits,
                             int32_t head_dim, float* out, float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
