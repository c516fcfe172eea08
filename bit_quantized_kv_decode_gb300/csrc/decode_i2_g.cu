// Decode-attention kernel instances for 2-bit caches with 1, 2 or 8 query heads
// per KV head (the run-time head grouping of DecodeParams).
#define KVQ_GQ4 false
#define KVQ_FN launch_decode_i2_g
#include "decode_i2.cu"
