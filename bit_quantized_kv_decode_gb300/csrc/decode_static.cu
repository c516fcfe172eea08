// kvq_decode_attn_static: decode attention for callers that cannot allocate
// device memory.
//
// Some callers have no way to obtain a workspace: an inference runtime that
// forbids device allocations once its memory plan is fixed, a plugin ABI that
// hands a kernel only its input and output buffers, or code running where a
// cudaMalloc would synchronise the device or break a latency budget.  This
// entry point takes the same inputs and outputs as kvq_decode_attn but keeps
// the split-merge scratch (arrival counters and partial results) in a fixed
// array in device memory that belongs to the library: every GPU that loads
// the library holds these kKvqStaticScratchBytes until the process exits.
//
// Each call looks up that array's device address on the current device
// (cudaGetSymbolAddress, which loads the module on a device's first call)
// whenever the caller's stream is not being captured, so a device reset or a
// new context is picked up by the next ordinary call; a call made while the
// stream is being captured reuses the address found by the last ordinary call
// on that device, so make one call on each device before any stream capture
// (and again after a device reset).  All calls on a device share the one
// array and find the previous call's contents in it: the counters that must
// start at zero are cleared on the stream at every call, and calls whose
// kernels overlap on the GPU (different streams, no ordering) race on the
// array.  Nothing here allocates: no cudaMalloc, cudaFree or library routine
// that allocates.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kvq_entry.h"

namespace kvq {
namespace {

constexpr size_t kKvqStaticScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kKvqStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device: looked up
// again on every call whose stream is not being captured (a reset device or
// a new context gets a fresh address), taken from the last lookup on this
// device during a capture.
kvq_status scratch_on_current_device(cudaStream_t stream, void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return KVQ_ERR_DEVICE; }
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_DEVICE;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) { cudaGetLastError(); return KVQ_ERR_CUDA; }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) { cudaGetLastError(); return KVQ_ERR_CUDA; }
    g_scratch_ptr[dev] = p;
  }
  if (g_scratch_ptr[dev] == nullptr) return KVQ_ERR_CUDA;  // first call on this device inside a capture
  *ptr = g_scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace
}  // namespace kvq

extern "C" KVQ_API kvq_status kvq_decode_attn_static(const kvq_attn_desc* desc, const uint16_t* q,
                                                     const uint8_t* k_codes, const uint16_t* k_scale,
                                                     const uint16_t* k_zero, const uint8_t* v_codes,
                                                     const uint16_t* v_scale, const uint16_t* v_zero,
                                                     const int32_t* seq_lens, const int32_t* page_table, float* out,
                                                     float* lse, uint32_t* dev_status, void* stream) {
  size_t need = 0;
  kvq_status s = kvq::decode_workspace_bounded(desc, kvq::kKvqStaticScratchBytes, &need);
  if (s != KVQ_OK) return s;
  if (need > kvq::kKvqStaticScratchBytes) return KVQ_ERR_WORKSPACE;  // larger than the fixed scratch
  s = kvq::check_device(nullptr);  // an unsupported device is KVQ_ERR_DEVICE, before any symbol lookup
  if (s != KVQ_OK) return s;
  void* scratch = nullptr;
  s = kvq::scratch_on_current_device(static_cast<cudaStream_t>(stream), &scratch);
  if (s != KVQ_OK) return s;
  return kvq::decode_attn_bounded(desc, q, k_codes, k_scale, k_zero, v_codes, v_scale, v_zero, seq_lens, page_table,
                                  out, lse, scratch, kvq::kKvqStaticScratchBytes, kvq::kKvqStaticScratchBytes,
                                  dev_status, stream);
}
