// inkling_rel_attn_decode_noalloc: the decode entry point for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain a device buffer of their own: a plugin
// or extension running inside a host framework that owns all device memory
// and forbids allocation while a step executes, a language binding with no
// access to the CUDA allocator, or a latency-critical loop that must never
// touch the allocator (cudaMalloc may synchronise the device).  Split-KV
// decode needs scratch space for its per-split partial outputs and its work
// counter; this entry point takes that scratch from one fixed, file-scope
// device array instead of from the caller.
//
// The array is kInklingNoallocScratchBytes (32 MiB) per GPU.  Every GPU that
// loads this library keeps it until the process exits.  All calls on a device
// share it and it keeps whatever the previous call left there: the work
// counter, the only part that must start at zero, is cleared on the stream
// before every launch, and the partials are always written before they are
// read.  Two calls whose kernels overlap on the GPU (different streams, or
// different host threads, without ordering between them) would race on the
// array, so callers must order them.
//
// The first call on each device looks up the array's device address with
// cudaGetSymbolAddress (a host-side name of a __device__ variable is not a
// device address) while that device is current, and caches it; make that
// first call outside any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kInklingNoallocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kInklingNoallocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[ira::kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device), or nullptr on failure.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= ira::kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return nullptr;
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int inkling_rel_attn_decode_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* page_table,
    int32_t page_table_stride, const int32_t* seq_lens, const float* rel_logits, int32_t B,
    int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size, int32_t num_pages, int32_t R,
    int32_t window, float scale, int32_t max_seq_len, void* out, float* lse_out,
    int32_t num_splits, int32_t* device_error, void* stream) {
  const size_t need = inkling_rel_attn_decode_workspace_size(B, H_q, H_kv, D, window, max_seq_len,
                                                             num_splits, 0);
  if (need > kInklingNoallocScratchBytes) return INKLING_ERR_WORKSPACE;
  // resolved on every call (cached after the first on each device), whether
  // or not this call splits, so the first call on a device is always the one
  // that does the look-up
  void* scratch = scratch_for_current_device();
  if (!scratch) return INKLING_ERR_CUDA;
  return inkling_rel_attn_decode(q, k_cache, v_cache, page_table, page_table_stride, seq_lens,
                                 rel_logits, B, H_q, H_kv, D, page_size, num_pages, R, window,
                                 scale, max_seq_len, out, lse_out, need > 0 ? scratch : nullptr,
                                 need > 0 ? kInklingNoallocScratchBytes : 0, num_splits,
                                 device_error, stream);
}
