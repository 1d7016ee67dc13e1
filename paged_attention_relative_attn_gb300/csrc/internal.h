// Host-side declarations shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "../../include/inkling_rel_attn.h"

namespace ira {

// Devices a process may drive for which per-device state is cached.
constexpr int kMaxDevices = 64;

// Raise `kern`'s dynamic shared-memory limit to `bytes` on the current device.
// Function attributes belong to each device's context, so this is done once
// per (kernel, device): `done` is the kernel's own kMaxDevices-entry table
// (zero-initialised), holding the limit already set on each device.  Returns
// false when the device query or the attribute call fails.
bool smem_limit_on_device(const void* kern, int bytes, std::atomic<int>* done);

// SMs of the current device (152 when the query fails).
int sm_count();

// Validated decode call, with the split plan resolved.
struct DecodeCall {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* page_table;
  int32_t pt_stride;
  const int32_t* seq_lens;
  const float* rel;
  int32_t B, H_q, H_kv, D, P, num_pages, R, window;
  int32_t QL;        // query tokens per sequence (1: plain decode)
  float scale;
  int32_t keys_max;  // host bound on visible keys per item
  int32_t S;         // split count (grid.x)
  int32_t chunk;     // keys per split (multiple of 64)
  void* out;
  float* lse_out;
  float* o_part;     // [B * QL, H_q, S, D] when S > 1
  float* lse_part;   // [B * QL, H_q, S]   when S > 1
  int32_t* counter;  // work-item counter (S > 1), zeroed by the launcher
  int32_t* dev_err;
  cudaStream_t stream;
};

struct PrefillCall {
  const void* q;
  const int32_t* cu_seqlens_q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* page_table;
  int32_t pt_stride;
  const int32_t* seq_lens;
  const float* rel;
  int32_t B, T, max_q_len, H_q, H_kv, D, P, num_pages, R, window;
  float scale;
  int32_t max_seq_len;
  void* out;
  float* lse_out;
  int32_t* dev_err;
  cudaStream_t stream;
};

struct KvAppendCall {
  const void* k_new;
  const void* v_new;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  const int32_t* page_table;
  int32_t pt_stride;
  int32_t B, T, H_kv, D, P, num_pages;
  void* k_cache;
  void* v_cache;
  int32_t* dev_err;
  cudaStream_t stream;
};

struct KvConvCall {
  const void* k_new;
  const void* v_new;
  const float* w_k;
  const float* w_v;
  void* state_k;
  void* state_v;
  const int32_t* state_slots;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  const int32_t* page_table;
  int32_t pt_stride;
  int32_t width, num_slots, B, T, max_q_len, H_kv, D, P, num_pages;
  void* k_cache;
  void* v_cache;
  int32_t* dev_err;
  cudaStream_t stream;
};

int launch_decode(const DecodeCall& c);        // returns INKLING_* code
int launch_prefill(const PrefillCall& c);      // returns INKLING_* code
int launch_kv_append(const KvAppendCall& c);   // returns INKLING_* code
int launch_kv_conv_append(const KvConvCall& c);  // returns INKLING_* code

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swizzle);

// Multi-token decode: query tokens per item (token group) for q_len tokens per
// sequence and G query heads per KV head -- the rows (token, head) of an item
// fill at most 16 (two 8-row MMA tiles).  Shared by the ABI helpers and the
// launcher so that the split plan and the kernel agree.
// (as many tokens as fit 16 rows: each K/V tile then passes through shared
// memory and the MMAs once for all of them -- for 4 tokens x 3 heads one
// 12-row item instead of two 6-row items.  INKLING_MTP_MAX_ROWS > 0 forces the
// bound.)
#ifndef INKLING_MTP_MAX_ROWS
#define INKLING_MTP_MAX_ROWS 0
#endif
inline int32_t decode_token_group(int32_t q_len, int32_t G) {
  if (q_len <= 1) return 1;
  const int32_t rows = INKLING_MTP_MAX_ROWS > 0 ? INKLING_MTP_MAX_ROWS : 16;
  int32_t tg = G > 0 ? rows / G : 1;
  if (tg < 1) tg = 1;
  return tg < q_len ? tg : q_len;
}

// Split plan shared by the ABI helpers and the launcher.
int32_t decode_keys_max(int32_t window, int32_t max_seq_len);
void decode_split_plan(int32_t keys_max, int32_t S_req, int32_t* S_out, int32_t* chunk_out);
size_t decode_workspace_bytes(int32_t B, int32_t H_q, int32_t D, int32_t S);
size_t align256(size_t x);

}  // namespace ira
