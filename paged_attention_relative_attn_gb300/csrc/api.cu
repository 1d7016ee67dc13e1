// C ABI of libinkling_rel_attn.so: argument validation, the split plan,
// workspace sizing, device checks and error strings.  See
// include/inkling_rel_attn.h for the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"

namespace ira {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int32_t decode_keys_max(int32_t window, int32_t max_seq_len) {
  int32_t k = std::max<int32_t>(max_seq_len, 1);
  if (window > 0 && window < k) k = window;
  return k;
}

// Resolve a split request into (S, chunk): chunk is a multiple of 64 keys and
// S = ceil(keys_max / chunk) <= 128.
void decode_split_plan(int32_t keys_max, int32_t S_req, int32_t* S_out, int32_t* chunk_out) {
  const int64_t keys = std::max<int32_t>(keys_max, 1);
  int64_t S = std::max<int32_t>(S_req, 1);
  S = std::min<int64_t>(S, 128);
  S = std::min<int64_t>(S, ceil_div(keys, 64));
  S = std::max<int64_t>(S, 1);
  int64_t chunk = ceil_div(ceil_div(keys, S), 64) * 64;
  S = ceil_div(keys, chunk);
  if (S <= 1) {
    S = 1;
    chunk = std::max<int64_t>(chunk, keys);
  }
  *S_out = (int32_t)S;
  *chunk_out = (int32_t)std::min<int64_t>(chunk, INT32_MAX);
}

// Workspace layout when S > 1: [work-item counter, 256 B][o_part fp32
// B*H_q*S*D][lse_part fp32 B*H_q*S], each part 256-byte aligned.
size_t decode_workspace_bytes(int32_t B, int32_t H_q, int32_t D, int32_t S) {
  if (S <= 1 || B <= 0 || H_q <= 0) return 0;
  const size_t rows = (size_t)B * H_q * S;
  return 256 + align256(rows * D * sizeof(float)) + align256(rows * sizeof(float));
}

// ---------------------------------------------------------------- tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank, void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                  CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estr[5];
  for (uint32_t i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dtype, rank, base, gdim, gstride, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool smem_limit_on_device(const void* kern, int bytes, std::atomic<int>* done) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
  if (dev < kMaxDevices && done[dev].load(std::memory_order_acquire) == bytes) return true;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return false;
  if (dev < kMaxDevices) done[dev].store(bytes, std::memory_order_release);
  return true;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 152;
  return n;
}

// ---------------------------------------------------------------- device info
struct DevInfo {
  int ok;  // 1 = sm_103, 0 = other, -1 = query failed
  int sms;
};

static DevInfo device_info() {
  static std::atomic<int> cached_ok[kMaxDevices];
  static std::atomic<int> cached_sms[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return {-1, 0};
  if (dev < kMaxDevices) {
    int ok = cached_ok[dev].load(std::memory_order_relaxed);
    if (ok != 0) return {ok > 0 ? 1 : 0, cached_sms[dev].load(std::memory_order_relaxed)};
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return {-1, 0};
  const int ok = (major == 10 && minor == 3) ? 1 : 0;
  if (dev < kMaxDevices) {
    cached_sms[dev].store(sms, std::memory_order_relaxed);
    cached_ok[dev].store(ok ? 1 : -1, std::memory_order_relaxed);
  }
  return {ok, sms};
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

static bool common_shape_ok(int32_t H_q, int32_t H_kv, int32_t D, int32_t P, int32_t num_pages,
                            int32_t R, int32_t pt_stride) {
  if (H_q <= 0 || H_kv <= 0 || H_q % H_kv != 0 || H_q / H_kv > 16) return false;
  if (D != 64 && D != 128) return false;
  if (P <= 0 || P % 16 != 0 || P > 256) return false;
  if (num_pages <= 0 || R <= 0 || pt_stride <= 0) return false;
  if ((int64_t)pt_stride * P > INT32_MAX) return false;
  return true;
}

}  // namespace ira

using namespace ira;

extern "C" {

int32_t inkling_rel_attn_version(void) { return 100; }

const char* inkling_rel_attn_error_string(int32_t code) {
  switch (code) {
    case INKLING_OK: return "success";
    case INKLING_ERR_ARG: return "invalid argument (NULL pointer, bad scalar or unsupported shape)";
    case INKLING_ERR_ALIGN: return "misaligned pointer (16 bytes for q/k/v/out/workspace, 4 otherwise)";
    case INKLING_ERR_WORKSPACE: return "workspace missing or too small";
    case INKLING_ERR_DEVICE: return "current CUDA device is not an sm_103 GPU (or no device)";
    case INKLING_ERR_CUDA: return "a CUDA call or kernel launch failed";
    default: return "unknown error code";
  }
}

int32_t inkling_rel_attn_choose_splits(int32_t B, int32_t H_kv, int32_t window, int32_t max_seq_len,
                                       int32_t num_sms) {
  if (num_sms <= 0) num_sms = 152;
  const int64_t keys = decode_keys_max(window, max_seq_len);
  if (B <= 0 || H_kv <= 0) return 1;
  const int64_t pairs = (int64_t)B * H_kv;
  const int64_t target = 3LL * num_sms;          // >= 3 CTAs per SM overall
  const int64_t s_fill = (target + pairs - 1) / pairs;
  const int64_t s_len = (keys + 255) / 256;      // each split >= 256 keys
  const int64_t s_cap = (keys + 1023) / 1024;    // each split <= 1024 keys
  int64_t S = std::max(s_cap, std::min(s_fill, s_len));
  S = std::max<int64_t>(1, std::min<int64_t>(S, 128));
  int32_t S_out, chunk;
  decode_split_plan((int32_t)keys, (int32_t)S, &S_out, &chunk);
  return S_out;
}

}  // extern "C"

namespace ira {
// Split plan of a (multi-token) decode call: keys per item, split count and
// keys per split.  q_len = 1 is plain decode.
static void decode_call_plan(int32_t B, int32_t q_len, int32_t H_q, int32_t H_kv, int32_t window,
                             int32_t max_seq_len, int32_t num_splits, int32_t num_sms,
                             int32_t* keys_out, int32_t* S_out, int32_t* chunk_out) {
  const int32_t G = H_kv > 0 ? H_q / H_kv : 1;
  const int32_t TG = decode_token_group(q_len, G);
  const int32_t NG = (std::max(q_len, 1) + TG - 1) / TG;
  // a group's keys: its first token's window plus the TG - 1 later positions
  const int32_t w_eff = window > 0 ? window + TG - 1 : 0;
  const int32_t keys = decode_keys_max(w_eff, max_seq_len);
  int32_t S_req = num_splits;
  if (S_req <= 0) {
    if (num_sms <= 0) {
      DevInfo di = device_info();
      num_sms = di.ok >= 0 && di.sms > 0 ? di.sms : 152;
    }
    S_req = inkling_rel_attn_choose_splits(
        (int32_t)std::min<int64_t>((int64_t)B * NG, INT32_MAX), H_kv, w_eff, max_seq_len, num_sms);
  }
  *keys_out = keys;
  decode_split_plan(keys, S_req, S_out, chunk_out);
}

// Validated decode of q_len >= 1 query tokens per sequence.
static int decode_call(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* page_table, int32_t page_table_stride,
                       const int32_t* seq_lens, const float* rel_logits, int32_t B, int32_t q_len,
                       int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size, int32_t num_pages,
                       int32_t R, int32_t window, float scale, int32_t max_seq_len, void* out,
                       float* lse_out, void* workspace, size_t workspace_bytes,
                       int32_t num_splits, int32_t* device_error, void* stream) {
  if (B < 0 || max_seq_len < 0 || q_len < 1 || q_len > 64) return INKLING_ERR_ARG;
  if (q_len > 1 && max_seq_len < q_len) return INKLING_ERR_ARG;
  if ((int64_t)B * q_len * H_q > INT32_MAX / 4) return INKLING_ERR_ARG;
  if (!common_shape_ok(H_q, H_kv, D, page_size, num_pages, R, page_table_stride)) return INKLING_ERR_ARG;
  if (!(scale == scale)) return INKLING_ERR_ARG;
  if (B == 0) return INKLING_OK;
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !rel_logits || !out)
    return INKLING_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(page_table, 4) || !aligned(seq_lens, 4) || !aligned(rel_logits, 4) ||
      !aligned(lse_out, 4) || !aligned(device_error, 4) || !aligned(workspace, 16))
    return INKLING_ERR_ALIGN;
  const DevInfo di = device_info();
  if (di.ok != 1) return INKLING_ERR_DEVICE;

  DecodeCall c;
  c.q = q;
  c.k_cache = k_cache;
  c.v_cache = v_cache;
  c.page_table = page_table;
  c.pt_stride = page_table_stride;
  c.seq_lens = seq_lens;
  c.rel = rel_logits;
  c.B = B;
  c.QL = q_len;
  c.H_q = H_q;
  c.H_kv = H_kv;
  c.D = D;
  c.P = page_size;
  c.num_pages = num_pages;
  c.R = R;
  c.window = window;
  c.scale = scale;
  decode_call_plan(B, q_len, H_q, H_kv, window, max_seq_len, num_splits, di.sms, &c.keys_max,
                   &c.S, &c.chunk);
  c.out = out;
  c.lse_out = lse_out;
  c.o_part = nullptr;
  c.lse_part = nullptr;
  c.counter = nullptr;
  if (c.S > 1) {
    const size_t need = decode_workspace_bytes(B * q_len, H_q, D, c.S);
    if (!workspace || workspace_bytes < need) return INKLING_ERR_WORKSPACE;
    const size_t rows = (size_t)B * q_len * H_q * c.S;
    char* ws = static_cast<char*>(workspace);
    c.counter = reinterpret_cast<int32_t*>(ws);
    c.o_part = reinterpret_cast<float*>(ws + 256);
    c.lse_part = reinterpret_cast<float*>(ws + 256 + align256(rows * D * sizeof(float)));
  }
  c.dev_err = device_error;
  c.stream = static_cast<cudaStream_t>(stream);
  return launch_decode(c);
}
}  // namespace ira

extern "C" {

size_t inkling_rel_attn_decode_workspace_size(int32_t B, int32_t H_q, int32_t H_kv, int32_t D,
                                              int32_t window, int32_t max_seq_len,
                                              int32_t num_splits, int32_t num_sms) {
  return inkling_rel_attn_decode_multi_workspace_size(B, 1, H_q, H_kv, D, window, max_seq_len,
                                                      num_splits, num_sms);
}

size_t inkling_rel_attn_decode_multi_workspace_size(int32_t B, int32_t q_len, int32_t H_q,
                                                    int32_t H_kv, int32_t D, int32_t window,
                                                    int32_t max_seq_len, int32_t num_splits,
                                                    int32_t num_sms) {
  if (B <= 0 || q_len < 1 || H_q <= 0 || H_kv <= 0) return 0;
  int32_t keys, S, chunk;
  decode_call_plan(B, q_len, H_q, H_kv, window, max_seq_len, num_splits, num_sms, &keys, &S,
                   &chunk);
  return decode_workspace_bytes(B * q_len, H_q, D, S);
}

size_t inkling_rel_attn_prefill_workspace_size(int32_t T, int32_t H_q, int32_t D) {
  (void)T;
  (void)H_q;
  (void)D;
  return 0;
}

int inkling_rel_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* page_table, int32_t page_table_stride,
                            const int32_t* seq_lens, const float* rel_logits, int32_t B, int32_t H_q,
                            int32_t H_kv, int32_t D, int32_t page_size, int32_t num_pages, int32_t R,
                            int32_t window, float scale, int32_t max_seq_len, void* out,
                            float* lse_out, void* workspace, size_t workspace_bytes,
                            int32_t num_splits, int32_t* device_error, void* stream) {
  return decode_call(q, k_cache, v_cache, page_table, page_table_stride, seq_lens, rel_logits, B, 1,
                     H_q, H_kv, D, page_size, num_pages, R, window, scale, max_seq_len, out,
                     lse_out, workspace, workspace_bytes, num_splits, device_error, stream);
}

int inkling_rel_attn_decode_multi(const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* page_table, int32_t page_table_stride,
                                  const int32_t* seq_lens, const float* rel_logits, int32_t B,
                                  int32_t q_len, int32_t H_q, int32_t H_kv, int32_t D,
                                  int32_t page_size, int32_t num_pages, int32_t R, int32_t window,
                                  float scale, int32_t max_seq_len, void* out, float* lse_out,
                                  void* workspace, size_t workspace_bytes, int32_t num_splits,
                                  int32_t* device_error, void* stream) {
  return decode_call(q, k_cache, v_cache, page_table, page_table_stride, seq_lens, rel_logits, B,
                     q_len, H_q, H_kv, D, page_size, num_pages, R, window, scale, max_seq_len, out,
                     lse_out, workspace, workspace_bytes, num_splits, device_error, stream);
}

int inkling_rel_attn_prefill(const void* q, const int32_t* cu_seqlens_q, const void* k_cache,
                             const void* v_cache, const int32_t* page_table, int32_t page_table_stride,
                             const int32_t* seq_lens, const float* rel_logits, int32_t B, int32_t T,
                             int32_t max_q_len, int32_t H_q, int32_t H_kv, int32_t D, int32_t page_size,
                             int32_t num_pages, int32_t R, int32_t window, float scale,
                             int32_t max_seq_len, void* out, float* lse_out, void* workspace,
                             size_t workspace_bytes, int32_t* device_error, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (B < 0 || T < 0 || max_q_len < 0 || max_seq_len < 0) return INKLING_ERR_ARG;
  if (!common_shape_ok(H_q, H_kv, D, page_size, num_pages, R, page_table_stride)) return INKLING_ERR_ARG;
  if (R % 4 != 0) return INKLING_ERR_ARG;
  if (!(scale == scale)) return INKLING_ERR_ARG;
  if (B == 0 || T == 0) return INKLING_OK;
  if (!q || !cu_seqlens_q || !k_cache || !v_cache || !page_table || !seq_lens || !rel_logits || !out)
    return INKLING_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(rel_logits, 16) || !aligned(page_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(cu_seqlens_q, 4) || !aligned(lse_out, 4) || !aligned(device_error, 4))
    return INKLING_ERR_ALIGN;
  const DevInfo di = device_info();
  if (di.ok != 1) return INKLING_ERR_DEVICE;
  PrefillCall c;
  c.q = q;
  c.cu_seqlens_q = cu_seqlens_q;
  c.k_cache = k_cache;
  c.v_cache = v_cache;
  c.page_table = page_table;
  c.pt_stride = page_table_stride;
  c.seq_lens = seq_lens;
  c.rel = rel_logits;
  c.B = B;
  c.T = T;
  c.max_q_len = max_q_len;
  c.H_q = H_q;
  c.H_kv = H_kv;
  c.D = D;
  c.P = page_size;
  c.num_pages = num_pages;
  c.R = R;
  c.window = window;
  c.scale = scale;
  c.max_seq_len = max_seq_len;
  c.out = out;
  c.lse_out = lse_out;
  c.dev_err = device_error;
  c.stream = static_cast<cudaStream_t>(stream);
  return launch_prefill(c);
}

int inkling_rel_attn_kv_append(const void* k_new, const void* v_new, const int32_t* cu_seqlens_q,
                               const int32_t* seq_lens, const int32_t* page_table,
                               int32_t page_table_stride, int32_t B, int32_t T, int32_t H_kv,
                               int32_t D, int32_t page_size, int32_t num_pages, void* k_cache,
                               void* v_cache, int32_t* device_error, void* stream) {
  if (B < 0 || T < 0 || H_kv <= 0 || (D != 64 && D != 128)) return INKLING_ERR_ARG;
  if (page_size <= 0 || page_size % 16 != 0 || page_size > 256) return INKLING_ERR_ARG;
  if (num_pages <= 0 || page_table_stride <= 0) return INKLING_ERR_ARG;
  if ((int64_t)page_table_stride * page_size > INT32_MAX) return INKLING_ERR_ARG;
  if (B == 0 || T == 0) return INKLING_OK;
  if (!k_new || !v_new || !cu_seqlens_q || !seq_lens || !page_table || !k_cache || !v_cache)
    return INKLING_ERR_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(cu_seqlens_q, 4) || !aligned(seq_lens, 4) ||
      !aligned(page_table, 4) || !aligned(device_error, 4))
    return INKLING_ERR_ALIGN;
  const DevInfo di = device_info();
  if (di.ok != 1) return INKLING_ERR_DEVICE;
  KvAppendCall c;
  c.k_new = k_new;
  c.v_new = v_new;
  c.cu_seqlens_q = cu_seqlens_q;
  c.seq_lens = seq_lens;
  c.page_table = page_table;
  c.pt_stride = page_table_stride;
  c.B = B;
  c.T = T;
  c.H_kv = H_kv;
  c.D = D;
  c.P = page_size;
  c.num_pages = num_pages;
  c.k_cache = k_cache;
  c.v_cache = v_cache;
  c.dev_err = device_error;
  c.stream = static_cast<cudaStream_t>(stream);
  return launch_kv_append(c);
}

int inkling_rel_attn_kv_conv_append(const void* k_new, const void* v_new,
                                    const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                                    const int32_t* page_table, int32_t page_table_stride,
                                    const float* conv_w_k, const float* conv_w_v, int32_t width,
                                    void* conv_state_k, void* conv_state_v,
                                    const int32_t* state_slots, int32_t num_slots, int32_t B,
                                    int32_t T, int32_t max_q_len, int32_t H_kv, int32_t D,
                                    int32_t page_size, int32_t num_pages, void* k_cache,
                                    void* v_cache, int32_t* device_error, void* stream) {
  if (B < 0 || T < 0 || H_kv <= 0 || (D != 64 && D != 128)) return INKLING_ERR_ARG;
  if (width < 1 || width > 8 || max_q_len < 0) return INKLING_ERR_ARG;
  if (page_size <= 0 || page_size % 16 != 0 || page_size > 256) return INKLING_ERR_ARG;
  if (num_pages <= 0 || page_table_stride <= 0) return INKLING_ERR_ARG;
  if ((int64_t)page_table_stride * page_size > INT32_MAX) return INKLING_ERR_ARG;
  if (width > 1 && num_slots <= 0) return INKLING_ERR_ARG;
  if (B == 0 || T == 0 || max_q_len == 0) return INKLING_OK;
  if (!k_new || !v_new || !cu_seqlens_q || !seq_lens || !page_table || !k_cache || !v_cache ||
      !conv_w_k || !conv_w_v)
    return INKLING_ERR_ARG;
  if (width > 1 && (!conv_state_k || !conv_state_v || !state_slots)) return INKLING_ERR_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(conv_state_k, 16) || !aligned(conv_state_v, 16) ||
      !aligned(conv_w_k, 4) || !aligned(conv_w_v, 4) || !aligned(state_slots, 4) ||
      !aligned(cu_seqlens_q, 4) || !aligned(seq_lens, 4) || !aligned(page_table, 4) ||
      !aligned(device_error, 4))
    return INKLING_ERR_ALIGN;
  const DevInfo di = device_info();
  if (di.ok != 1) return INKLING_ERR_DEVICE;
  KvConvCall c;
  c.k_new = k_new;
  c.v_new = v_new;
  c.w_k = conv_w_k;
  c.w_v = conv_w_v;
  c.state_k = conv_state_k;
  c.state_v = conv_state_v;
  c.state_slots = state_slots;
  c.cu_seqlens_q = cu_seqlens_q;
  c.seq_lens = seq_lens;
  c.page_table = page_table;
  c.pt_stride = page_table_stride;
  c.width = width;
  c.num_slots = width > 1 ? num_slots : 0;
  c.B = B;
  c.T = T;
  c.max_q_len = max_q_len;
  c.H_kv = H_kv;
  c.D = D;
  c.P = page_size;
  c.num_pages = num_pages;
  c.k_cache = k_cache;
  c.v_cache = v_cache;
  c.dev_err = device_error;
  c.stream = static_cast<cudaStream_t>(stream);
  return launch_kv_conv_append(c);
}

}  // extern "C"
