// Causal short convolution on K and V, fused ahead of the KV append.
//
// Operation: inkling_rel_attn_kv_conv_append in include/inkling_rel_attn.h
// (TensorRT-LLM PR #17062, "Architecture": two causal short convolutions
// inside attention, on K and on V, carrying per-request state across decode
// steps; "pyexecutor" row: a state pool with one row per request).
//
// y_t[c] = sum_j w[c, j] * x_{t-(w-1)+j}[c], depthwise over the H_kv * D
// channels of a token's row; the inputs before a request's new tokens come
// from its state row (its last w-1 inputs, oldest first), which is replaced
// by the last w-1 inputs of this call.  The convolved rows are written into
// the paged cache at the tokens' positions (as inkling_rel_attn_kv_append).
//
// Grid: x = channel blocks of 8 * 64 channels, y = (sequence, segment of
// 32..64 new tokens), z = K or V: small CTAs, many of them, all resident at
// once.  The launcher picks the segment length that spreads the CTAs most
// evenly over the SMs (for 4 x 2048 tokens: 54, eight CTAs on every SM
// rather than seven on most and six on the rest).  A
// thread owns 8 adjacent channels (16-byte loads and stores, 512 contiguous
// bytes per warp and token), keeps the last w-1 inputs in registers and walks
// its segment's tokens in order.  Its input rows arrive through a private
// shared-memory ring: while token t is convolved, the 16-byte row of token
// t + 6 is being copied (cp.async, one commit group per token), so six rows
// stay in flight without holding registers.  The cache slot advances with the
// position (one page-table read per page crossed, no division per token).  Only the first segment of a sequence reads the old state
// (later segments start w-1 tokens back inside the new tokens, since a segment
// is longer than any window), and the same thread that read a channel's old
// state writes its new one -- so the pool row is updated in place without a
// race between CTAs.  fp32 accumulation with the taps in order j = 0 .. w-1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "plan.cuh"

namespace ira {

constexpr int kConvThreads = 64;
constexpr int kConvSegMin = 32;  // new tokens per CTA: 32..64 (more than the widest window)
constexpr int kConvSegMax = 64;
constexpr int kConvSegCost = 8;  // a CTA's fixed work, in tokens, for the segment choice
constexpr int kConvChan = 8;     // channels per thread
constexpr int kRingSlots = 8;    // shared-memory ring slots per thread (one token row each)
constexpr int kRingAhead = 6;    // token rows in flight per thread

// 16-byte global -> shared copies (L2 only), committed and waited on per token
__device__ __forceinline__ void ring_copy(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void ring_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void ring_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct KvConvParams {
  const uint4* x[2];       // k_new, v_new: [T][C / 8] of 8 x bf16
  const float* w[2];       // [C][width]
  uint4* state[2];         // [num_slots][width - 1][C / 8]
  uint4* cache[2];         // [num_pages][P][C / 8]
  const int32_t* cu;
  const int32_t* seq_lens;
  const int32_t* page_table;
  const int32_t* slots;
  int32_t* dev_err;
  int B, T, pt_stride, P, num_pages, num_slots, C8, segs, seg_len;
};

// bf16 -> fp32 is exact: the bf16 bits are the high half of the float.
__device__ __forceinline__ void bf8_to_f8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 f8_to_bf8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&a);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int W>
__global__ void __launch_bounds__(kConvThreads)
    kv_conv_append_kernel(const __grid_constant__ KvConvParams p) {
  constexpr int NS = W - 1;  // state rows
  const int which = blockIdx.z;
  const int b = blockIdx.y / p.segs;
  const int seg = blockIdx.y - b * p.segs;
  const int c8 = blockIdx.x * kConvThreads + threadIdx.x;
  const bool reporter = threadIdx.x == 0 && blockIdx.x == 0 && which == 0;

  const int t0 = __ldg(p.cu + b);
  const int q_len = __ldg(p.cu + b + 1) - t0;
  const int s0 = seg * p.seg_len;
  if (q_len <= 0 || s0 >= q_len) return;
  const int L = __ldg(p.seq_lens + b);
  const int slot = NS > 0 ? __ldg(p.slots + b) : 0;
  if (q_len > L || t0 < 0 || t0 + q_len > p.T) {
    if (reporter && seg == 0) report(p.dev_err, INKLING_DEVERR_BAD_CHUNK);
    return;
  }
  if (NS > 0 && (slot < 0 || slot >= p.num_slots)) {
    if (reporter && seg == 0) report(p.dev_err, INKLING_DEVERR_BAD_SLOT);
    return;
  }
  if (seg == p.segs - 1 && s0 + p.seg_len < q_len && reporter)
    report(p.dev_err, INKLING_DEVERR_BAD_CHUNK);  // tokens past max_q_len are not written
  if (c8 >= p.C8) return;

  const uint4* __restrict__ x = p.x[which] + (size_t)t0 * p.C8 + c8;
  uint4* __restrict__ st = p.state[which] + (size_t)slot * NS * p.C8 + c8;
  uint4* __restrict__ cache = p.cache[which] + c8;
  const int32_t* pt_row = p.page_table + (size_t)b * p.pt_stride;

  // taps of this thread's 8 channels: 8 * W contiguous floats, read as 2 * W
  // 16-byte vectors when the tap array is 16-byte aligned
  float wt[kConvChan][W];
  {
    const float* wp = p.w[which] + (size_t)c8 * kConvChan * W;
    if ((reinterpret_cast<uintptr_t>(p.w[which]) & 15) == 0) {
#pragma unroll
      for (int v = 0; v < 2 * W; ++v) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(wp) + v);
        wt[(4 * v) / W][(4 * v) % W] = f.x;
        wt[(4 * v + 1) / W][(4 * v + 1) % W] = f.y;
        wt[(4 * v + 2) / W][(4 * v + 2) % W] = f.z;
        wt[(4 * v + 3) / W][(4 * v + 3) % W] = f.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < kConvChan; ++c)
#pragma unroll
        for (int j = 0; j < W; ++j) wt[c][j] = __ldg(wp + c * W + j);
    }
  }

  // the w-1 inputs before the segment: chunk-relative r = s0 - NS + j
  uint4 win[NS > 0 ? NS : 1];
#pragma unroll
  for (int j = 0; j < NS; ++j) {
    if (seg == 0) win[j] = st[(size_t)j * p.C8];  // r = j - NS < 0: state row j
    else win[j] = __ldcs(x + (size_t)(s0 - NS + j) * p.C8);
  }

  const int s1 = min(s0 + p.seg_len, q_len);
  int lp = (L - q_len + s0) / p.P;             // logical page of the segment's first token
  int in_page = (L - q_len + s0) - lp * p.P;   // its slot
  size_t row0 = 0;                             // first row of the current physical page
  bool page_ok = false;
  auto enter_page = [&]() {  // checks once per page crossed
    if (lp >= p.pt_stride) {
      page_ok = false;
      if (threadIdx.x == 0) report(p.dev_err, INKLING_DEVERR_SEQ_TOO_LONG);
      return;
    }
    const int page = __ldg(pt_row + lp);
    page_ok = page >= 0 && page < p.num_pages;
    if (!page_ok && threadIdx.x == 0) report(p.dev_err, INKLING_DEVERR_BAD_PAGE);
    row0 = (size_t)page * p.P * p.C8;
  };
  enter_page();
  // rolling prefetch: token t + kRingAhead is copied into this thread's slot
  // of a shared-memory ring while token t is convolved (one commit group per
  // token, so the wait for token t leaves kRingAhead copies in flight)
  __shared__ uint4 ring[kRingSlots][kConvThreads];
  const uint32_t my_slot0 = (uint32_t)__cvta_generic_to_shared(&ring[0][threadIdx.x]);
  constexpr uint32_t kSlotStride = kConvThreads * 16;
#pragma unroll
  for (int u = 0; u < kRingAhead; ++u) {
    if (s0 + u < s1) ring_copy(my_slot0 + u * kSlotStride, x + (size_t)(s0 + u) * p.C8);
    ring_commit();
  }
  int rs = 0;  // ring slot of token t
  for (int t = s0; t < s1; ++t) {
    {
      const int tn = t + kRingAhead;
      int sn = rs + kRingAhead;
      sn = sn >= kRingSlots ? sn - kRingSlots : sn;
      if (tn < s1) ring_copy(my_slot0 + sn * kSlotStride, x + (size_t)tn * p.C8);
      ring_commit();
    }
    ring_wait<kRingAhead>();
    const uint4 xt = ring[rs][threadIdx.x];
    rs = rs + 1 == kRingSlots ? 0 : rs + 1;
    float acc[kConvChan];
#pragma unroll
    for (int c = 0; c < kConvChan; ++c) acc[c] = 0.f;
#pragma unroll
    for (int j = 0; j < W; ++j) {
      float v[8];
      bf8_to_f8(j < NS ? win[j < NS ? j : 0] : xt, v);
#pragma unroll
      for (int c = 0; c < kConvChan; ++c) acc[c] = fmaf(wt[c][j], v[c], acc[c]);
    }
#pragma unroll
    for (int j = 0; j + 1 < NS; ++j) win[j] = win[j + 1];
    if (NS > 0) win[NS > 0 ? NS - 1 : 0] = xt;
    if (page_ok) cache[row0 + (size_t)in_page * p.C8] = f8_to_bf8(acc);
    if (++in_page == p.P && t + 1 < s1) {  // the next token starts the next logical page
      in_page = 0;
      ++lp;
      enter_page();
    }
  }
  ring_wait<0>();

  // new state: the last w-1 inputs of the sequence.  When all its new tokens
  // fall in this first segment, the window now holds exactly those (it began
  // as the old state and took every new token); otherwise they are the last
  // w-1 new tokens (q_len > seg_len >= w-1).
  if (seg == 0) {
    if (q_len <= p.seg_len) {
#pragma unroll
      for (int j = 0; j < NS; ++j) st[(size_t)j * p.C8] = win[j];
    } else {
#pragma unroll
      for (int j = 0; j < NS; ++j) st[(size_t)j * p.C8] = __ldcs(x + (size_t)(q_len - NS + j) * p.C8);
    }
  }
}

int launch_kv_conv_append(const KvConvCall& c) {
  KvConvParams prm;
  prm.x[0] = static_cast<const uint4*>(c.k_new);
  prm.x[1] = static_cast<const uint4*>(c.v_new);
  prm.w[0] = c.w_k;
  prm.w[1] = c.w_v;
  prm.state[0] = static_cast<uint4*>(c.state_k);
  prm.state[1] = static_cast<uint4*>(c.state_v);
  prm.cache[0] = static_cast<uint4*>(c.k_cache);
  prm.cache[1] = static_cast<uint4*>(c.v_cache);
  prm.cu = c.cu_seqlens_q;
  prm.seq_lens = c.seq_lens;
  prm.page_table = c.page_table;
  prm.slots = c.state_slots;
  prm.dev_err = c.dev_err;
  prm.B = c.B;
  prm.T = c.T;
  prm.pt_stride = c.pt_stride;
  prm.P = c.P;
  prm.num_pages = c.num_pages;
  prm.num_slots = c.num_slots;
  prm.C8 = c.H_kv * c.D / kConvChan;
  // segment length: the fewest CTAs on the busiest SM, weighted by the
  // tokens each walks plus its fixed work
  {
    const int nsm = sm_count();
    const int64_t cblocks = (prm.C8 + kConvThreads - 1) / kConvThreads;
    int64_t best = -1;
    prm.seg_len = kConvSegMax;
    for (int len = kConvSegMax; len >= kConvSegMin; --len) {
      const int64_t segs = (c.max_q_len + len - 1) / len;
      if (len < kConvSegMax && (int64_t)c.B * segs > 65535) break;  // grid y limit: keep longer segments
      const int64_t ctas = 2 * cblocks * (int64_t)c.B * segs;
      const int64_t cost = (ctas + nsm - 1) / nsm * (len + kConvSegCost);
      if (best < 0 || cost < best) {
        best = cost;
        prm.seg_len = len;
      }
    }
  }
  prm.segs = (c.max_q_len + prm.seg_len - 1) / prm.seg_len;
  const int64_t gy = (int64_t)c.B * prm.segs;  // (sequence, segment) pairs
  if (gy <= 0 || gy > 65535) return INKLING_ERR_ARG;
  const dim3 grid((prm.C8 + kConvThreads - 1) / kConvThreads, (unsigned)gy, 2);
  switch (c.width) {
    case 1: kv_conv_append_kernel<1><<<grid, kConvThreads, 0, c.stream>>>(prm); break;
    case 2: kv_conv_append_kernel<2><<<grid, kConvThreads, 0, c.stream>>>(prm); break;
    case 3: kv_conv_append_kernel<3><<<grid, kConvThreads, 0, c.stream>>>(prm); break;
    case 4: kv_conv_append_kernel<4><<<grid, kConvThreads, 0, c.stream>>>(prm); break;
    case 5: kv_conv_append_kernel<5><<<grid, kConvThreads, 0, c.stream>>>(prm); break;
    case 6: kv_conv_append_kernel<6><<<grid, kConvThreads, 0, c.stream>>>(prm); break;
    case 7: kv_conv_append_kernel<7><<<grid, kConvThreads, 0, c.stream>>>(prm); break;
    case 8: kv_conv_append_kernel<8><<<grid, kConvThreads, 0, c.stream>>>(prm); break;
    default: return INKLING_ERR_ARG;
  }
  return cudaGetLastError() == cudaSuccess ? INKLING_OK : INKLING_ERR_CUDA;
}

}  // namespace ira
