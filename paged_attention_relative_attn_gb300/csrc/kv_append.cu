// KV append: write the new tokens' K and V rows into the paged cache.
//
// Operation: inkling_rel_attn_kv_append in include/inkling_rel_attn.h
// (TensorRT-LLM PR #17062, commit notes: the attention op writes the step's
// K/V into the paged cache before reading it).
//
// One warp per token: find its sequence (binary search over cu_seqlens_q),
// its position (the last q_len tokens of the sequence), its physical page and
// slot, then copy the token's K row and V row (H_kv * D bf16 each, contiguous
// in both the input and the cache) with 16-byte loads and stores, coalesced
// across the warp.  The inputs are read once (streaming loads); the cache rows
// are written with ordinary stores so that the attention kernel that follows
// finds them in L2.
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "plan.cuh"

namespace ira {

constexpr int kAppendThreads = 256;

struct KvAppendParams {
  const uint4* k_new;
  const uint4* v_new;
  const int32_t* cu;
  const int32_t* seq_lens;
  const int32_t* page_table;
  uint4* k_cache;
  uint4* v_cache;
  int32_t* dev_err;
  int B, T, pt_stride, P, num_pages, row16;  // row16: 16-byte units per token row
};

__global__ void __launch_bounds__(kAppendThreads)
    kv_append_kernel(const __grid_constant__ KvAppendParams p) {
  const int lane = threadIdx.x & 31;
  const int t = (int)((blockIdx.x * (unsigned)kAppendThreads + threadIdx.x) >> 5);
  if (t >= p.T) return;
  // the sequence owning token t: the last b with cu[b] <= t
  if (!(__ldg(p.cu) <= t && t < __ldg(p.cu + p.B))) {
    if (lane == 0) report(p.dev_err, INKLING_DEVERR_BAD_CHUNK);
    return;
  }
  int lo = 0, hi = p.B;  // cu[lo] <= t < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.cu + mid) <= t) lo = mid;
    else hi = mid;
  }
  const int b = lo;
  const int t0 = __ldg(p.cu + b);
  const int q_len = __ldg(p.cu + b + 1) - t0;
  const int L = __ldg(p.seq_lens + b);
  const int pos = L - q_len + (t - t0);
  if (q_len > L || pos < 0) {
    if (lane == 0) report(p.dev_err, INKLING_DEVERR_BAD_CHUNK);
    return;
  }
  const int lp = pos / p.P;
  if (lp >= p.pt_stride) {
    if (lane == 0) report(p.dev_err, INKLING_DEVERR_SEQ_TOO_LONG);
    return;
  }
  const int page = __ldg(p.page_table + (size_t)b * p.pt_stride + lp);
  if (page < 0 || page >= p.num_pages) {
    if (lane == 0) report(p.dev_err, INKLING_DEVERR_BAD_PAGE);
    return;
  }
  const size_t dst = ((size_t)page * p.P + (pos - lp * p.P)) * p.row16;
  const size_t src = (size_t)t * p.row16;
  const uint4* __restrict__ kn = p.k_new + src;
  const uint4* __restrict__ vn = p.v_new + src;
  uint4* __restrict__ kd = p.k_cache + dst;
  uint4* __restrict__ vd = p.v_cache + dst;
  // four 16-byte units of K and four of V per lane in flight before storing
  int u = lane;
  for (; u + 96 < p.row16; u += 128) {
    uint4 k[4], v[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      k[x] = __ldcs(kn + u + 32 * x);
      v[x] = __ldcs(vn + u + 32 * x);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      kd[u + 32 * x] = k[x];
      vd[u + 32 * x] = v[x];
    }
  }
  for (; u < p.row16; u += 32) {
    const uint4 k = __ldcs(kn + u);
    const uint4 v = __ldcs(vn + u);
    kd[u] = k;
    vd[u] = v;
  }
}

int launch_kv_append(const KvAppendCall& c) {
  KvAppendParams prm;
  prm.k_new = static_cast<const uint4*>(c.k_new);
  prm.v_new = static_cast<const uint4*>(c.v_new);
  prm.cu = c.cu_seqlens_q;
  prm.seq_lens = c.seq_lens;
  prm.page_table = c.page_table;
  prm.k_cache = static_cast<uint4*>(c.k_cache);
  prm.v_cache = static_cast<uint4*>(c.v_cache);
  prm.dev_err = c.dev_err;
  prm.B = c.B;
  prm.T = c.T;
  prm.pt_stride = c.pt_stride;
  prm.P = c.P;
  prm.num_pages = c.num_pages;
  prm.row16 = c.H_kv * c.D * 2 / 16;
  const int64_t threads = (int64_t)c.T * 32;
  const int64_t blocks = (threads + kAppendThreads - 1) / kAppendThreads;
  if (blocks > INT32_MAX) return INKLING_ERR_ARG;
  kv_append_kernel<<<(unsigned)blocks, kAppendThreads, 0, c.stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? INKLING_OK : INKLING_ERR_CUDA;
}

}  // namespace ira
