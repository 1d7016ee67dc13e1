// Split-KV paged decode with a learned relative-position bias, and the
// log-sum-exp merge of the splits.
//
// Operation: inkling_rel_attn_decode in include/inkling_rel_attn.h (Support
// Inkling-NVFP4 model, TensorRT-LLM PR #17062, "Architecture" and
// "Implementation"; split-KV from Fail fast on Inkling's unsupported GPU
// architectures, vLLM PR #51560, "Changes").
//
// Design: a persistent grid (two CTAs per SM) walks work items
// (sequence, KV head, split).  Each CTA has
//  * a producer warp (warp 4) that takes the next item (static stride, or an
//    atomic counter when splits make items uneven), publishes the item's key
//    range to the consumers through a small shared-memory ring, and walks the
//    range in tiles of <= 64 keys: it looks the physical page up in the page
//    table and issues TMA loads of that KV head's K and V rows (box = 64 dims x
//    1 head x rows x 1 page, 128-byte swizzle) into a ring of stages guarded by
//    full/empty mbarriers.  The first tile of a range starts mid-page so its
//    box runs past the page end (zero-filled, never fetched); the last tile is
//    placed so its box starts before the page (also zero-filled): only the
//    bytes of visible keys are read.  The ring runs across item boundaries, so
//    the next item's K/V stream in while the consumers finish the current one.
//  * four consumer warps that each own 16 rows of every tile and compute the
//    transposed products S^T = K Q^T and O^T += V^T P^T with mma.sync m16n8k16
//    (the rows of an item -- the GQA group's query heads, or (token, head)
//    pairs of a token group for multi-token decode -- are the N side, one or
//    two 8-wide n-tiles, so M is never padded), add the bias read from L2
//    (the producer prefetches each item's rel_logits rows there; each tile's
//    values are loaded one tile ahead), mask, and keep an online softmax per
//    row with warp shuffles over the keys (the row max is re-reduced only when
//    a score exceeds the running one by more than a factor 2^8).  P goes from the accumulator layout
//    to the B-operand layout with movmatrix.  With one n-tile the q fragments
//    stay in registers for the whole item; with two they are read from the
//    item's shared-memory slot (rows padded to 272 bytes, one ldmatrix per
//    k-step), which keeps the two-n-tile consumer inside its registers.  At the end of an item the four
//    warps' (m, l, O) are combined through shared memory (one buffer per warp,
//    or two buffers in two rounds where that leaves room for a third stage)
//    and written as the final bf16 output or, when the sequence spans several
//    splits, as a normalised fp32 partial plus its lse for the merge kernel.
// The kernel is launched with programmatic stream serialization: its CTAs may
// start their set-up while the previous kernel on the stream finishes, and wait
// (griddepcontrol) for it before reading or writing anything in global memory.
// Reduction order depends only on logical key positions and host scalars,
// never on page ids or on which CTA ran an item, so results are bit-identical
// under any physical page permutation and any schedule.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "internal.h"
#include "plan.cuh"
#include "ptx.cuh"

namespace ira {

constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kDecodeThreads = kConsumerThreads + 32;
constexpr int kItemSlots = 3;
constexpr float kMaxSlack = 8.f;  // log2 units: scores may exceed the exponent base by 2^8
#ifndef INKLING_DECODE_CTAS_PER_SM
#define INKLING_DECODE_CTAS_PER_SM 2
#endif
#ifndef INKLING_DECODE_SMEM_BUDGET_KB
#define INKLING_DECODE_SMEM_BUDGET_KB 111
#endif
#ifndef INKLING_DECODE_MAX_STAGES
#define INKLING_DECODE_MAX_STAGES 4
#endif
#ifndef INKLING_DECODE_BALANCED
#define INKLING_DECODE_BALANCED 1
#endif
constexpr int kCtasPerSm = INKLING_DECODE_CTAS_PER_SM;

struct DecodeParams {
  CUtensorMap tmap_k;  // [num_pages][P][H_kv][D] bf16, box {64, 1, BH, 1}
  CUtensorMap tmap_v;
  const __nv_bfloat16* q;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const float* rel;
  __nv_bfloat16* out;
  float* lse_out;
  float* o_part;
  float* lse_part;
  int32_t* dev_err;
  int32_t* counter;  // dynamic scheduling (zeroed before launch), or nullptr
  int B, pt_stride, H_q, H_kv, G, P, num_pages, R, window;
  int QL, TG, NG;  // query tokens per sequence, tokens per item (group), groups per sequence
  int S, chunk, stages;
  int bias_prefetch;  // rel_logits rows are 16-byte aligned: L2 prefetch allowed
  float scale_log2;
};

// Visible key range [lo, pos] of token group `grp` of a sequence -- its
// queries are tokens first .. first + tn - 1 of the sequence's last QL tokens,
// at positions pos - tn + 1 .. pos; lo is the first one's window start -- and
// the sequence's split count (the same for all its groups: the largest any
// group needs).  Identical in the decode and merge kernels.  A sequence with
// fewer than QL tokens has nothing visible (the host validates lengths; the
// kernel reports it).
struct SeqPlan {
  int L, pos, lo, nvis, n_s, first, tn;
};
template <bool MULTI>
__device__ __forceinline__ SeqPlan seq_plan(int L, int pt_stride, int P, int window, int chunk,
                                            int S, int QL, int TG, int NG, int grp) {
  SeqPlan s;
  const int cap = pt_stride * P;
  if (L > cap) L = cap;
  if (L < 0) L = 0;
  s.L = L;
  if constexpr (!MULTI) {  // one query token, at position L - 1
    s.first = 0;
    s.tn = 1;
    s.pos = L - 1;
    s.lo = (window > 0) ? max(0, s.pos - window + 1) : 0;
    s.nvis = L > 0 ? s.pos - s.lo + 1 : 0;
    const int n = (s.nvis + chunk - 1) / chunk;
    s.n_s = n > S ? S : n;
    return s;
  }
  s.first = grp * TG;
  s.tn = min(TG, QL - s.first);
  const bool ok = L >= QL;
  s.pos = L - QL + s.first + s.tn - 1;
  s.lo = (window > 0) ? max(0, s.pos - s.tn + 1 - window + 1) : 0;
  s.nvis = ok ? s.pos - s.lo + 1 : 0;
  int nmax = 0;
  if (ok) {
    for (int g = 0; g < NG; ++g) {  // every group's key count
      const int tn = min(TG, QL - g * TG);
      const int pos = L - QL + g * TG + tn - 1;
      const int lo = (window > 0) ? max(0, pos - tn + 1 - window + 1) : 0;
      nmax = max(nmax, (pos - lo + chunk) / chunk);
    }
  }
  s.n_s = nmax > S ? S : nmax;
  return s;
}

// One work item as published by the producer: keys [a, e] of sequence b,
// KV head hkv, token group starting at packed token t0 with tn tokens (the
// last at position pos), split `split` of n_s (a > e: nothing in this split).
struct ItemRec {
  int b, hkv, split, n_s, a, e, pos, nvis, t0, tn;
};

// Shared-memory layout (byte offsets from the 1024-aligned base), computed
// identically on host and device.
struct DecodeSmem {
  int stage_bytes, stages, slot_bytes, ring_off, comb_off, pre_off, bar_off, total;
  __host__ __device__ DecodeSmem(int D, int G, int NT, int stages_, int n_prefix, int comb_slots) {
    stage_bytes = 2 * (D / 64) * kHalfBytes;
    stages = stages_;
    // item record + q rows; with two n-tiles the rows are padded by 16 bytes
    // (read by ldmatrix per k-step: eight rows then fall in distinct banks)
    const int qpitch = NT == 2 ? D * 2 + 16 : D * 2;
    const int qrows = NT == 2 ? 16 : G;  // two n-tiles: ldmatrix reads all 16 rows
    slot_bytes = 128 + ((qrows * qpitch + 127) / 128) * 128;
    ring_off = stages * stage_bytes;
    comb_off = ring_off + kItemSlots * slot_bytes;
    const int comb_bytes = comb_slots * G * (D + 4) * 4 + 2 * kConsumerWarps * 8 * NT * 4;
    pre_off = comb_off + ((comb_bytes + 127) / 128) * 128;
    bar_off = pre_off + ((n_prefix * 4 + 127) / 128) * 128;
    total = bar_off + (2 * stages + 2 * kItemSlots) * 8 + 16;
  }
};

// MULTI: several query tokens per sequence (the rows of an item are
// (token, head) pairs, each with its own position, mask and bias row); the
// single-token instantiations keep the plain per-key mask.
// COMB2: the item combine in two rounds through two O buffers instead of one
// per consumer warp (the smaller buffer leaves room for a third stage).
template <int D, int NT, int BH, bool MULTI, bool COMB2>
__global__ void __launch_bounds__(kDecodeThreads, kCtasPerSm)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int HALVES = D / 64;
  constexpr int TILE_BYTES = HALVES * kHalfBytes;
  constexpr int KS = D / 16;  // k-steps of QK^T, m-tiles of PV
  // With one n-tile, QK^T accumulates over two chains (even / odd k-steps):
  // the chain of dependent MMAs halves; two n-tiles already give two chains.
  constexpr bool kTwoChains = NT == 1;
  // O is rescaled only when some row's running max moved (warp vote); with
  // one n-tile of multi-token rows the vote costs more than it saves.
  constexpr bool kLazyRescale = !(MULTI && NT == 1);
  constexpr int HP = 8 * NT;  // padded heads per group
  // Two n-tiles: the q fragments are read from the item slot at every k-step
  // (ldmatrix) instead of being held in 32 registers for the whole item, and
  // the slot is released when the item's last QK^T is done.
  constexpr bool kQSmem = NT == 2;
  constexpr int QP = kQSmem ? D * 2 + 16 : D * 2;  // bytes per q row in a slot

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = p.G;
  const int S = p.S;
  const int NR = p.TG * G;   // rows (token, head) of a full item
  const bool dense = S > 1;  // items enumerated through a per-sequence prefix sum
  constexpr int kCombSlots = COMB2 ? 2 : kConsumerWarps;
  const DecodeSmem L(D, NR, NT, p.stages, dense ? p.B + 1 : 0, kCombSlots);
  const int stages = L.stages;
  const int STAGE_BYTES = L.stage_bytes;

  float* comb_o = reinterpret_cast<float*>(smem + L.comb_off);  // [comb_slots][NR][D+4]
  float* comb_m = comb_o + kCombSlots * NR * (D + 4);             // [4][HP]
  float* comb_l = comb_m + kConsumerWarps * HP;                   // [4][HP]
  int* prefix = reinterpret_cast<int*>(smem + L.pre_off);         // [B+1] items before b
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  // full[s] = bars[s], empty[s] = bars[stages + s]; item ring after
  uint64_t* rfull = bars + 2 * stages;
  uint64_t* rempty = rfull + kItemSlots;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(rempty + kItemSlots);
  auto slot_rec = [&](int s) { return reinterpret_cast<ItemRec*>(smem + L.ring_off + s * L.slot_bytes); };
  auto slot_q = [&](int s) { return smem + L.ring_off + s * L.slot_bytes + 128; };

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[stages + s]), kConsumerWarps);
    }
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(smem_u32(&rfull[i]), 1);
      mbar_init(smem_u32(&rempty[i]), kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if constexpr (kQSmem) {
    for (int i = tid; i < kItemSlots * (L.slot_bytes - 128) / 16; i += kDecodeThreads) {
      const int s = i / ((L.slot_bytes - 128) / 16), o = i - s * ((L.slot_bytes - 128) / 16);
      *reinterpret_cast<uint4*>(slot_q(s) + 16 * o) = make_uint4(0, 0, 0, 0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  // launched with programmatic stream serialization: the set-up above may
  // overlap the previous kernel on the stream; nothing it wrote is read (or
  // overwritten) before that kernel has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // =================================================================== producer
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      tmap_prefetch(&p.tmap_k);
      tmap_prefetch(&p.tmap_v);
    }
    const uint64_t pol = policy_evict_first();

    // dense item space: prefix[b] = items of sequences < b (H_kv * NG * max(n_s, 1) each)
    int total = p.B * p.H_kv * p.NG;
    if (dense) {
      int carry = 0;
      for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int cnt = 0;
        if (b < p.B) {
          const SeqPlan sp = seq_plan<MULTI>(__ldg(p.seq_lens + b), p.pt_stride, p.P, p.window,
                                             p.chunk, S, p.QL, p.TG, p.NG, 0);
          cnt = p.H_kv * p.NG * max(sp.n_s, 1);
        }
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += v;
        }
        if (b < p.B) prefix[b] = carry + incl - cnt;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) prefix[p.B] = carry;
      total = carry;
      __syncwarp();
    }

    // item id -> (b, hkv, token group, split) and its key range
    auto locate = [&](int id, int& b, int& hkv, int& grp, int& split) {
      if (dense) {
        int lo = 0, hi = p.B - 1;  // last b with prefix[b] <= id
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (prefix[mid] <= id) lo = mid;
          else hi = mid - 1;
        }
        b = lo;
        const int rest = id - prefix[b];
        if constexpr (MULTI) {
          const int nsb = (prefix[b + 1] - prefix[b]) / (p.H_kv * p.NG);
          hkv = rest / (p.NG * nsb);
          const int rest2 = rest - hkv * p.NG * nsb;
          grp = rest2 / nsb;
          split = rest2 - grp * nsb;
        } else {
          const int nsb = (prefix[b + 1] - prefix[b]) / p.H_kv;
          hkv = rest / nsb;
          grp = 0;
          split = rest - hkv * nsb;
        }
      } else if constexpr (MULTI) {
        b = id / (p.H_kv * p.NG);
        const int rest = id - b * p.H_kv * p.NG;
        hkv = rest / p.NG;
        grp = rest - hkv * p.NG;
        split = 0;
      } else {
        b = id / p.H_kv;
        hkv = id - b * p.H_kv;
        grp = 0;
        split = 0;
      }
    };
    int n_static = 0;
    auto next_id = [&]() -> int {
      int id;
      if (p.counter) {
        id = 0;
        if (lane == 0) id = atomicAdd(p.counter, 1);
        id = __shfl_sync(0xffffffffu, id, 0);
      } else {
        id = blockIdx.x + (n_static++) * gridDim.x;
      }
      return id;
    };
    auto resolve = [&](int id, int Lraw) -> ItemRec {
      ItemRec r;
      r.b = -1;
      r.hkv = r.split = r.n_s = r.a = r.e = r.pos = r.nvis = r.t0 = r.tn = 0;
      if (id >= total) return r;
      int grp;
      locate(id, r.b, r.hkv, grp, r.split);
      const SeqPlan sp =
          seq_plan<MULTI>(Lraw, p.pt_stride, p.P, p.window, p.chunk, S, p.QL, p.TG, p.NG, grp);
      if (lane == 0 && r.hkv == 0 && r.split == 0 && grp == 0) {
        if (Lraw > p.pt_stride * p.P) report(p.dev_err, INKLING_DEVERR_SEQ_TOO_LONG);
        if (MULTI && Lraw < p.QL) report(p.dev_err, INKLING_DEVERR_BAD_CHUNK);
      }
      r.n_s = sp.n_s;
      r.pos = sp.pos;
      r.nvis = sp.nvis;
      r.t0 = r.b * p.QL + sp.first;
      r.tn = sp.tn;
      r.a = sp.lo + r.split * p.chunk;
      if constexpr (MULTI) r.e = (r.split >= sp.n_s - 1) ? sp.pos : min(r.a + p.chunk - 1, sp.pos);
      else r.e = (r.split >= sp.n_s - 1) ? sp.pos : r.a + p.chunk - 1;
      return r;
    };
    auto seq_len_of = [&](int id) -> int {  // issued early, consumed later
      if (id >= total) return 0;
      int b, h, gr, s;
      locate(id, b, h, gr, s);
      return __ldg(p.seq_lens + b);
    };

    int ki = 0;  // items published
    bool ok = true;
    // publish an item: its record and q rows into ring slot ki % kItemSlots,
    // and a prefetch of its bias rows into L2
    auto publish = [&](const ItemRec& r) -> bool {
      const int slot = ki % kItemSlots;
      bool good = true;
      if (ki >= kItemSlots && lane == 0)
        good = mbar_wait(smem_u32(&rempty[slot]), ((ki / kItemSlots) - 1) & 1, abort_flag);
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) return false;
      if (lane == 0) {
        *slot_rec(slot) = r;
        const uint32_t fb = smem_u32(&rfull[slot]);
        if (r.b >= 0 && r.nvis > 0) {
          // q rows (token i, head gh) in order i * G + gh: one copy per token
          const uint32_t tbytes = G * D * 2;
          if constexpr (kQSmem) {  // one copy per row, at the padded pitch
            const int ntok = MULTI ? r.tn : 1;
            mbar_arrive_expect_tx(fb, ntok * tbytes);
            for (int i = 0; i < ntok; ++i) {
              const size_t tok = MULTI ? (size_t)(r.t0 + i) : (size_t)r.b;
              for (int gh = 0; gh < G; ++gh)
                bulk_load(smem_u32(slot_q(slot)) + (i * G + gh) * QP,
                          p.q + (tok * p.H_q + r.hkv * G + gh) * D, D * 2, fb);
            }
          } else if constexpr (MULTI) {
            mbar_arrive_expect_tx(fb, r.tn * tbytes);
            for (int i = 0; i < r.tn; ++i)
              bulk_load(smem_u32(slot_q(slot)) + i * tbytes,
                        p.q + ((size_t)(r.t0 + i) * p.H_q + r.hkv * G) * D, tbytes, fb);
          } else {
            mbar_arrive_expect_tx(fb, tbytes);
            bulk_load(smem_u32(slot_q(slot)), p.q + ((size_t)r.b * p.H_q + r.hkv * G) * D, tbytes,
                      fb);
          }
        } else {
          mbar_arrive(fb);
        }
      }
      if constexpr (MULTI) {
        if (r.b >= 0 && r.nvis > 0 && r.a <= r.e && p.bias_prefetch && lane < r.tn * G) {
          const int i = lane / G, gh = lane - (lane / G) * G;
          const int pr = r.pos - (r.tn - 1) + i;  // this row's position
          const int dlo = max(0, min(pr - r.e, p.R - 1)) & ~3;
          const int dhi = min(max(0, min(pr - r.a, p.R - 1)) + 4, p.R) & ~3;
          const float* row = p.rel + ((size_t)(r.t0 + i) * p.H_q + r.hkv * G + gh) * p.R;
          if (dhi > dlo) bulk_prefetch_l2(row + dlo, (uint32_t)(dhi - dlo) * 4);
        }
      } else if (r.b >= 0 && r.nvis > 0 && p.bias_prefetch && lane < G) {
        const int dlo = min(r.pos - r.e, p.R - 1) & ~3;
        const int dhi = min(min(r.pos - r.a, p.R - 1) + 4, p.R) & ~3;
        const float* row = p.rel + ((size_t)r.b * p.H_q + r.hkv * G + lane) * p.R;
        if (dhi > dlo) bulk_prefetch_l2(row + dlo, (uint32_t)(dhi - dlo) * 4);
      }
      ++ki;
      return true;
    };

    // page ids, fetched 32 at a time per item; the next item's first batch is
    // loaded while the current item's tiles are issued
    int cur_base = 0, cur_page = 0, nxt_base = 0, nxt_page = 0;
    const int32_t* cur_row = p.page_table;
    const int32_t* nxt_row = p.page_table;
    auto batch_load = [&](const int32_t* row, int base) -> int {
      const int idx = base + lane;
      return (idx < p.pt_stride) ? __ldg(row + idx) : 0;
    };
    auto page_of = [&](int lp) -> int {  // warp-uniform
      if (lp < cur_base || lp >= cur_base + 32) {
        cur_base = lp;
        cur_page = batch_load(cur_row, lp);
      }
      return __shfl_sync(0xffffffffu, cur_page, lp - cur_base);
    };

    int pid = next_id();
    int pL = seq_len_of(pid);
    ItemRec cur = resolve(pid, pL);
    ok = publish(cur);
    if (ok && cur.b >= 0) {
      cur_row = p.page_table + (size_t)cur.b * p.pt_stride;
      cur_base = cur.a / p.P;
      cur_page = batch_load(cur_row, cur_base);
      pid = next_id();
      pL = seq_len_of(pid);
    }
    int kt = 0;  // tiles issued (global over items)
    while (ok && cur.b >= 0) {
      ItemRec nxt;
      bool nxt_done = false;
      auto do_next = [&]() {  // resolve + publish the following item, prefetch its pages
        nxt = resolve(pid, pL);
        ok = publish(nxt);
        if (ok && nxt.b >= 0) {
          nxt_row = p.page_table + (size_t)nxt.b * p.pt_stride;
          nxt_base = nxt.a / p.P;
          nxt_page = batch_load(nxt_row, nxt_base);
          pid = next_id();
          pL = seq_len_of(pid);
        }
        nxt_done = true;
      };
      int local = 0;
      if (cur.nvis > 0 && (!MULTI || cur.a <= cur.e)) {
        if constexpr (BH == 64) {
          PlanBig plan(cur.a, cur.e, p.P);
          while (!plan.done()) {
            const int st = kt % stages;
            if (kt >= stages && lane == 0)
              ok = mbar_wait(smem_u32(&bars[stages + st]), ((kt / stages) - 1) & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            int lp, slot0;
            plan.next(lp, slot0);
            const int page = page_of(lp);
            if (lane == 0) {
              if (page < 0 || page >= p.num_pages) report(p.dev_err, INKLING_DEVERR_BAD_PAGE);
              const uint32_t kdst = smem_u32(smem + st * STAGE_BYTES);
              const uint32_t vdst = kdst + TILE_BYTES;
              const uint32_t fb = smem_u32(&bars[st]);
              mbar_arrive_expect_tx(fb, 2 * TILE_BYTES);
#pragma unroll
              for (int h = 0; h < HALVES; ++h) {
                tma_load_4d(kdst + h * kHalfBytes, &p.tmap_k, fb, h * 64, cur.hkv, slot0, page, pol);
                tma_load_4d(vdst + h * kHalfBytes, &p.tmap_v, fb, h * 64, cur.hkv, slot0, page, pol);
              }
            }
            __syncwarp();
            ++kt;
            if (++local == 2) do_next();
            if (!ok) break;
          }
        } else {
          PlanSmall plan(cur.a, cur.e);
          while (!plan.done()) {
            const int st = kt % stages;
            if (kt >= stages && lane == 0)
              ok = mbar_wait(smem_u32(&bars[stages + st]), ((kt / stages) - 1) & 1, abort_flag);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            const Tile t = plan.next();
            int nbox = 0;
            int pages[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int k0 = t.jbase + 16 * c;
              const bool need = (k0 <= t.khi) && (k0 + 15 >= t.klo);
              pages[c] = need ? page_of(k0 / p.P) : 0;
              nbox += need ? 1 : 0;
            }
            if (lane == 0) {
              const uint32_t kdst = smem_u32(smem + st * STAGE_BYTES);
              const uint32_t vdst = kdst + TILE_BYTES;
              const uint32_t fb = smem_u32(&bars[st]);
              mbar_arrive_expect_tx(fb, nbox * 2 * HALVES * 16 * 128);
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const int k0 = t.jbase + 16 * c;
                if (!((k0 <= t.khi) && (k0 + 15 >= t.klo))) continue;
                if (pages[c] < 0 || pages[c] >= p.num_pages)
                  report(p.dev_err, INKLING_DEVERR_BAD_PAGE);
                const int slot = k0 % p.P;
#pragma unroll
                for (int h = 0; h < HALVES; ++h) {
                  tma_load_4d(kdst + h * kHalfBytes + c * 16 * 128, &p.tmap_k, fb, h * 64, cur.hkv,
                              slot, pages[c], pol);
                  tma_load_4d(vdst + h * kHalfBytes + c * 16 * 128, &p.tmap_v, fb, h * 64, cur.hkv,
                              slot, pages[c], pol);
                }
              }
            }
            __syncwarp();
            ++kt;
            if (++local == 2) do_next();
            if (!ok) break;
          }
        }
      }
      if (!ok) break;
      if (!nxt_done) do_next();
      if (!ok) break;
      cur = nxt;
      cur_row = nxt_row;
      cur_base = nxt_base;
      cur_page = nxt_page;
    }
    if (!ok && lane == 0) {
      report(p.dev_err, INKLING_DEVERR_TIMEOUT);
      // drain: copies already issued into stages / slots nobody consumes
      for (int j = max(0, kt - stages); j < kt; ++j)
        mbar_wait_drain(smem_u32(&bars[j % stages]), (j / stages) & 1);
      for (int j = max(0, ki - kItemSlots); j < ki; ++j)
        mbar_wait_drain(smem_u32(&rfull[j % kItemSlots]), (j / kItemSlots) & 1);
    }
    return;
  }

  // =================================================================== consumers
  const int g = lane >> 2;  // accumulator row group
  const int c4 = lane & 3;  // thread in group
  const int r0 = warp * 16;
  const int k_row = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;  // K: matrices (rows, chunk)
  const int k_chi = lane >> 4;
  const int v_row = r0 + (lane & 7) + ((lane >> 4) & 1) * 8;  // V^T: matrices (chunk, rows)
  const int v_chi = (lane >> 3) & 1;
  const int sw = lane & 7;  // (row & 7) for the 128-byte swizzle
  const float sl2 = p.scale_log2;
  const int R = p.R;

  int kt = 0;
  bool ok = true;
  for (int ki = 0;; ++ki) {
    // ---- next item: record and q rows from the ring
    const int slot = ki % kItemSlots;
    if (!mbar_wait_warp(smem_u32(&rfull[slot]), (ki / kItemSlots) & 1, abort_flag)) {
      ok = false;
      break;
    }
    const ItemRec r = *slot_rec(slot);
    const bool final_out = r.n_s <= 1;
    const int NRi = MULTI ? r.tn * G : G;  // live rows of this item
    uint32_t qf[kQSmem ? 1 : KS][NT][2];
    const uint32_t q_smem = smem_u32(slot_q(slot));
    if (!kQSmem && r.b >= 0 && r.nvis > 0) {
      const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(slot_q(slot));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int head = nt * 8 + g;
        const bool live = head < NRi;
        const __nv_bfloat16* qrow = qs + (live ? head : 0) * D;
#pragma unroll
        for (int ks = 0; ks < (kQSmem ? 0 : KS); ++ks) {
          qf[ks][nt][0] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4) : 0u;
          qf[ks][nt][1] = live ? *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4 + 8) : 0u;
        }
      }
    }
    __syncwarp();
    // slot free: q is in registers (two n-tiles: once the item's QK^T is done)
    auto release_slot = [&]() {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&rempty[slot]));
    };
    if (!kQSmem || r.b < 0) release_slot();
    if (r.b < 0) break;

    // output row of item row rr = (token i, head gh)
    auto out_row = [&](int rr) -> size_t {
      if constexpr (MULTI) {
        const int i = rr / G;
        return (size_t)(r.t0 + i) * p.H_q + r.hkv * G + (rr - i * G);
      } else {
        return (size_t)r.b * p.H_q + r.hkv * G + rr;
      }
    };
    if (kQSmem && (r.nvis == 0 || (MULTI && r.a > r.e))) release_slot();
    if (r.nvis == 0) {  // nothing visible: out = 0, lse = -inf
      for (int i = tid; i < NRi * D; i += kConsumerThreads) {
        const int rr = i / D, d = i - rr * D;
        const size_t row = out_row(rr);
        p.out[row * D + d] = __float2bfloat16(0.f);
        if (d == 0 && p.lse_out) p.lse_out[row] = -INFINITY;
      }
      continue;
    }
    if (MULTI && r.a > r.e) {  // a split past this group's keys: an empty partial
      for (int i = tid; i < NRi * D; i += kConsumerThreads) {
        const int rr = i / D, d = i - rr * D;
        const size_t row = out_row(rr);
        p.o_part[(row * S + r.split) * D + d] = 0.f;
        if (d == 0) p.lse_part[row * S + r.split] = -INFINITY;
      }
      continue;
    }

    const float* rel_g = p.rel + ((size_t)r.b * p.H_q + r.hkv * G) * R;
    // MULTI: position and bias row of this thread's 2 * NT score rows
    int row_pos[NT][2];
    const float* row_rel[NT][2];
    if constexpr (MULTI) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          int rr = nt * 8 + 2 * c4 + j;
          rr = rr < NRi ? rr : NRi - 1;
          const int i = rr / G;
          row_pos[nt][j] = r.pos - (r.tn - 1) + i;
          row_rel[nt][j] = p.rel + ((size_t)(r.t0 + i) * p.H_q + r.hkv * G + (rr - i * G)) * R;
        }
    }
    // key `key` seen by the row at position pr (MULTI: causal + window per row)
    auto row_sees = [&](int key, int pr) {
      return key <= pr && (p.window <= 0 || pr - key < p.window);
    };
    // MULTI: every row of the group sees all 16 keys of this warp's slice
    // (inside the tile's range, at or before the group's first position and
    // inside the window of its last): no per-score mask, and every bias index
    // pos - key is already >= 0.  Warp-uniform.
    auto all_see = [&](const Tile& t, int key0) {
      return key0 >= t.klo && key0 + 15 <= t.khi && key0 + 15 <= r.pos - (r.tn - 1) &&
             (p.window <= 0 || r.pos - key0 < p.window);
    };
    // bias of this thread's 4*NT scores of a tile (already in L2; loaded one
    // tile ahead of its use)
    auto load_bias = [&](const Tile& t, float (&bv)[NT][4]) {
      const int key0 = t.jbase + r0;
      if constexpr (MULTI) {
        if (all_see(t, key0)) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int key = key0 + g + 8 * (i >> 1);
              bv[nt][i] = __ldg(row_rel[nt][i & 1] + min(row_pos[nt][i & 1] - key, R - 1));
            }
          return;
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = key0 + g + 8 * (i >> 1);
          if constexpr (MULTI) {
            const int pr = row_pos[nt][i & 1];
            const bool v = key >= t.klo && key <= t.khi && row_sees(key, pr);
            bv[nt][i] = __ldg(row_rel[nt][i & 1] + (v ? min(pr - key, R - 1) : 0));
          } else {
            int h = nt * 8 + 2 * c4 + (i & 1);
            h = h < G ? h : G - 1;
            const bool v = key >= t.klo && key <= t.khi;
            const int dcl = v ? min(r.pos - key, R - 1) : 0;
            bv[nt][i] = __ldg(rel_g + (size_t)h * R + dcl);
          }
        }
    };

    float m_run[NT][2], l_run[NT][2];
    float o_acc[KS][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o_acc[mt][nt][i] = 0.f;
    }

    auto tile_body = [&](const Tile& t, int st, const float (&bv)[NT][4]) {
      const int key0 = t.jbase + r0;  // key of this warp's first row
      if (!(key0 <= t.khi && key0 + 15 >= t.klo)) return;
      const bool part = (key0 < t.klo) || (key0 + 15 > t.khi);
      const uint32_t kb = smem_u32(smem + st * STAGE_BYTES);
      const uint32_t vb = kb + TILE_BYTES;

      // ---- S^T = K Q^T  (16 keys x 8*NT heads)
      float sacc[NT][4];
      float sacc2[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          sacc[nt][i] = 0.f;
          sacc2[nt][i] = 0.f;
        }
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int chunk = 2 * ks + k_chi;
        const uint32_t addr =
            kb + (chunk >> 3) * kHalfBytes + k_row * 128 + (((chunk & 7) ^ sw) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
        uint32_t b[NT][2];
        if constexpr (kQSmem) {
          // rows (lane & 7) + 8 (lane >> 4), columns 16 ks + 8 ((lane >> 3) & 1):
          // registers = rows 0-7 / 8-15 at k = 2 c4 and 2 c4 + 8
          const uint32_t qa = q_smem + ((lane & 7) + 8 * (lane >> 4)) * QP + 32 * ks +
                              16 * ((lane >> 3) & 1);
          ldsm_x4(qa, b[0][0], b[0][1], b[NT - 1][0], b[NT - 1][1]);
        } else {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            b[nt][0] = qf[kQSmem ? 0 : ks][nt][0];
            b[nt][1] = qf[kQSmem ? 0 : ks][nt][1];
          }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (kTwoChains && (ks & 1))
            mma_16816(sacc2[nt], a0, a1, a2, a3, b[nt][0], b[nt][1]);
          else
            mma_16816(sacc[nt], a0, a1, a2, a3, b[nt][0], b[nt][1]);
        }
      }
      if constexpr (kTwoChains) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) sacc[nt][i] += sacc2[nt][i];
      }

      // ---- scale + bias + mask (log2 domain)
      if (MULTI && all_see(t, key0)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) sacc[nt][i] = fmaf(sacc[nt][i], sl2, bv[nt][i] * kLog2e);
      } else {
        bool vk[2] = {true, true};  // validity of keys g, g+8
        if (part) {
          vk[0] = (key0 + g >= t.klo) && (key0 + g <= t.khi);
          vk[1] = (key0 + g + 8 >= t.klo) && (key0 + g + 8 <= t.khi);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int kr = i >> 1;
            const float s = fmaf(sacc[nt][i], sl2, bv[nt][i] * kLog2e);
            bool ok_k = vk[kr];
            if constexpr (MULTI) ok_k = ok_k && row_sees(key0 + g + 8 * kr, row_pos[nt][i & 1]);
            sacc[nt][i] = ok_k ? s : -INFINITY;
          }
        }
      }

      // ---- online softmax per head (over this warp's 16 keys)
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // the running max (the exponent base) is re-reduced over the warp only
        // when a score exceeds it by more than kMaxSlack (log2 units); until
        // then p <= 2^kMaxSlack, and O and l need no rescale
        float mx0 = fmaxf(sacc[nt][0], sacc[nt][2]);
        float mx1 = fmaxf(sacc[nt][1], sacc[nt][3]);
        float mn0 = m_run[nt][0], mn1 = m_run[nt][1];
        if (__any_sync(0xffffffffu, mx0 > mn0 + kMaxSlack || mx1 > mn1 + kMaxSlack)) {
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          mn0 = fmaxf(mn0, mx0);
          mn1 = fmaxf(mn1, mx1);
        }
        const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float al0 = ex2(m_run[nt][0] - base0);
        const float al1 = ex2(m_run[nt][1] - base1);
        const float p0 = ex2(sacc[nt][0] - base0);
        const float p1 = ex2(sacc[nt][1] - base1);
        const float p2 = ex2(sacc[nt][2] - base0);
        const float p3 = ex2(sacc[nt][3] - base1);
        l_run[nt][0] = fmaf(l_run[nt][0], al0, p0 + p2);
        l_run[nt][1] = fmaf(l_run[nt][1], al1, p1 + p3);
        m_run[nt][0] = mn0;
        m_run[nt][1] = mn1;
        if (!kLazyRescale || !__all_sync(0xffffffffu, al0 == 1.f && al1 == 1.f))
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o_acc[mt][nt][0] *= al0;
          o_acc[mt][nt][2] *= al0;
          o_acc[mt][nt][1] *= al1;
          o_acc[mt][nt][3] *= al1;
        }
        pb[nt][0] = movmatrix_t(pack_bf16(p0, p1));  // keys 2c4..+1 of head g
        pb[nt][1] = movmatrix_t(pack_bf16(p2, p3));  // keys 8+2c4..+1
      }

      // ---- O^T += V^T P^T
      auto pv = [&](uint32_t zm01, uint32_t zm89, auto masked) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int chunk = 2 * mt + v_chi;
          const uint32_t addr =
              vb + (chunk >> 3) * kHalfBytes + v_row * 128 + (((chunk & 7) ^ sw) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(addr, a0, a1, a2, a3);
          if constexpr (decltype(masked)::value) {
            a0 &= zm01;
            a1 &= zm01;
            a2 &= zm89;
            a3 &= zm89;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_16816(o_acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
        }
      };
      if (part) {  // zero V rows of invalid keys (they may hold NaN)
        const int kk = key0 + 2 * c4;
        const uint32_t zm01 = ((kk >= t.klo && kk <= t.khi) ? 0x0000ffffu : 0u) |
                              ((kk + 1 >= t.klo && kk + 1 <= t.khi) ? 0xffff0000u : 0u);
        const uint32_t zm89 = ((kk + 8 >= t.klo && kk + 8 <= t.khi) ? 0x0000ffffu : 0u) |
                              ((kk + 9 >= t.klo && kk + 9 <= t.khi) ? 0xffff0000u : 0u);
        pv(zm01, zm89, std::true_type{});
      } else {
        pv(0xffffffffu, 0xffffffffu, std::false_type{});
      }
    };

    // ---- tile loop (same walk as the producer), bias loaded one tile ahead
    auto run_tiles = [&](auto& plan, auto next_fn) -> bool {
      Tile t = next_fn(plan);
      float bv[NT][4];
      load_bias(t, bv);
      while (true) {
        const int st = kt % stages;
        if (!mbar_wait_warp(smem_u32(&bars[st]), (kt / stages) & 1, abort_flag)) return false;
        const bool more = !plan.done();
        Tile tn = t;
        float bn[NT][4];
        if (more) {
          tn = next_fn(plan);
          load_bias(tn, bn);
        }
        tile_body(t, st, bv);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars[stages + st]));
        ++kt;
        if (!more) return true;
        t = tn;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) bv[nt][i] = bn[nt][i];
      }
    };
    if constexpr (BH == 64) {
      PlanBig plan(r.a, r.e, p.P);
      ok = run_tiles(plan, [](PlanBig& pl) {
        int lp, s0;
        return pl.next(lp, s0);
      });
    } else {
      PlanSmall plan(r.a, r.e);
      ok = run_tiles(plan, [](PlanSmall& pl) { return pl.next(); });
    }
    if (kQSmem) release_slot();
    if (!ok) break;

    // ---- finish the item: sum l over the lanes of the 16 keys
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float v = l_run[nt][j];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        l_run[nt][j] = v;
      }
    // Combine the four warps' (m, l, O): through one O buffer per warp, or in
    // two rounds through two (warps 2 and 3 hand theirs to warps 0 and 1,
    // which merge them in registers, same fragment layout), after which every
    // thread combines the buffers.  In the merge, rows past NRi (padding) read
    // row NRi - 1; they are never stored.
    constexpr int OP = D + 4;
    auto put = [&](int slot) {
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int head = nt * 8 + 2 * c4 + (i & 1);
            if (head < NRi) {
              const int dim = 16 * mt + g + 8 * (i >> 1);
              comb_o[(slot * NR + head) * OP + dim] = o_acc[mt][nt][i];
            }
          }
      if (g == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int head = nt * 8 + 2 * c4 + j;
            comb_m[slot * HP + head] = m_run[nt][j];
            comb_l[slot * HP + head] = l_run[nt][j];
          }
      }
    };
    named_bar_sync(1, kConsumerThreads);  // previous item's readers of comb_* are done
    if constexpr (!COMB2) {
      put(warp);
    } else {
      if (warp >= 2) put(warp - 2);
      named_bar_sync(1, kConsumerThreads);
      if (warp < 2) {
        float sa[NT][2], sb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            int head = nt * 8 + 2 * c4 + j;
            head = head < NRi ? head : NRi - 1;
            const float mo = comb_m[warp * HP + head], lo = comb_l[warp * HP + head];
            const float mx = fmaxf(m_run[nt][j], mo);
            const float base = mx == -INFINITY ? 0.f : mx;
            sa[nt][j] = ex2(m_run[nt][j] - base);
            sb[nt][j] = ex2(mo - base);
            l_run[nt][j] = fmaf(sa[nt][j], l_run[nt][j], sb[nt][j] * lo);
            m_run[nt][j] = mx;
          }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              int head = nt * 8 + 2 * c4 + (i & 1);
              head = head < NRi ? head : NRi - 1;
              const int dim = 16 * mt + g + 8 * (i >> 1);
              o_acc[mt][nt][i] = fmaf(sa[nt][i & 1], o_acc[mt][nt][i],
                                      sb[nt][i & 1] * comb_o[(warp * NR + head) * OP + dim]);
            }
      }
      named_bar_sync(1, kConsumerThreads);  // warps 2 and 3's partials are consumed
      if (warp < 2) put(warp);
    }
    named_bar_sync(1, kConsumerThreads);
    // Per row (one thread each): the common max M, each buffer's scale
    // 2^(m_w - M), the sum Ls and the lse, which this thread stores.  The
    // scales replace the maxima in comb_m, 1 / Ls and the output row index go
    // to comb_l (the thread reads its row's l values before it overwrites
    // them).
    // MULTI, M = -inf: no key of this item is visible to the row (a split may
    // lie wholly past a row's position): an empty result, o = 0 and lse = -inf,
    // which the merge weighs at zero.  With one token every key of an item is
    // visible to its rows.
    if (tid < NRi) {
      const int h = tid;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kCombSlots; ++w) M = fmaxf(M, comb_m[w * HP + h]);
      float sc[kCombSlots], Ls = 0.f;
#pragma unroll
      for (int w = 0; w < kCombSlots; ++w) {
        sc[w] = (!MULTI || M > -INFINITY) ? ex2(comb_m[w * HP + h] - M) : 0.f;
        Ls = fmaf(sc[w], comb_l[w * HP + h], Ls);
      }
      float lse;
      if constexpr (MULTI) lse = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -INFINITY;
      else lse = (M + log2f(Ls)) * kLn2;
      const size_t row = out_row(h);
      if (final_out) {
        if (p.lse_out) p.lse_out[row] = lse;
      } else {
        p.lse_part[row * S + r.split] = lse;
      }
#pragma unroll
      for (int w = 0; w < kCombSlots; ++w) comb_m[w * HP + h] = sc[w];
      if constexpr (MULTI) comb_l[h] = Ls > 0.f ? 1.f / Ls : 0.f;
      else comb_l[h] = 1.f / Ls;
      reinterpret_cast<int*>(comb_l)[HP + h] = (int)row;
    }
    named_bar_sync(1, kConsumerThreads);
    // o = (sum_w 2^(m_w - M) O_w) * (1 / Ls), four outputs per thread at a time: all
    // four read their buffers before any is stored (a global store between
    // them would order every later shared-memory read after it)
    constexpr int kOut = 4;
    for (int i0 = 0; i0 < NRi * D; i0 += kOut * kConsumerThreads) {
      float ov[kOut];
      int rowv[kOut];
#pragma unroll
      for (int u = 0; u < kOut; ++u) {
        int i = i0 + u * kConsumerThreads + tid;
        i = i < NRi * D ? i : 0;
        const int h = i / D, d = i - h * D;
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kCombSlots; ++w) o = fmaf(comb_m[w * HP + h], comb_o[(w * NR + h) * OP + d], o);
        ov[u] = o * comb_l[h];
        rowv[u] = reinterpret_cast<const int*>(comb_l)[HP + h];
      }
#pragma unroll
      for (int u = 0; u < kOut; ++u) {
        const int i = i0 + u * kConsumerThreads + tid;
        if (i >= NRi * D) break;
        const int d = i % D;
        const size_t row = (size_t)rowv[u];
        if (final_out) p.out[row * D + d] = __float2bfloat16(ov[u]);
        else p.o_part[(row * S + r.split) * D + d] = ov[u];
      }
    }
  }
  if (!ok && lane == 0) report(p.dev_err, INKLING_DEVERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// Merge: out = sum_s exp(lse_s - LSE) o_s, LSE = log sum_s exp(lse_s).
// One warp per (query token, query head); sequences that used one split were
// written directly by the decode kernel and are skipped.  Empty splits carry
// lse = -inf and weigh nothing.
struct MergeParams {
  const int32_t* seq_lens;
  const float* o_part;
  const float* lse_part;
  __nv_bfloat16* out;
  float* lse_out;
  int B, H_q, pt_stride, P, window, chunk, S, QL, TG, NG;
};

template <int D, bool MULTI>
__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * 4 + warp;  // (packed token, head)
  if (idx >= p.B * p.QL * p.H_q) return;
  const int t = idx / p.H_q;
  const int b = t / p.QL;
  const SeqPlan sp = seq_plan<MULTI>(p.seq_lens[b], p.pt_stride, p.P, p.window, p.chunk, p.S,
                                     p.QL, p.TG, p.NG, (t - b * p.QL) / p.TG);
  const int n = sp.n_s;
  if (n <= 1) return;
  const float* lse = p.lse_part + (size_t)idx * p.S;
  float M = -INFINITY;
  for (int s = lane; s < n; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float z = 0.f;
  for (int s = lane; s < n; s += 32) z += ex2((lse[s] - M) * kLog2e);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
  const float LSE = M > -INFINITY ? M + logf(z) : -INFINITY;
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;
  const float* o = p.o_part + (size_t)idx * p.S * D + lane * PER;
  for (int s = 0; s < n && LSE > -INFINITY; ++s) {
    const float w = ex2((lse[s] - LSE) * kLog2e);
    if constexpr (PER == 4) {
      const float4 v = *reinterpret_cast<const float4*>(o + (size_t)s * D);
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]);
      acc[3] = fmaf(w, v.w, acc[3]);
    } else {
#pragma unroll
      for (int j = 0; j < PER; ++j) acc[j] = fmaf(w, o[(size_t)s * D + j], acc[j]);
    }
  }
  __nv_bfloat16* dst = p.out + (size_t)idx * D + lane * PER;
#pragma unroll
  for (int j = 0; j < PER; ++j) dst[j] = __float2bfloat16(acc[j]);
  if (lane == 0 && p.lse_out) p.lse_out[idx] = LSE;
}

// ---------------------------------------------------------------------------
// Host launcher

template <int D, int NT, int BH, bool MULTI, bool COMB2 = false>
static int launch_decode_t(const DecodeCall& c, const DecodeParams& prm, int smem_bytes, int grid) {
  auto kern = decode_kernel<D, NT, BH, MULTI, COMB2>;
  static std::atomic<int> limit_set[kMaxDevices];
  if (!smem_limit_on_device(reinterpret_cast<const void*>(kern), 227 * 1024, limit_set))
    return INKLING_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, prm) != cudaSuccess) return INKLING_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return INKLING_ERR_CUDA;
  return INKLING_OK;
}

int launch_decode(const DecodeCall& c) {
  DecodeParams prm;
  memset(&prm, 0, sizeof(prm));
  const int BH = (c.P % 64 == 0) ? 64 : 16;
  {
    uint64_t dims[4] = {(uint64_t)c.D, (uint64_t)c.H_kv, (uint64_t)c.P, (uint64_t)c.num_pages};
    uint64_t strides[3] = {(uint64_t)c.D * 2, (uint64_t)c.H_kv * c.D * 2,
                           (uint64_t)c.P * c.H_kv * c.D * 2};
    uint32_t box[4] = {64, 1, (uint32_t)BH, 1};
    if (!encode_tiled(&prm.tmap_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(c.k_cache),
                      dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return INKLING_ERR_CUDA;
    if (!encode_tiled(&prm.tmap_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(c.v_cache),
                      dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return INKLING_ERR_CUDA;
  }
  const int G = c.H_q / c.H_kv;
  // several query tokens per sequence: items take groups of TG tokens, TG * G
  // rows at most 16 (two 8-row MMA tiles); each group reads its K/V once
  const int QL = std::max(1, c.QL);
  const int TG = decode_token_group(QL, G);
  const int NG = (QL + TG - 1) / TG;
  const int NR = TG * G;
  const int NT = (NR <= 8) ? 1 : 2;
  prm.q = static_cast<const __nv_bfloat16*>(c.q);
  prm.page_table = c.page_table;
  prm.seq_lens = c.seq_lens;
  prm.rel = c.rel;
  prm.out = static_cast<__nv_bfloat16*>(c.out);
  prm.lse_out = c.lse_out;
  prm.o_part = c.o_part;
  prm.lse_part = c.lse_part;
  prm.dev_err = c.dev_err;
  prm.counter = c.counter;
  prm.B = c.B;
  prm.pt_stride = c.pt_stride;
  prm.H_q = c.H_q;
  prm.H_kv = c.H_kv;
  prm.G = G;
  prm.P = c.P;
  prm.num_pages = c.num_pages;
  prm.R = c.R;
  prm.window = c.window;
  prm.QL = QL;
  prm.TG = TG;
  prm.NG = NG;
  prm.S = c.S;
  prm.chunk = c.chunk;
  prm.scale_log2 = c.scale * kLog2e;
  prm.bias_prefetch = (c.R % 4 == 0) && ((reinterpret_cast<uintptr_t>(c.rel) & 15) == 0);
  const int n_prefix = c.S > 1 ? c.B + 1 : 0;
  // kCtasPerSm CTAs per SM: keep each CTA under the budget; 2..max stages
  const int budget = INKLING_DECODE_SMEM_BUDGET_KB * 1024;
  int stages = INKLING_DECODE_MAX_STAGES;
  // The item combine takes one O buffer per consumer warp, or half as many in
  // two rounds (warps 2, 3 hand theirs to warps 0, 1): the two-round combine
  // costs per-item latency, so it is used only where it makes room for a
  // third stage -- which happens only for D = 128 with one n-tile (rows 5..8).
  const auto fits3 = [&](int slots) {
    return DecodeSmem(c.D, NR, NT, 3, n_prefix, slots).total <= budget;
  };
  const bool comb2 = c.D == 128 && NT == 1 && !fits3(kConsumerWarps) && fits3(2);
  const int comb_slots = comb2 ? 2 : kConsumerWarps;
  while (stages > 2 && DecodeSmem(c.D, NR, NT, stages, n_prefix, comb_slots).total > budget)
    --stages;
  prm.stages = stages;
  const int smem = 1024 + DecodeSmem(c.D, NR, NT, stages, n_prefix, comb_slots).total;
  if (smem > 227 * 1024) return INKLING_ERR_ARG;  // batch too large for the item prefix table

  // Static schedule (one split per sequence): give every CTA the same number
  // of items (a grid of ceil(items / waves) CTAs), so the last wave is not a
  // partial one.  Dynamic schedule (splits): fill every slot.
  const int total_items = c.B * c.H_kv * NG * c.S;
  const int slots = kCtasPerSm * sm_count();
  int grid = std::min(total_items, slots);
  if (!c.counter && INKLING_DECODE_BALANCED) {
    const int waves = (total_items + slots - 1) / slots;
    grid = (total_items + waves - 1) / waves;
  }
  grid = std::max(1, grid);
  if (c.counter && cudaMemsetAsync(c.counter, 0, sizeof(int32_t), c.stream) != cudaSuccess)
    return INKLING_ERR_CUDA;

  int rc;
  if (QL == 1) {
    if (c.D == 128) {
      if (BH == 64)
        rc = NT == 1 ? (comb2 ? launch_decode_t<128, 1, 64, false, true>(c, prm, smem, grid)
                              : launch_decode_t<128, 1, 64, false>(c, prm, smem, grid))
                     : launch_decode_t<128, 2, 64, false>(c, prm, smem, grid);
      else
        rc = NT == 1 ? (comb2 ? launch_decode_t<128, 1, 16, false, true>(c, prm, smem, grid)
                              : launch_decode_t<128, 1, 16, false>(c, prm, smem, grid))
                     : launch_decode_t<128, 2, 16, false>(c, prm, smem, grid);
    } else {
      if (BH == 64)
        rc = NT == 1 ? launch_decode_t<64, 1, 64, false>(c, prm, smem, grid)
                     : launch_decode_t<64, 2, 64, false>(c, prm, smem, grid);
      else
        rc = NT == 1 ? launch_decode_t<64, 1, 16, false>(c, prm, smem, grid)
                     : launch_decode_t<64, 2, 16, false>(c, prm, smem, grid);
    }
  } else {
    if (c.D == 128) {
      if (BH == 64)
        rc = NT == 1 ? (comb2 ? launch_decode_t<128, 1, 64, true, true>(c, prm, smem, grid)
                              : launch_decode_t<128, 1, 64, true>(c, prm, smem, grid))
                     : launch_decode_t<128, 2, 64, true>(c, prm, smem, grid);
      else
        rc = NT == 1 ? (comb2 ? launch_decode_t<128, 1, 16, true, true>(c, prm, smem, grid)
                              : launch_decode_t<128, 1, 16, true>(c, prm, smem, grid))
                     : launch_decode_t<128, 2, 16, true>(c, prm, smem, grid);
    } else {
      if (BH == 64)
        rc = NT == 1 ? launch_decode_t<64, 1, 64, true>(c, prm, smem, grid)
                     : launch_decode_t<64, 2, 64, true>(c, prm, smem, grid);
      else
        rc = NT == 1 ? launch_decode_t<64, 1, 16, true>(c, prm, smem, grid)
                     : launch_decode_t<64, 2, 16, true>(c, prm, smem, grid);
    }
  }
  if (rc != INKLING_OK || c.S <= 1) return rc;

  MergeParams mp;
  mp.seq_lens = c.seq_lens;
  mp.o_part = c.o_part;
  mp.lse_part = c.lse_part;
  mp.out = static_cast<__nv_bfloat16*>(c.out);
  mp.lse_out = c.lse_out;
  mp.B = c.B;
  mp.H_q = c.H_q;
  mp.pt_stride = c.pt_stride;
  mp.P = c.P;
  mp.window = c.window;
  mp.chunk = c.chunk;
  mp.S = c.S;
  mp.QL = QL;
  mp.TG = TG;
  mp.NG = NG;
  const int blocks = (int)(((int64_t)c.B * QL * c.H_q + 3) / 4);
  if (QL == 1) {
    if (c.D == 128) merge_kernel<128, false><<<blocks, 128, 0, c.stream>>>(mp);
    else merge_kernel<64, false><<<blocks, 128, 0, c.stream>>>(mp);
  } else {
    if (c.D == 128) merge_kernel<128, true><<<blocks, 128, 0, c.stream>>>(mp);
    else merge_kernel<64, true><<<blocks, 128, 0, c.stream>>>(mp);
  }
  if (cudaGetLastError() != cudaSuccess) return INKLING_ERR_CUDA;
  return INKLING_OK;
}

}  // namespace ira
