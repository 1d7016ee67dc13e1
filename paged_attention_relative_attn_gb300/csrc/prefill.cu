// Chunked / paged prefill with a learned relative-position bias on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Operation: inkling_rel_attn_prefill in include/inkling_rel_attn.h (Support
// Inkling-NVFP4 model, TensorRT-LLM PR #17062, "Implementation": paged prefill
// applying the relative bias to the scores; "Architecture": bias per (query
// token, head, relative distance), sliding window 512 / full causal).
//
// One CTA per (128-query tile of one sequence, query head; a sequence's
// tiles launch last tile first, the longest key ranges ahead of the shortest),
// 12 warps:
//  * warp 0 loads the Q tile once (TMA) and then the K tiles of the tile's
//    visible key range into a 3-stage ring, in page-respecting tiles of 64
//    keys exactly like the decode kernel; warp 6 loads the V tiles the same
//    way into a 2-stage ring (128-byte swizzle);
//  * warp 7 loads the bias bands (below) into a 3-buffer ring (L2
//    evict-normal: consecutive tiles' bands share a 16-byte piece, which then
//    comes from DRAM once);
//  * warp 1 owns tensor memory (three S buffers of 64 columns, and two O
//    accumulators of D columns, one per half of the key columns) and one of
//    its threads issues the MMAs: S_k = Q K_k^T (A and B from shared memory,
//    K-major) and O += P_k V_k (A = P from tensor memory, B = V MN-major from
//    shared memory).  S_0, S_1 and S_2 go first; then, as soon as P_k is
//    written, PV_k is issued, and once PV_k has completed, S_{k+3} into the
//    buffer it has just read, so the QK^T of a tile is ready two softmax
//    periods ahead.  Its shared-memory descriptors are computed once;
//  * warps 2-5 and 8-11 are two softmax warpgroups sharing every row: a
//    thread owns one query row (one TMEM lane) and one half of the key
//    columns of each tile.  It reads S with tcgen05.ld, adds the bias, applies
//    the causal / window mask, keeps its half's running max lazily (its O is
//    rescaled in tensor memory only when the max grows by more than 2^8) and
//    writes P (bf16) back over its S columns with tcgen05.st; the epilogue
//    merges the two halves and stores the normalised output (full tiles
//    through shared memory and TMA).  The scores, exponent arguments and row
//    sums use packed fp32 pairs (fma / add .f32x2), the row max three-input
//    max.
// Every mbarrier wait lets the hardware suspend the waiting warp until the
// phase completes instead of polling (a suspend-time hint).
//
// The bias is the dominant HBM stream: every query row reads its own band of
// rel_logits, 64 distances per key tile, each element exactly once.  Rows are
// assigned to TMEM lanes interleaved by four (lane y of lane group j holds
// query row j + 4y; Q is loaded in that row order by four TMA maps, one per
// token residue mod 4), so that within a group of 32 rows the band start
// moves by exactly 4 floats per row: one box of a sheared 3-D view of
// rel_logits loads a whole group, and every row's band has the same alignment
// and is read with conflict-free 16-byte shared loads.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "internal.h"
#include "plan.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace ira {

constexpr int kPrefThreads = 384;
constexpr int kQRows = 128;
constexpr int kKStages = 3;  // K tiles: released when QK^T has read them
constexpr int kVStages = 2;  // V tiles: released when PV has read them
constexpr int kBiasBufs = 3;
constexpr int kSBufs = 3;  // S tiles in tensor memory: S_{k+3} is computed while softmax k+1 and k+2 run
constexpr int kBiasPitch = 68;                       // floats per row band (64 + alignment)
constexpr int kBiasWarpBytes = 32 * kBiasPitch * 4;  // 32 rows of one warp
constexpr int kBiasBufBytes = 4 * kBiasWarpBytes;    // 128 rows
constexpr float kRescaleThreshold = 8.0f;            // log2 units: rescale O when max grows > 2^8

struct PrefillParams {
  CUtensorMap tmap_q[4];    // tokens r + 4y of q: {D, H_q, y}, box {64, 1, 32}
  CUtensorMap tmap_out[4];  // tokens r + 4y of out: {D, H_q, y}, box {64, 1, 32}, 128B swizzle
  CUtensorMap tmap_k;     // [num_pages][P][H_kv][D] bf16, box {64, 1, BH, 1}
  CUtensorMap tmap_v;
  CUtensorMap tmap_bias;  // sheared view of rel_logits: {x col, token, row-in-group}, box {68, 1, 32}
  int bias_tokens;        // tokens whose whole 32-row group box stays inside the tensor
  const float* rel;
  const int32_t* cu_seqlens_q;
  const int32_t* seq_lens;
  const int32_t* page_table;
  __nv_bfloat16* out;
  float* lse_out;
  int32_t* dev_err;
  int B, T, H_q, H_kv, G, P, num_pages, R, window, pt_stride, tiles_per_seq, max_q_len;
  float scale_log2;
  float scale;
};

template <int D>
struct PrefillSmem {
  static constexpr int HALVES = D / 64;
  static constexpr int QHALF = kQRows * 128;
  static constexpr int Q_BYTES = HALVES * QHALF;
  static constexpr int TILE_BYTES = HALVES * kHalfBytes;
  static constexpr int K_OFF = Q_BYTES;
  static constexpr int V_OFF = K_OFF + kKStages * TILE_BYTES;
  static constexpr int BIAS_OFF = V_OFF + kVStages * TILE_BYTES;
  static constexpr int X_OFF = BIAS_OFF + kBiasBufs * kBiasBufBytes;  // row exchange [2][2][128]
  static constexpr int BAR_OFF = X_OFF + 2 * 2 * kQRows * 4;
  // q_full, k_full/empty, v_full/empty, s_full[2], p_full[2], pv_done, b_full/empty, x_bar[4],
  // o_done
  static constexpr int NBARS = 1 + 2 * kKStages + 2 * kVStages + 3 * kSBufs + 2 * kBiasBufs + 4 + 1;
  static constexpr int TOTAL = BAR_OFF + NBARS * 8 + 16;
};

// L2 policy of the bias loads: evict-normal (an evict-first line holding the
// 16 bytes that two consecutive key tiles' bands share is gone before the
// second band is loaded, and is then read from DRAM twice)
__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// mbarrier waits that let the hardware suspend the warp (up to kSuspendNs)
// until the phase completes, instead of polling.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_s(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait_s(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait_s(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > kWaitTimeoutNs) {
      *abort = 1;
      return false;
    }
  }
}
__device__ __forceinline__ bool waitw(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (__all_sync(0xffffffffu, mbar_try_wait_s(bar, parity))) return true;
  const unsigned long long t0 = globaltimer();
  const bool leader = (threadIdx.x & 31) == 0;
  for (;;) {
    if (__all_sync(0xffffffffu, mbar_try_wait_s(bar, parity))) return true;
    int stop = 0;
    if (leader) {
      if (*abort) {
        stop = 1;
      } else if (globaltimer() - t0 > kWaitTimeoutNs) {
        *abort = 1;
        stop = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
  }
}

// Packed fp32 pairs (two lanes of one 64-bit register, .x in the low half):
// fma / add on both halves in one instruction, rounding as two fma.rn / add.rn.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three (NaN operands ignored, as fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Scores of one column half (32 keys) of a 64-key tile for one query row:
// s[cc] = scale * S[cc] + bias, the bias read from the row's band in shared
// memory.  `half_band` points at the part of the band holding this half's 32
// distances (+3); key column cc of the half sits at float OFF + 31 - cc, OFF
// being the warp-uniform alignment of the band.  Only this gather differs
// between the four alignments.
template <int OFF>
__device__ __forceinline__ void half_scores(float (&s)[32], const uint32_t (&sraw)[32],
                                            const float* half_band, float scale) {
  const float4* src = reinterpret_cast<const float4*>(half_band);
  float bb[36];
#pragma unroll
  for (int q = 0; q < 9; ++q) {
    const float4 v = src[q];
    bb[4 * q + 0] = v.x;
    bb[4 * q + 1] = v.y;
    bb[4 * q + 2] = v.z;
    bb[4 * q + 3] = v.w;
  }
  const uint64_t sc2 = f2_pack(scale, scale);
#pragma unroll
  for (int cc = 0; cc < 32; cc += 2)
    f2_unpack(f2_fma(f2_pack(__uint_as_float(sraw[cc]), __uint_as_float(sraw[cc + 1])), sc2,
                     f2_pack(bb[OFF + 31 - cc], bb[OFF + 30 - cc])),
              s[cc], s[cc + 1]);
}

template <int D, int BH>
__global__ void __launch_bounds__(kPrefThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillParams p) {
  using SM = PrefillSmem<D>;
  constexpr int HALVES = SM::HALVES;
  constexpr int TILE_BYTES = SM::TILE_BYTES;
  // S buffers [0, 64 * kSBufs); O_A [kOCol, kOCol + D) accumulates key columns
  // 0..31 of every tile, O_B [kOCol + 128, ...) columns 32..63 (merged in the
  // epilogue)
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kOCol = 64 * kSBufs;
  constexpr uint32_t kOHalfStride = 128;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = blockIdx.x;
  const int b = blockIdx.y / p.tiles_per_seq;
  // a sequence's query tiles run last tile first: later tiles see more keys,
  // so a call ends on its shortest CTAs
  const int qt = p.tiles_per_seq - 1 - (int)(blockIdx.y - b * p.tiles_per_seq);
  if (b >= p.B) return;

  // ---- the sequence's scalars, loaded together; their latency overlaps the
  // barrier and TMEM set-up below, and nothing reads them before it
  const int tb = __ldg(p.cu_seqlens_q + b);
  const int te = __ldg(p.cu_seqlens_q + b + 1);
  const int L_in = __ldg(p.seq_lens + b);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + kKStages;
  uint64_t* v_full = k_empty + kKStages;
  uint64_t* v_empty = v_full + kVStages;
  uint64_t* s_full = v_empty + kVStages;
  uint64_t* p_full = s_full + kSBufs;   // one barrier per S buffer: phases are
  uint64_t* pv_done = p_full + kSBufs;  // kSBufs tiles apart, parity waits stay exact
  uint64_t* b_full = pv_done + kSBufs;
  uint64_t* b_empty = b_full + kBiasBufs;
  uint64_t* x_bar = b_empty + kBiasBufs;  // per lane group: the two softmax warps of a row
  // every MMA of the CTA has completed (one phase, committed after the last PV).
  // The softmax warps cannot use pv_done for this: one half may reach its
  // epilogue while PV_{n-2} is still pending, and phase n-1 has the parity of
  // phase n-3.
  uint64_t* o_done = x_bar + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(o_done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (tid == 0) {
    mbar_init(smem_u32(q_full), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    for (int s = 0; s < kSBufs; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&p_full[s]), 8);  // the eight softmax warps
      mbar_init(smem_u32(&pv_done[s]), 1);
    }
    for (int s = 0; s < 4; ++s) mbar_init(smem_u32(&x_bar[s]), 2);
    mbar_init(smem_u32(o_done), 1);
    for (int s = 0; s < kBiasBufs; ++s) {
      mbar_init(smem_u32(&b_full[s]), 1);   // the bias loader warp
      mbar_init(smem_u32(&b_empty[s]), 8);  // the eight softmax warps
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- the query tile and its key range (identical in every thread); a CTA
  // with nothing to do frees its TMEM and leaves
  const int q_len = te - tb;
  int L = L_in;
  bool run = q_len > 0 && qt * kQRows < q_len;
  if (run) {
    const int cap = p.pt_stride * p.P;
    if (L > cap) {
      if (tid == 0 && h == 0 && qt == 0) report(p.dev_err, INKLING_DEVERR_SEQ_TOO_LONG);
      L = cap;
    }
    if (q_len > L || tb < 0 || tb + q_len > p.T) {
      if (tid == 0 && h == 0 && qt == 0) report(p.dev_err, INKLING_DEVERR_BAD_CHUNK);
      run = false;
    } else if (q_len > p.max_q_len && tid == 0 && h == 0 && qt == 0) {
      report(p.dev_err, INKLING_DEVERR_BAD_CHUNK);  // tiles past the grid are not computed
    }
  }
  if (!run) {
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  const int t0 = tb + qt * kQRows;
  const int nrows = min(kQRows, q_len - qt * kQRows);
  const int pos0 = L - q_len + qt * kQRows;  // position of row 0
  const int khi_all = pos0 + nrows - 1;
  const int klo_all = p.window > 0 ? max(0, pos0 - p.window + 1) : 0;
  const int hkv = h / p.G;
  const int R = p.R;

  // =================================================================== loaders
  if (warp == 0 || warp == 6) {
    // warp 0: the Q tile, then K tiles into a kKStages ring; warp 6: V tiles
    // into a kVStages ring.  Both walk the same page-respecting tile plan.
    const bool is_k = warp == 0;
    if (lane == 0) {
      if (is_k) {
        for (int r = 0; r < 4; ++r) tmap_prefetch(&p.tmap_q[r]);
        tmap_prefetch(&p.tmap_k);
        // Q tile: row group j (rows j + 4y) = tokens t0 + j + 4y
        int ngroups = 0;
        for (int j = 0; j < 4; ++j) ngroups += (j < nrows) ? 1 : 0;
        const uint64_t pol_q = policy_evict_first();
        mbar_arrive_expect_tx(smem_u32(q_full), ngroups * HALVES * 32 * 128);
        for (int j = 0; j < 4; ++j) {
          if (j >= nrows) continue;
          const int tok = t0 + j;
          for (int hh = 0; hh < HALVES; ++hh)
            tma_load_3d(smem_u32(smem + hh * SM::QHALF + 32 * j * 128), &p.tmap_q[tok & 3],
                        smem_u32(q_full), hh * 64, h, tok >> 2, pol_q);
        }
      } else {
        tmap_prefetch(&p.tmap_v);
      }
    }
    const CUtensorMap* tmap = is_k ? &p.tmap_k : &p.tmap_v;
    const int nst = is_k ? kKStages : kVStages;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    uint8_t* ring = smem + (is_k ? SM::K_OFF : SM::V_OFF);
    const uint64_t pol_kv = policy_evict_last();
    const int32_t* pt_row = p.page_table + (size_t)b * p.pt_stride;
    int batch_base = -1000000;
    int my_page = 0;
    auto page_of = [&](int lp) -> int {  // warp-uniform
      if (lp < batch_base || lp >= batch_base + 32) {
        batch_base = lp;
        const int idx = lp + lane;
        my_page = (idx < p.pt_stride) ? __ldg(pt_row + idx) : 0;
      }
      return __shfl_sync(0xffffffffu, my_page, lp - batch_base);
    };
    int kt = 0;
    bool ok = true;
    if constexpr (BH == 64) {
      PlanBig plan(klo_all, khi_all, p.P);
      while (!plan.done()) {
        const int st = kt % nst;
        if (kt >= nst && lane == 0)
          ok = wait1(smem_u32(&empty[st]), ((kt / nst) - 1) & 1, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        int lp, slot0;
        plan.next(lp, slot0);
        const int page = page_of(lp);
        if (lane == 0) {
          if (is_k && (page < 0 || page >= p.num_pages)) report(p.dev_err, INKLING_DEVERR_BAD_PAGE);
          const uint32_t dst = smem_u32(ring + st * TILE_BYTES);
          const uint32_t fb = smem_u32(&full[st]);
          mbar_arrive_expect_tx(fb, TILE_BYTES);
          for (int hh = 0; hh < HALVES; ++hh)
            tma_load_4d(dst + hh * kHalfBytes, tmap, fb, hh * 64, hkv, slot0, page, pol_kv);
        }
        __syncwarp();
        ++kt;
      }
    } else {
      PlanSmall plan(klo_all, khi_all);
      while (!plan.done()) {
        const int st = kt % nst;
        if (kt >= nst && lane == 0)
          ok = wait1(smem_u32(&empty[st]), ((kt / nst) - 1) & 1, abort_flag);
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
          const uint32_t dst = smem_u32(ring + st * TILE_BYTES);
          const uint32_t fb = smem_u32(&full[st]);
          mbar_arrive_expect_tx(fb, nbox * HALVES * 16 * 128);
          for (int c = 0; c < 4; ++c) {
            const int k0 = t.jbase + 16 * c;
            if (!((k0 <= t.khi) && (k0 + 15 >= t.klo))) continue;
            if (is_k && (pages[c] < 0 || pages[c] >= p.num_pages))
              report(p.dev_err, INKLING_DEVERR_BAD_PAGE);
            for (int hh = 0; hh < HALVES; ++hh)
              tma_load_4d(dst + hh * kHalfBytes + c * 16 * 128, tmap, fb, hh * 64, hkv, k0 % p.P,
                          pages[c], pol_kv);
          }
        }
        __syncwarp();
        ++kt;
      }
    }
    if (!ok && lane == 0) {
      report(p.dev_err, INKLING_DEVERR_TIMEOUT);
      for (int j = max(0, kt - nst); j < kt; ++j)
        mbar_wait_drain(smem_u32(&full[j % nst]), (j / nst) & 1);
      if (is_k) mbar_wait_drain(smem_u32(q_full), 0);
    }
  }
  // =================================================================== MMA issuer
  else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16(kQRows, kTileRows, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kQRows, D, true);
      const uint32_t q_base = smem_u32(smem);
      bool ok = wait1(smem_u32(q_full), 0, abort_flag);
      tc_fence_after();
      int k = 0;
      if (ok) {
        // walk the same tiles as the loader (only the count matters here)
        int ntiles = 0;
        if constexpr (BH == 64) {
          PlanBig plan(klo_all, khi_all, p.P);
          int lp, s0;
          while (!plan.done()) {
            plan.next(lp, s0);
            ++ntiles;
          }
        } else {
          PlanSmall plan(klo_all, khi_all);
          while (!plan.done()) {
            plan.next();
            ++ntiles;
          }
        }
        // Shared-memory descriptors, computed once: a descriptor's start
        // address field is bits 0..13 of (address >> 4), so the descriptor of
        // base + off is that of base plus off >> 4 (all offsets stay inside
        // shared memory: no carry out of the field).
        const uint64_t q_desc0 = smem_desc_sw128(q_base, 16, 1024);
        const uint64_t k_desc0 = smem_desc_sw128(smem_u32(smem + SM::K_OFF), 16, 1024);
        const uint64_t v_desc0 = smem_desc_sw128(smem_u32(smem + SM::V_OFF), kHalfBytes, 1024);
        // One MMA of S_kn = Q K_kn^T (k-step kk, into S buffer kn % kSBufs).
        auto s_mma = [&](int kn, int kk) {
          const uint32_t koff = (uint32_t)((kn % kKStages) * TILE_BYTES) >> 4;
          const uint64_t adesc = q_desc0 + (uint32_t)(((kk >> 2) * SM::QHALF + (kk & 3) * 32) >> 4);
          const uint64_t bdesc =
              k_desc0 + koff + (uint32_t)(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
          tc_mma_ss(tmem + 64 * (kn % kSBufs), adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
        };
        // S_kn may start once K_kn is in and its buffer's previous P
        // (P_{kn - kSBufs}) has been read by its PV
        auto s_ready = [&](int kn) -> bool {
          if (!wait1(smem_u32(&k_full[kn % kKStages]), (kn / kKStages) & 1, abort_flag)) return false;
          if (kn >= kSBufs) {
            const int kq = kn - kSBufs;
            if (!wait1(smem_u32(&pv_done[kq % kSBufs]), (kq / kSBufs) & 1, abort_flag)) return false;
          }
          return true;
        };
        // S_0, S_1 and S_2 ahead; then at each step k: PV_k as soon as P_k is
        // written, and S_{k+3} into the buffer PV_k has just read (after PV_k
        // completes), so the QK^T of a tile is ready two softmax periods early.
        for (int kn = 0; kn < kSBufs && kn < ntiles && ok; ++kn) {
          ok = s_ready(kn);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) s_mma(kn, kk);
          tc_commit(smem_u32(&s_full[kn % kSBufs]));
          tc_commit(smem_u32(&k_empty[kn % kKStages]));
        }
        for (k = 0; k < ntiles && ok; ++k) {
          const int kn = k + kSBufs;
          ok = wait1(smem_u32(&v_full[k % kVStages]), (k / kVStages) & 1, abort_flag);
          if (ok) ok = wait1(smem_u32(&p_full[k % kSBufs]), (k / kSBufs) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t v_desc = v_desc0 + ((uint32_t)((k % kVStages) * TILE_BYTES) >> 4);
          // PV_k: keys 0..31 -> O_A (P at S columns 0..15), keys 32..63 -> O_B
          // (P at S columns 32..47)
#pragma unroll
          for (int j = 0; j < kTileRows / 16; ++j) {
            const int kk = (j >> 1) | ((j & 1) << 1);
            const uint64_t bdesc = v_desc + (uint32_t)((kk * 16 * 128) >> 4);
            const uint32_t o = tmem + kOCol + (kk >= 2 ? kOHalfStride : 0);
            const uint32_t a = tmem + 64 * (k % kSBufs) + (kk >= 2 ? 32 + 8 * (kk - 2) : 8 * kk);
            tc_mma_ts(o, a, bdesc, idesc_pv, (k > 0 || (kk & 1)) ? 1u : 0u);
          }
          tc_commit(smem_u32(&pv_done[k % kSBufs]));
          tc_commit(smem_u32(&v_empty[k % kVStages]));
          if (kn < ntiles) {
            ok = s_ready(kn);  // K_{k+3} in, PV_k (the reader of this buffer) done
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) s_mma(kn, kk);
            tc_commit(smem_u32(&s_full[kn % kSBufs]));
            tc_commit(smem_u32(&k_empty[kn % kKStages]));
          }
        }
      }
      tc_commit(smem_u32(o_done));  // arrives once every MMA issued above has completed
      if (!ok) {
        report(p.dev_err, INKLING_DEVERR_TIMEOUT);
        // let the MMAs already issued finish before tensor memory is released
        mbar_wait_drain(smem_u32(o_done), 0);
      }
    }
    __syncwarp();
  }
  // =================================================================== softmax
  else if ((warp >= 2 && warp < 6) || warp >= 8) {
    // Two warpgroups share every row: warps 2-5 take key columns 0..31 of
    // each tile, warps 8-11 columns 32..63.  Each half runs its own online
    // softmax (max, sum) into its own O accumulator in tensor memory, so the
    // two never wait on each other inside the key loop; the epilogue merges
    // the halves (exchange of (m, l) through shared memory, paired by an
    // mbarrier) and each warpgroup writes half of the output columns.
    const int grp = warp >= 8 ? 1 : 0;
    const int lg = warp & 3;         // TMEM lane group of this warp
    const int i = lg + 4 * lane;     // query row of this thread within the tile
    const bool valid = i < nrows;
    const int pi = pos0 + i;         // its absolute position
    const int lo_i = p.window > 0 ? max(0, pi - p.window + 1) : 0;
    const size_t row_off = ((size_t)(valid ? t0 + i : t0) * p.H_q + h) * R;
    const float clampv = valid ? __ldg(p.rel + row_off + R - 1) : 0.f;
    const uint32_t tlane = tmem + ((uint32_t)(32 * lg) << 16);
    const uint32_t o_mine = tlane + kOCol + kOHalfStride * grp;
    const float scale = p.scale;
    const float* my_half0 = reinterpret_cast<const float*>(smem + SM::BIAS_OFF) +
                            lg * 32 * kBiasPitch + lane * kBiasPitch + 32 * (1 - grp);
    float* xbuf = reinterpret_cast<float*>(smem + SM::X_OFF);  // [2 value][2 grp][128 rows]
    const int c0 = 32 * grp;  // first key column of this half

    using PlanT = typename std::conditional<BH == 64, PlanBig, PlanSmall>::type;
    PlanT cur = [&]() {
      if constexpr (BH == 64) return PlanBig(klo_all, khi_all, p.P);
      else return PlanSmall(klo_all, khi_all);
    }();

    float m_use = -INFINITY, l_part = 0.f;  // this half's running max (natural units) and sum
    bool ok = true;
    int k = 0;
    for (; !cur.done(); ++k) {
      Tile t;
      if constexpr (BH == 64) {
        int lp, s0;
        t = cur.next(lp, s0);
      } else {
        t = cur.next();
      }
      const int buf = k % kBiasBufs;
      if (!waitw(smem_u32(&b_full[buf]), (k / kBiasBufs) & 1, abort_flag)) {
        ok = false;
        break;
      }
      if (!waitw(smem_u32(&s_full[k % kSBufs]), (k / kSBufs) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sraw[32];
      tmem_ld32(tlane + 64 * (k % kSBufs) + c0, sraw);
      tmem_ld_wait();
      // visible key columns of this row in this tile, and in my half
      int cl = max(lo_i, t.klo) - t.jbase;
      int ch = min(pi, t.khi) - t.jbase;
      if (!valid) {
        cl = 64;
        ch = -1;
      }
      const int hl = max(cl, c0), hh = min(ch, c0 + 31);
      const int dtop = pi - t.jbase;
      const bool full_vis = __all_sync(0xffffffffu, hl == c0 && hh == c0 + 31);
      float s[32];
      if (pos0 - t.jbase - 63 >= R) {
        // every distance of the tile is past the table (row 0 is the nearest):
        // all of them take its last column, and no band was loaded
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) s[cc] = fmaf(__uint_as_float(sraw[cc]), scale, clampv);
      } else {
        const int off = (pos0 + lg - t.jbase - 63) & 3;
        const float* half_band = my_half0 + buf * (kBiasBufBytes / 4);
        switch (off) {
          case 0: half_scores<0>(s, sraw, half_band, scale); break;
          case 1: half_scores<1>(s, sraw, half_band, scale); break;
          case 2: half_scores<2>(s, sraw, half_band, scale); break;
          default: half_scores<3>(s, sraw, half_band, scale); break;
        }
        if (__any_sync(0xffffffffu, valid && hl <= hh && dtop - hl >= R)) {
          // distances past the table take its last column (the band holds
          // other values there)
#pragma unroll
          for (int cc = 0; cc < 32; ++cc)
            if (dtop - (c0 + cc) >= R) s[cc] = fmaf(__uint_as_float(sraw[cc]), scale, clampv);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&b_empty[buf]));  // band read: the loader may refill it
      if (!full_vis) {
        // my half's visible columns as a bit mask: column cc is visible iff
        // hl <= c0 + cc <= hh
        const int lo = hl - c0, hi = hh - c0;
        const uint32_t vis = lo > hi ? 0u : ((0xffffffffu >> (31 - hi)) & (0xffffffffu << lo));
#pragma unroll
        for (int cc = 0; cc < 32; ++cc) s[cc] = (vis & (1u << cc)) ? s[cc] : -INFINITY;
      }

      float mx;
      {
        float r11[11];  // 32 -> 11 -> 4 -> 1 with three-input max
#pragma unroll
        for (int j = 0; j < 10; ++j) r11[j] = fmax3(s[3 * j], s[3 * j + 1], s[3 * j + 2]);
        r11[10] = fmaxf(s[30], s[31]);
        const float r0 = fmax3(r11[0], r11[1], r11[2]), r1 = fmax3(r11[3], r11[4], r11[5]);
        const float r2 = fmax3(r11[6], r11[7], r11[8]), r3 = fmaxf(r11[9], r11[10]);
        mx = fmax3(r0, r1, fmaxf(r2, r3));
      }
      float m_new = m_use, alpha = 1.f;
      bool resc = false;
      if (mx > -INFINITY) {
        if (m_use == -INFINITY) {
          m_new = mx;  // first visible keys of this row in my half: my O row is still zero
        } else if (mx > m_use + kRescaleThreshold * kLn2) {
          m_new = mx;
          alpha = ex2((m_use - mx) * kLog2e);
          resc = true;
        }
      }
      if (__any_sync(0xffffffffu, resc)) {
        // my O holds PV_0..PV_{k-1}; wait for the last one, then rescale it
        if (!waitw(smem_u32(&pv_done[(k - 1) % kSBufs]), ((k - 1) / kSBufs) & 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(o_mine + 32 * cc, o);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
          tmem_st32(o_mine + 32 * cc, o);
        }
        tmem_st_wait();
      }
      m_use = m_new;
      l_part *= alpha;
      const float nmu = (m_use == -INFINITY) ? 0.f : -m_use * kLog2e;
      uint32_t pk[16];
      {
        const uint64_t l2e2 = f2_pack(kLog2e, kLog2e), nmu2 = f2_pack(nmu, nmu);
        uint64_t acc[4] = {0, 0, 0, 0};  // four packed partial sums (+0.0 bits)
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          float a0, a1;
          f2_unpack(f2_fma(f2_pack(s[2 * m], s[2 * m + 1]), l2e2, nmu2), a0, a1);
          const float p0 = ex2(a0), p1 = ex2(a1);
          acc[m & 3] = f2_add(acc[m & 3], f2_pack(p0, p1));
          pk[m] = pack_bf16(p0, p1);
        }
        float u0, u1;
        f2_unpack(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), u0, u1);
        l_part += u0 + u1;
      }
      // my half of P (16 bf16 pairs) over the first 16 of my own S columns
      // (which I have already read): half A at columns 0..15, half B at 32..47
      tmem_st16(tlane + 64 * (k % kSBufs) + c0, pk);
      tmem_st_wait();

      if (t.dirty) {
        // rows outside [klo, khi] may hold other keys' values (NaN included):
        // zero them in V so that P = 0 times V stays 0 in the tensor core
        const int st = k % kVStages;
        if (!waitw(smem_u32(&v_full[st]), (k / kVStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const int vlo = t.klo - t.jbase, vhi = t.khi - t.jbase;
        uint8_t* vtile = smem + SM::V_OFF + st * TILE_BYTES;
        const int sid = grp * 128 + lg * 32 + lane;  // 0..255
        for (int u = sid; u < 64 * HALVES * 8; u += 256) {
          const int row = u / (HALVES * 8);
          const int rest = u - row * HALVES * 8;
          if (row >= vlo && row <= vhi) continue;
          *reinterpret_cast<uint4*>(vtile + (rest >> 3) * kHalfBytes + row * 128 + (rest & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&p_full[k % kSBufs]));
    }

    // ---- epilogue: merge the two halves, O / l -> bf16 (half the columns each)
    if (ok && k > 0) ok = waitw(smem_u32(o_done), 0, abort_flag);
    float M = m_use, L = l_part, sc_a = 1.f, sc_b = 0.f;
    if (ok) {
      xbuf[(0 * 2 + grp) * 128 + i] = m_use;
      xbuf[(1 * 2 + grp) * 128 + i] = l_part;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&x_bar[lg]));
      ok = waitw(smem_u32(&x_bar[lg]), 0, abort_flag);
      if (ok) {
        const float ma = xbuf[(0 * 2 + 0) * 128 + i], mb = xbuf[(0 * 2 + 1) * 128 + i];
        const float la = xbuf[(1 * 2 + 0) * 128 + i], lb = xbuf[(1 * 2 + 1) * 128 + i];
        M = fmaxf(ma, mb);
        sc_a = M == -INFINITY ? 0.f : ex2((ma - M) * kLog2e);
        sc_b = M == -INFINITY ? 0.f : ex2((mb - M) * kLog2e);
        L = sc_a * la + sc_b * lb;
      }
    }
    if (ok) {
      tc_fence_after();
      const float inv = L > 0.f ? 1.f / L : 0.f;
      sc_a *= inv;
      sc_b *= inv;
      // A full tile (D = 128) leaves through shared memory -- the Q buffer,
      // free now that every MMA has completed -- and one TMA store per warp
      // (its 32 rows x D/2 columns); rows of a partial tile past the sequence
      // belong to the next one, so those tiles are stored row by row.
      const bool via_smem = D == 128 && nrows == kQRows;
      uint8_t* stage = smem + (grp * 4 + lg) * 4096;  // 32 rows x 128 B, 128B-swizzled
      __nv_bfloat16* orow = p.out + ((size_t)(t0 + i) * p.H_q + h) * D + (D / 2) * grp;
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t oa[32], ob[32];
        tmem_ld32(tlane + kOCol + (D / 2) * grp + 32 * cc, oa);
        tmem_ld32(tlane + kOCol + kOHalfStride + (D / 2) * grp + 32 * cc, ob);
        tmem_ld_wait();
        uint32_t pkd[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          pkd[x] = pack_bf16(
              fmaf(__uint_as_float(oa[2 * x]), sc_a, __uint_as_float(ob[2 * x]) * sc_b),
              fmaf(__uint_as_float(oa[2 * x + 1]), sc_a, __uint_as_float(ob[2 * x + 1]) * sc_b));
        if (via_smem) {
#pragma unroll
          for (int x = 0; x < 4; ++x) {  // 16-byte chunk 4cc + x of my 128-byte row
            const int c = 4 * cc + x;
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_uint4(pkd[4 * x], pkd[4 * x + 1], pkd[4 * x + 2], pkd[4 * x + 3]);
          }
        } else if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cc);
#pragma unroll
          for (int x = 0; x < 4; ++x)
            dst[x] = make_uint4(pkd[4 * x], pkd[4 * x + 1], pkd[4 * x + 2], pkd[4 * x + 3]);
        }
      }
      if (via_smem) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int tok = t0 + lg;  // rows lg + 4y = tokens tok + 4y
          tma_store_3d(&p.tmap_out[tok & 3], smem_u32(stage), (D / 2) * grp, h, tok >> 2);
          bulk_commit_group();
          bulk_wait_group0();  // complete before the CTA (and its shared memory) ends
        }
        __syncwarp();
      }
      if (valid && grp == 0 && p.lse_out)
        p.lse_out[(size_t)(t0 + i) * p.H_q + h] = L > 0.f ? M + log2f(L) * kLn2 : -INFINITY;
    } else if (lane == 0) {
      report(p.dev_err, INKLING_DEVERR_TIMEOUT);
    }
    tc_fence_before();
  }
  // =================================================================== bias loaders
  else if (warp == 7) {
    // warp 7: the row bands of rel_logits for each key tile.  Row y of lane
    // group j is query token t0 + j + 4y; its band is the 68 floats of its
    // bias row starting at floor4(dtop - 63), dtop = its position - jbase.
    // Within a group the band start moves by exactly 4 floats per row, so one
    // TMA box of a sheared view (token stride plus 4 floats per row) loads the
    // whole group.
    const uint64_t pol_b = policy_evict_normal();
    using PlanT = typename std::conditional<BH == 64, PlanBig, PlanSmall>::type;
    PlanT pl = [&]() {
      if constexpr (BH == 64) return PlanBig(klo_all, khi_all, p.P);
      else return PlanSmall(klo_all, khi_all);
    }();
    const uint32_t band_smem = smem_u32(smem + SM::BIAS_OFF);
    int k = 0;
    bool ok = true;
    while (!pl.done()) {
      Tile t;
      if constexpr (BH == 64) {
        int lp, s0;
        t = pl.next(lp, s0);
      } else {
        t = pl.next();
      }
      const int buf = k % kBiasBufs;
      if (k >= kBiasBufs &&
          !waitw(smem_u32(&b_empty[buf]), ((k / kBiasBufs) - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      const uint32_t fb = smem_u32(&b_full[buf]);
      const uint32_t buf_smem = band_smem + buf * kBiasBufBytes;
      // a tile whose every distance is past the table needs no band
      const bool beyond = pos0 - t.jbase - 63 >= R;
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // row group j: rows j + 4y = tokens t0 + j + 4y
        if (j >= nrows || beyond) continue;
        const int tf = t0 + j;
        const int lo4_0 = (pos0 + j - t.jbase - 63) & ~3;
        // the map's bounds are checked on the sheared x: a negative x would
        // zero-fill entries whose true column x + 4y is valid, so such boxes
        // take the per-row path too
        if (tf < p.bias_tokens && h * R + lo4_0 >= 0) {
          // one box of the sheared view: row y of the group starts 4y floats
          // later than row 0, exactly the shift of its band
          if (lane == 0) {
            const int lo4 = lo4_0;
            mbar_expect_tx(fb, 32 * kBiasPitch * 4);
            tma_load_3d(buf_smem + j * kBiasWarpBytes, &p.tmap_bias, fb, h * R + lo4, tf, 0,
                        pol_b);
          }
        } else {
          // the box could reach past the end of the tensor: per-row copies
          const int ii = j + 4 * lane;
          if (ii >= nrows) continue;
          const int pp = pos0 + ii;
          const int lo_r = p.window > 0 ? max(0, pp - p.window + 1) : 0;
          const int vlo = max(lo_r, t.klo), vhi = min(pp, t.khi);
          if (vlo > vhi) continue;
          const int dtop = pp - t.jbase;
          const int lo4 = (dtop - 63) & ~3;
          const int dmin = pp - vhi, dmax = min(pp - vlo, R - 1);
          if (dmin > dmax) continue;
          const int c_lo = (dmin - lo4) >> 2, c_hi = (dmax - lo4) >> 2;
          const uint32_t bytes = (uint32_t)(c_hi - c_lo + 1) * 16;
          const uint32_t dst = buf_smem + j * kBiasWarpBytes + lane * kBiasPitch * 4 + c_lo * 16;
          const float* src = p.rel + ((size_t)(t0 + ii) * p.H_q + h) * R + lo4 + 4 * c_lo;
          mbar_expect_tx(fb, bytes);
          bulk_load(dst, src, bytes, fb);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(fb);
      ++k;
    }
    if (!ok && lane == 0) {
      report(p.dev_err, INKLING_DEVERR_TIMEOUT);
      for (int j = max(0, k - kBiasBufs); j < k; ++j)
        mbar_wait_drain(smem_u32(&b_full[j % kBiasBufs]), (j / kBiasBufs) & 1);
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host launcher

template <int D, int BH>
static int launch_prefill_t(const PrefillCall& c, const PrefillParams& prm, dim3 grid) {
  auto kern = prefill_kernel<D, BH>;
  const int smem = 1024 + PrefillSmem<D>::TOTAL;
  static std::atomic<int> limit_set[kMaxDevices];
  if (!smem_limit_on_device(reinterpret_cast<const void*>(kern), smem, limit_set))
    return INKLING_ERR_CUDA;
  kern<<<grid, kPrefThreads, smem, c.stream>>>(prm);
  if (cudaGetLastError() != cudaSuccess) return INKLING_ERR_CUDA;
  return INKLING_OK;
}

int launch_prefill(const PrefillCall& c) {
  PrefillParams prm;
  memset(&prm, 0, sizeof(prm));
  const int BH = (c.P % 64 == 0) ? 64 : 16;
  const uint64_t tok_bytes = (uint64_t)c.H_q * c.D * 2;
  for (int r = 0; r < 4; ++r) {
    const uint64_t rows = c.T > r ? (uint64_t)(c.T - r + 3) / 4 : 1;
    uint64_t dims[3] = {(uint64_t)c.D, (uint64_t)c.H_q, rows};
    uint64_t strides[2] = {(uint64_t)c.D * 2, 4 * tok_bytes};
    uint32_t box[3] = {64, 1, 32};
    const char* base = static_cast<const char*>(c.q) + (c.T > r ? r : 0) * tok_bytes;
    if (!encode_tiled(&prm.tmap_q[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<char*>(base),
                      dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
      return INKLING_ERR_CUDA;
  }
  for (int r = 0; r < 4; ++r) {  // out, same row split as q (D = 128 only)
    if (c.D != 128) break;
    const uint64_t rows = c.T > r ? (uint64_t)(c.T - r + 3) / 4 : 1;
    uint64_t dims[3] = {(uint64_t)c.D, (uint64_t)c.H_q, rows};
    uint64_t strides[2] = {(uint64_t)c.D * 2, 4 * tok_bytes};
    uint32_t box[3] = {64, 1, 32};
    char* base = static_cast<char*>(c.out) + (c.T > r ? r : 0) * tok_bytes;
    if (!encode_tiled(&prm.tmap_out[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides,
                      box, CU_TENSOR_MAP_SWIZZLE_128B))
      return INKLING_ERR_CUDA;
  }
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
  {
    // sheared view of rel_logits [T][H_q][R] fp32: element (x, z, y) at
    // rel + z*H_q*R + y*(4*H_q*R + 4) + x  -- token z + 4y, column x + 4y.
    // Tokens z past bias_tokens are out of the map (their boxes use per-row
    // copies), so no box ever touches memory past the end of the tensor.
    const uint64_t row = (uint64_t)c.H_q * c.R;
    // (needs rows of at least 64 floats so that the 124-float shear of the
    // last box row stays inside the following token row)
    const int64_t ok_tokens = row >= 64 ? (int64_t)c.T - 126 : 0;
    prm.bias_tokens = (int)std::max<int64_t>(0, ok_tokens);
    uint64_t dims[3] = {row, (uint64_t)std::max<int64_t>(1, ok_tokens), 32};
    uint64_t strides[2] = {row * 4, (4 * row + 4) * 4};
    uint32_t box[3] = {(uint32_t)kBiasPitch, 1, 32};
    if (!encode_tiled(&prm.tmap_bias, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                      const_cast<float*>(c.rel), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
      return INKLING_ERR_CUDA;
  }
  prm.rel = c.rel;
  prm.cu_seqlens_q = c.cu_seqlens_q;
  prm.seq_lens = c.seq_lens;
  prm.page_table = c.page_table;
  prm.out = static_cast<__nv_bfloat16*>(c.out);
  prm.lse_out = c.lse_out;
  prm.dev_err = c.dev_err;
  prm.B = c.B;
  prm.T = c.T;
  prm.H_q = c.H_q;
  prm.H_kv = c.H_kv;
  prm.G = c.H_q / c.H_kv;
  prm.P = c.P;
  prm.num_pages = c.num_pages;
  prm.R = c.R;
  prm.window = c.window;
  prm.pt_stride = c.pt_stride;
  prm.max_q_len = c.max_q_len;
  prm.tiles_per_seq = std::max(1, (c.max_q_len + kQRows - 1) / kQRows);
  prm.scale_log2 = c.scale * kLog2e;
  prm.scale = c.scale;
  if (c.max_q_len <= 0) return INKLING_OK;
  dim3 grid(c.H_q, c.B * prm.tiles_per_seq);
  if (c.D == 128)
    return BH == 64 ? launch_prefill_t<128, 64>(c, prm, grid) : launch_prefill_t<128, 16>(c, prm, grid);
  return BH == 64 ? launch_prefill_t<64, 64>(c, prm, grid) : launch_prefill_t<64, 16>(c, prm, grid);
}

}  // namespace ira
