// Split-KV paged decode with a learned relative-position bias, and the
// log-sum-exp merge of the splits.
//
// Operation: inkling_rel_attn_decode in include/inkling_rel_attn.h (Support
// Inkling-NVFP4 model, TensorRT-LLM PR #17062, "Architecture" and
// "Implementation"; split-KV from Fail fast on Inkling's unsupported GPU
// architectures, vLLM PR #51560, "Changes").
//
// Design (one CTA per (split, KV head, sequence)):
//  * warp 4 (producer) walks the CTA's logical key range in tiles of <= 64
//    keys, looks the physical page up in the page table and issues TMA loads
//    of the K and V rows of this KV head (box = 64 dims x 1 head x rows x 1
//    page, 128-byte swizzle) into a ring of shared-memory stages guarded by
//    full/empty mbarriers.  The first tile of a range starts mid-page so the
//    box runs past the page end (zero-filled, never read from HBM); the last
//    tile is placed so the box starts before the page (also zero-filled).
//    Only the bytes of visible keys are fetched.
//  * warps 0-3 (consumers) each own 16 rows of every tile and compute the
//    transposed products S^T = K Q^T and O^T += V^T P^T with mma.sync
//    m16n8k16 (the GQA group of <= 8 query heads is the N=8 side, so no
//    padding of M), add the bias from a shared-memory copy of the needed
//    slice of rel_logits (pre-multiplied by log2 e), mask, and run an online
//    softmax per head with warp shuffles over the keys.  P is moved from the
//    accumulator layout into the B-operand layout with movmatrix.
//  * at the end the four warps' (m, l, O) are combined through shared memory
//    and written either as the final bf16 output or, when the sequence spans
//    several splits, as a normalised fp32 partial plus its lse for the merge.
// Reduction order depends only on logical key positions and host scalars, so
// results are bit-identical under any physical page permutation.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace ira {

constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = 32 * (kConsumerWarps + 1);
constexpr int kTileRows = 64;
constexpr int kHalfBytes = kTileRows * 128;  // 64 rows x 64 bf16

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
  int pt_stride, H_q, H_kv, G, P, num_pages, R, window;
  int S, chunk, stages, nb;
  float scale_log2;
};

// Visible key range [lo, pos] of the decode query of a sequence and its split
// count; identical in the decode and merge kernels.
struct SeqPlan {
  int L, pos, lo, nvis, n_s;
};
__device__ __forceinline__ SeqPlan seq_plan(int L, int pt_stride, int P, int window, int chunk,
                                            int S) {
  SeqPlan s;
  const int cap = pt_stride * P;
  if (L > cap) L = cap;
  if (L < 0) L = 0;
  s.L = L;
  s.pos = L - 1;
  s.lo = (window > 0) ? max(0, s.pos - window + 1) : 0;
  s.nvis = L > 0 ? s.pos - s.lo + 1 : 0;
  int n = (s.nvis + chunk - 1) / chunk;
  s.n_s = n > S ? S : n;
  return s;
}

// One tile of the logical key range: rows r of the stage hold key jbase + r;
// keys [klo, khi] are the valid ones.
struct Tile {
  int jbase, klo, khi;
};

// Tile walk for page sizes that are a multiple of 64 (box of 64 rows): tiles
// never cross a page; see the file comment for the placement of the first
// and last tile.
struct PlanBig {
  int e, P, jt;
  __device__ PlanBig(int a, int e_, int P_) : e(e_), P(P_), jt(a) {}
  __device__ bool done() const { return jt > e; }
  // returns the tile and, for the loader, the logical page and first slot
  __device__ Tile next(int& lpage, int& slot0) {
    const int lp = jt / P;
    const int pstart = lp * P;
    const int pe = pstart + P - 1;
    int et = min(jt + 63, pe);
    et = min(et, e);
    const bool rev = (et == e) && (jt == pstart) && (et - jt < 63);
    Tile t;
    t.jbase = rev ? et - 63 : jt;
    t.klo = jt;
    t.khi = et;
    lpage = lp;
    slot0 = t.jbase - pstart;
    jt = et + 1;
    return t;
  }
};

// Tile walk for other page sizes (multiple of 16): 64-aligned logical
// blocks, each assembled from four 16-row boxes; boxes that hold no valid key
// are not loaded.
struct PlanSmall {
  int a, e, jt;
  __device__ PlanSmall(int a_, int e_) : a(a_), e(e_), jt(a_ & ~63) {}
  __device__ bool done() const { return jt > e; }
  __device__ Tile next() {
    Tile t;
    t.jbase = jt;
    t.klo = max(a, jt);
    t.khi = min(e, jt + 63);
    jt += 64;
    return t;
  }
};

template <int BH>
struct PlanSel;
template <>
struct PlanSel<64> {
  using type = PlanBig;
};
template <>
struct PlanSel<16> {
  using type = PlanSmall;
};

__device__ __forceinline__ void report(int32_t* err, int bit) {
  if (err) atomicOr(err, bit);
}

template <int D, int NT, int BH>
__global__ void __launch_bounds__(kDecodeThreads)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int HALVES = D / 64;
  constexpr int TILE_BYTES = HALVES * kHalfBytes;
  constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  constexpr int KS = D / 16;  // k-steps of QK^T, m-tiles of PV
  constexpr int HP = 8 * NT;  // padded heads per group

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int split = blockIdx.x;
  const int hkv = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int G = p.G;
  const int S = p.S;

  const int Lraw = p.seq_lens[b];
  const SeqPlan sp = seq_plan(Lraw, p.pt_stride, p.P, p.window, p.chunk, S);
  if (Lraw > p.pt_stride * p.P && tid == 0 && split == 0 && hkv == 0)
    report(p.dev_err, INKLING_DEVERR_SEQ_TOO_LONG);
  if (split >= max(sp.n_s, 1)) return;
  const bool final_out = sp.n_s <= 1;

  if (sp.nvis == 0) {  // empty sequence: out = 0, lse = -inf
    for (int i = tid; i < G * D; i += kDecodeThreads) {
      const int h = i / D, d = i - h * D;
      const size_t row = (size_t)b * p.H_q + hkv * G + h;
      p.out[row * D + d] = __float2bfloat16(0.f);
      if (d == 0 && p.lse_out) p.lse_out[row] = -INFINITY;
    }
    return;
  }

  const int a = sp.lo + split * p.chunk;
  const int e = (split == sp.n_s - 1) ? sp.pos : a + p.chunk - 1;

  // ---- shared memory carve-up
  const int stages = p.stages;
  float* bias_s = reinterpret_cast<float*>(smem + stages * STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + stages * STAGE_BYTES + ((G * p.nb * 4 + 15) & ~15));
  // full[s] = bars[s], empty[s] = bars[stages + s]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * stages);

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&bars[s]), 1);
      mbar_init(smem_u32(&bars[stages + s]), kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  using Plan = typename PlanSel<BH>::type;

  // =================================================================== producer
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      tmap_prefetch(&p.tmap_k);
      tmap_prefetch(&p.tmap_v);
    }
    const uint64_t pol = policy_evict_first();
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
    Plan plan = [&]() {
      if constexpr (BH == 64) return PlanBig(a, e, p.P);
      else return PlanSmall(a, e);
    }();
    int k = 0;
    bool ok = true;
    while (!plan.done()) {
      const int st = k % stages;
      if (k >= stages && lane == 0) ok = mbar_wait(smem_u32(&bars[stages + st]), ((k / stages) - 1) & 1, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const uint32_t kdst = smem_u32(smem + st * STAGE_BYTES);
      const uint32_t vdst = kdst + TILE_BYTES;
      const uint32_t fb = smem_u32(&bars[st]);
      if constexpr (BH == 64) {
        int lp, slot0;
        plan.next(lp, slot0);
        int page = page_of(lp);
        if (page < 0 || page >= p.num_pages) {
          if (lane == 0) report(p.dev_err, INKLING_DEVERR_BAD_PAGE);
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, 2 * TILE_BYTES);
#pragma unroll
          for (int h = 0; h < HALVES; ++h) {
            tma_load_4d(kdst + h * kHalfBytes, &p.tmap_k, fb, h * 64, hkv, slot0, page, pol);
            tma_load_4d(vdst + h * kHalfBytes, &p.tmap_v, fb, h * 64, hkv, slot0, page, pol);
          }
        }
      } else {
        const Tile t = plan.next();
        int nbox = 0;
        int pages[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int k0 = t.jbase + 16 * c;
          const bool need = (k0 <= t.khi) && (k0 + 15 >= t.klo);
          pages[c] = need ? page_of(k0 / p.P) : 0;
          if (need) {
            ++nbox;
            if ((pages[c] < 0 || pages[c] >= p.num_pages) && lane == 0)
              report(p.dev_err, INKLING_DEVERR_BAD_PAGE);
          }
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, nbox * 2 * HALVES * 16 * 128);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int k0 = t.jbase + 16 * c;
            if (!((k0 <= t.khi) && (k0 + 15 >= t.klo))) continue;
            const int slot = k0 % p.P;
#pragma unroll
            for (int h = 0; h < HALVES; ++h) {
              tma_load_4d(kdst + h * kHalfBytes + c * 16 * 128, &p.tmap_k, fb, h * 64, hkv, slot,
                          pages[c], pol);
              tma_load_4d(vdst + h * kHalfBytes + c * 16 * 128, &p.tmap_v, fb, h * 64, hkv, slot,
                          pages[c], pol);
            }
          }
        }
      }
      __syncwarp();
      ++k;
    }
    if (!ok && lane == 0) {
      report(p.dev_err, INKLING_DEVERR_TIMEOUT);
      // drain: wait for the copies already issued into stages nobody consumes
      for (int j = max(0, k - stages); j < k; ++j)
        mbar_wait_drain(smem_u32(&bars[j % stages]), (j / stages) & 1);
    }
    return;
  }

  // =================================================================== consumers
  const int g = lane >> 2;  // accumulator row group
  const int c4 = lane & 3;  // thread in group

  // Q^T fragments (B operand): head g (+8 per n-tile), dims 16ks + 2c4 (+8)
  uint32_t qf[KS][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = nt * 8 + g;
    const bool live = head < G;
    const __nv_bfloat16* qrow = p.q + ((size_t)b * p.H_q + hkv * G + (live ? head : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qf[ks][nt][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4)) : 0u;
      qf[ks][nt][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c4 + 8)) : 0u;
    }
  }

  // bias slice: distances [dlo, dhi] (clamped to R-1) for the G heads
  const int R = p.R;
  const int dlo = min(sp.pos - e, R - 1);
  const int dhi = min(sp.pos - a, R - 1);
  const int cnt = dhi - dlo + 1;
  const bool bias_in_smem = cnt <= p.nb;
  const float* rel_g = p.rel + ((size_t)b * p.H_q + hkv * G) * R;
  if (bias_in_smem) {
    for (int i = tid; i < G * cnt; i += 32 * kConsumerWarps) {
      const int h = i / cnt, kk = i - h * cnt;
      bias_s[h * p.nb + kk] = __ldg(rel_g + (size_t)h * R + dlo + kk) * kLog2e;
    }
  }
  named_bar_sync(1, 32 * kConsumerWarps);

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

  // per-thread ldmatrix addressing inside a stage
  const int r0 = warp * 16;
  const int k_row = r0 + (lane & 7) + ((lane >> 3) & 1) * 8;  // K: matrices (rows, chunk)
  const int k_chi = lane >> 4;
  const int v_row = r0 + (lane & 7) + ((lane >> 4) & 1) * 8;  // V^T: matrices (chunk, rows)
  const int v_chi = (lane >> 3) & 1;
  const int sw = lane & 7;  // (row & 7) for the 128-byte swizzle
  const float sl2 = p.scale_log2;

  Plan plan = [&]() {
    if constexpr (BH == 64) return PlanBig(a, e, p.P);
    else return PlanSmall(a, e);
  }();
  int k = 0;
  bool ok = true;
  while (!plan.done()) {
    Tile t;
    if constexpr (BH == 64) {
      int lp, s0;
      t = plan.next(lp, s0);
    } else {
      t = plan.next();
    }
    const int st = k % stages;
    bool got = true;
    if (lane == 0) got = mbar_wait(smem_u32(&bars[st]), (k / stages) & 1, abort_flag);
    got = __shfl_sync(0xffffffffu, got, 0);
    if (!got) {
      ok = false;
      break;
    }
    const int key0 = t.jbase + r0;  // key of this warp's first row
    if (key0 <= t.khi && key0 + 15 >= t.klo) {
      const bool part = (key0 < t.klo) || (key0 + 15 > t.khi);
      const uint32_t kb = smem_u32(smem + st * STAGE_BYTES);
      const uint32_t vb = kb + TILE_BYTES;

      // ---- S^T = K Q^T  (16 keys x 8*NT heads)
      float sacc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int chunk = 2 * ks + k_chi;
        const uint32_t addr = kb + (chunk >> 3) * kHalfBytes + k_row * 128 + (((chunk & 7) ^ sw) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(sacc[nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
      }

      // ---- scale + bias + mask (log2 domain)
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
          int h = nt * 8 + 2 * c4 + (i & 1);
          h = h < G ? h : G - 1;
          const int dist = sp.pos - (key0 + g + 8 * kr);
          const int dcl = min(dist, R - 1);
          float bias;
          if (bias_in_smem) {
            const int di = vk[kr] ? dcl - dlo : 0;
            bias = bias_s[h * p.nb + di];
          } else {
            bias = vk[kr] ? __ldg(rel_g + (size_t)h * R + dcl) * kLog2e : 0.f;
          }
          const float s = fmaf(sacc[nt][i], sl2, bias);
          sacc[nt][i] = vk[kr] ? s : -INFINITY;
        }
      }

      // ---- online softmax per head (over this warp's 16 keys)
      uint32_t pb[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float mx0 = fmaxf(sacc[nt][0], sacc[nt][2]);
        float mx1 = fmaxf(sacc[nt][1], sacc[nt][3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m_run[nt][0], mx0);
        const float mn1 = fmaxf(m_run[nt][1], mx1);
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
      uint32_t zm01 = 0xffffffffu, zm89 = 0xffffffffu;
      if (part) {  // zero V rows of invalid keys (they may hold NaN)
        const int kk = key0 + 2 * c4;
        zm01 = ((kk >= t.klo && kk <= t.khi) ? 0x0000ffffu : 0u) |
               ((kk + 1 >= t.klo && kk + 1 <= t.khi) ? 0xffff0000u : 0u);
        zm89 = ((kk + 8 >= t.klo && kk + 8 <= t.khi) ? 0x0000ffffu : 0u) |
               ((kk + 9 >= t.klo && kk + 9 <= t.khi) ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int chunk = 2 * mt + v_chi;
        const uint32_t addr = vb + (chunk >> 3) * kHalfBytes + v_row * 128 + (((chunk & 7) ^ sw) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(addr, a0, a1, a2, a3);
        a0 &= zm01;
        a1 &= zm01;
        a2 &= zm89;
        a3 &= zm89;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(o_acc[mt][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars[stages + st]));
    ++k;
  }

  // ---- finish: sum l over the 16 keys' lanes
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

  named_bar_sync(1, 32 * kConsumerWarps);  // all stages consumed; reuse them
  if (!ok || *abort_flag) {
    if (tid == 0) report(p.dev_err, INKLING_DEVERR_TIMEOUT);
    return;
  }
  constexpr int OP = D + 4;  // padded row of the combine buffer
  float* comb_o = reinterpret_cast<float*>(smem);                  // [4][HP][OP]
  float* comb_m = comb_o + kConsumerWarps * HP * OP;               // [4][HP]
  float* comb_l = comb_m + kConsumerWarps * HP;                    // [4][HP]
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int dim = 16 * mt + g + 8 * (i >> 1);
        const int head = nt * 8 + 2 * c4 + (i & 1);
        comb_o[(warp * HP + head) * OP + dim] = o_acc[mt][nt][i];
      }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int head = nt * 8 + 2 * c4 + j;
        comb_m[warp * HP + head] = m_run[nt][j];
        comb_l[warp * HP + head] = l_run[nt][j];
      }
  }
  named_bar_sync(1, 32 * kConsumerWarps);

  for (int i = tid; i < G * D; i += 32 * kConsumerWarps) {
    const int h = i / D, d = i - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, comb_m[w * HP + h]);
    float Ls = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float sc = ex2(comb_m[w * HP + h] - M);
      Ls = fmaf(sc, comb_l[w * HP + h], Ls);
      o = fmaf(sc, comb_o[(w * HP + h) * OP + d], o);
    }
    o = o / Ls;
    const float lse = (M + log2f(Ls)) * kLn2;
    const size_t row = (size_t)b * p.H_q + hkv * G + h;
    if (final_out) {
      p.out[row * D + d] = __float2bfloat16(o);
      if (d == 0 && p.lse_out) p.lse_out[row] = lse;
    } else {
      p.o_part[(row * S + split) * D + d] = o;
      if (d == 0) p.lse_part[row * S + split] = lse;
    }
  }
}

// ---------------------------------------------------------------------------
// Merge: out = sum_s exp(lse_s - LSE) o_s, LSE = log sum_s exp(lse_s).
// One warp per (sequence, query head); sequences that used one split were
// written directly by the decode kernel and are skipped.
struct MergeParams {
  const int32_t* seq_lens;
  const float* o_part;
  const float* lse_part;
  __nv_bfloat16* out;
  float* lse_out;
  int B, H_q, pt_stride, P, window, chunk, S;
};

template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const MergeParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int idx = blockIdx.x * 4 + warp;
  if (idx >= p.B * p.H_q) return;
  const int b = idx / p.H_q;
  const SeqPlan sp = seq_plan(p.seq_lens[b], p.pt_stride, p.P, p.window, p.chunk, p.S);
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
  const float LSE = M + logf(z);
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;
  const float* o = p.o_part + (size_t)idx * p.S * D + lane * PER;
  for (int s = 0; s < n; ++s) {
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

template <int D, int NT, int BH>
static int launch_decode_t(const DecodeCall& c, const DecodeParams& prm, int smem_bytes) {
  auto kern = decode_kernel<D, NT, BH>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  if (attr_err != cudaSuccess) return INKLING_ERR_CUDA;
  dim3 grid(c.S, c.H_kv, c.B);
  kern<<<grid, kDecodeThreads, smem_bytes, c.stream>>>(prm);
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
  prm.q = static_cast<const __nv_bfloat16*>(c.q);
  prm.page_table = c.page_table;
  prm.seq_lens = c.seq_lens;
  prm.rel = c.rel;
  prm.out = static_cast<__nv_bfloat16*>(c.out);
  prm.lse_out = c.lse_out;
  prm.o_part = c.o_part;
  prm.lse_part = c.lse_part;
  prm.dev_err = c.dev_err;
  prm.pt_stride = c.pt_stride;
  prm.H_q = c.H_q;
  prm.H_kv = c.H_kv;
  prm.G = G;
  prm.P = c.P;
  prm.num_pages = c.num_pages;
  prm.R = c.R;
  prm.window = c.window;
  prm.S = c.S;
  prm.chunk = c.chunk;
  prm.scale_log2 = c.scale * kLog2e;

  // bias entries per head: the widest distance range one CTA can need
  const int keys_cta = (c.S > 1) ? c.chunk : c.keys_max;
  prm.nb = std::max(1, std::min(c.R, keys_cta));
  const int NT = (G <= 8) ? 1 : 2;
  const int stage_bytes = 2 * (c.D / 64) * kHalfBytes;
  const int bias_bytes = ((G * prm.nb * 4 + 15) / 16) * 16;
  // aim at two CTAs per SM; keep 2..4 stages
  const int budget = 110 * 1024 - bias_bytes - 1024 - 256;
  int stages = std::max(2, std::min(4, budget / stage_bytes));
  const int combine_bytes = kConsumerWarps * 8 * NT * (c.D + 4) * 4 + 2 * kConsumerWarps * 8 * NT * 4;
  while (stages * stage_bytes < combine_bytes) ++stages;
  prm.stages = stages;
  int smem = 1024 + stages * stage_bytes + bias_bytes + 2 * stages * 8 + 16;
  if (smem > 227 * 1024) {  // very long bias rows: fall back to reading bias from global
    prm.nb = 1;
    smem = 1024 + stages * stage_bytes + 16 + 2 * stages * 8 + 16;
  }

  int rc;
  if (c.D == 128) {
    if (BH == 64)
      rc = NT == 1 ? launch_decode_t<128, 1, 64>(c, prm, smem) : launch_decode_t<128, 2, 64>(c, prm, smem);
    else
      rc = NT == 1 ? launch_decode_t<128, 1, 16>(c, prm, smem) : launch_decode_t<128, 2, 16>(c, prm, smem);
  } else {
    if (BH == 64)
      rc = NT == 1 ? launch_decode_t<64, 1, 64>(c, prm, smem) : launch_decode_t<64, 2, 64>(c, prm, smem);
    else
      rc = NT == 1 ? launch_decode_t<64, 1, 16>(c, prm, smem) : launch_decode_t<64, 2, 16>(c, prm, smem);
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
  const int blocks = (c.B * c.H_q + 3) / 4;
  if (c.D == 128)
    merge_kernel<128><<<blocks, 128, 0, c.stream>>>(mp);
  else
    merge_kernel<64><<<blocks, 128, 0, c.stream>>>(mp);
  if (cudaGetLastError() != cudaSuccess) return INKLING_ERR_CUDA;
  return INKLING_OK;
}

}  // namespace ira
