// Walk of a sequence's logical key range in tiles of at most 64 keys, each
// loaded by TMA from the paged cache (shared by the decode and prefill kernels).
//
// A tile's shared-memory rows r = 0..63 hold keys jbase + r; keys [klo, khi]
// are the valid ones.  Everything else in the tile is either zero (the TMA box
// ran outside the page and was zero-filled without reading memory) or stale /
// neighbouring data, which consumers mask.
#pragma once

#include <stdint.h>

#include "../../include/inkling_rel_attn.h"

namespace ira {

constexpr int kTileRows = 64;
constexpr int kHalfBytes = kTileRows * 128;  // 64 rows x 64 bf16 (one swizzled half)

// One tile of a key range: row r of the stage holds key jbase + r; keys
// [klo, khi] are the valid ones.  `dirty` is set when rows outside [klo, khi]
// may hold in-bounds data of other keys (possibly NaN) rather than zeros.
struct Tile {
  int jbase, klo, khi;
  bool dirty;
};

// Tile walk for page sizes that are a multiple of 64 (box of 64 rows).  Tiles
// never cross a page.  The first tile of a range starts at its first key,
// mid-page, so the box may run past the page end: those rows are out of the
// tensor's slot range and TMA zero-fills them without touching memory.  The
// last tile, when it starts at a page boundary, is placed so that its box ENDS
// at the last key (a negative first slot): the rows before the page are again
// zero-filled.  So only visible keys' bytes are fetched; only a range that
// starts and ends inside one page loads a few in-bounds rows past its end.
struct PlanBig {
  int e, P, jt, lp2;  // lp2 = log2(P) when P is a power of two, else -1
  __device__ PlanBig(int a, int e_, int P_) : e(e_), P(P_), jt(a) {
    lp2 = (P_ & (P_ - 1)) == 0 ? __ffs(P_) - 1 : -1;
  }
  __device__ bool done() const { return jt > e; }
  __device__ Tile next(int& lpage, int& slot0) {
    const int lp = lp2 >= 0 ? (jt >> lp2) : jt / P;
    const int pstart = lp * P;
    const int pe = pstart + P - 1;
    int et = min(jt + 63, pe);
    et = min(et, e);
    const bool rev = (et == e) && (jt == pstart) && (et - jt < 63);
    Tile t;
    t.jbase = rev ? et - 63 : jt;
    t.klo = jt;
    t.khi = et;
    t.dirty = !rev && (et == e) && (et < pe) && (et - jt < 63);
    lpage = lp;
    slot0 = t.jbase - pstart;
    jt = et + 1;
    return t;
  }
};

// Tile walk for other page sizes (multiple of 16): 64-aligned logical blocks,
// each assembled from four 16-row boxes; boxes with no valid key are skipped
// (their rows keep stale data, so a partial block is dirty).
struct PlanSmall {
  int a, e, jt;
  __device__ PlanSmall(int a_, int e_) : a(a_), e(e_), jt(a_ & ~63) {}
  __device__ bool done() const { return jt > e; }
  __device__ Tile next() {
    Tile t;
    t.jbase = jt;
    t.klo = max(a, jt);
    t.khi = min(e, jt + 63);
    t.dirty = (t.klo != jt) || (t.khi != jt + 63);
    jt += 64;
    return t;
  }
};

__device__ __forceinline__ void report(int32_t* err, int bit) {
  if (err) atomicOr(err, bit);
}


}  // namespace ira
