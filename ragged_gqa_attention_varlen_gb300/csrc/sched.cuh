// sched.cuh -- decoding of the device-built ragged tile schedule.
//
// The schedule kernel (sched.cu) sorts the sequences by the work of one of
// their tiles, longest first, and stores per order position the prefix count
// of tiles.  Persistent kernels draw tile numbers from a counter in that
// order, so the longest tiles start first (longest-processing-time greedy
// list scheduling).  Which CTA runs a tile never changes what the tile
// computes, so results stay bitwise reproducible.
#pragma once
#include "attn_internal.h"
#include "sm103.cuh"

namespace attn {

// One forward/dq tile: kRowsQ/G tokens of one sequence times G heads.
struct QTile {
  int b;        // sequence
  int tok;      // first local query token of the tile
  int hg;       // head group (heads hg*G .. hg*G+G-1)
  int Lq, Lk;   // sequence lengths
  int q0, k0;   // packed offsets of the sequence's first query / key
  int kt0, nkt; // key tiles [kt0, kt0 + nkt) hold every key the tile's queries may attend to
};

// One dk/dv tile: kKeys keys of one sequence.
struct KTile {
  int b, key, Lq, Lk, q0, k0;
  int tb0, ntb;  // query blocks [tb0, tb0 + ntb) (kRowsQ/G tokens each) that may attend to it
};

__device__ __forceinline__ bool masking(const Params& p) {
  return p.causal || p.wl >= 0 || p.wr >= 0;
}

// Right window of the mask (causal caps it at 0); negative = unbounded.
__device__ __forceinline__ int right_window(const Params& p) { return p.causal ? 0 : p.wr; }

// Key j of local query i is admissible when i + Lk - Lq - wl <= j <= i + Lk - Lq + wr
// (each bound only where its window is set).  Tiles whose every pair fails
// this are skipped: they would contribute P = 0 exactly.

// Key tiles [*kt0, *kt0 + *nkt) cover every key that a query of local tokens
// [qa, qb] may attend to (nkt = 0 when none may attend to any key).
__device__ __forceinline__ void key_tile_span(const Params& p, int Lq, int Lk, int qa, int qb,
                                              int& kt0, int& nkt) {
  int64_t lo = 0, hi = static_cast<int64_t>(Lk) - 1;
  if (masking(p)) {
    const int64_t off = static_cast<int64_t>(Lk) - Lq;
    const int wr = right_window(p);
    if (p.wl >= 0) lo = max(lo, qa + off - p.wl);
    if (wr >= 0) hi = min(hi, qb + off + wr);
  }
  if (lo > hi) {
    kt0 = 0;
    nkt = 0;
    return;
  }
  kt0 = static_cast<int>(lo / kKeys);
  nkt = static_cast<int>(hi / kKeys) - kt0 + 1;
}

// Query blocks [*tb0, *tb0 + *ntb) of `blk` tokens cover every query that may
// attend to a key of local keys [ja, jb].
__device__ __forceinline__ void query_block_span(const Params& p, int Lq, int Lk, int ja, int jb,
                                                 int blk, int& tb0, int& ntb) {
  int64_t lo = 0, hi = static_cast<int64_t>(Lq) - 1;
  if (masking(p)) {
    const int64_t off = static_cast<int64_t>(Lk) - Lq;
    const int wr = right_window(p);
    if (wr >= 0) lo = max(lo, ja - off - wr);
    if (p.wl >= 0) hi = min(hi, jb - off + p.wl);
  }
  if (lo > hi) {
    tb0 = 0;
    ntb = 0;
    return;
  }
  tb0 = static_cast<int>(lo / blk);
  ntb = static_cast<int>(hi / blk) - tb0 + 1;
}

// Key tiles [*kt0, *kt0 + *nkt) of a sequence hold every key that some query
// may attend to (the admissible keys form one run: j >= Lk - Lq - wl and
// j <= Lq - 1 + Lk - Lq + wr where the windows are set).  The dk/dv schedule
// holds only these tiles, so no dk/dv tile is without queries; the rows of
// the other keys are zeroed by the dk/dv kernel's prologue.
__device__ __forceinline__ void dkdv_key_span(const Params& p, int Lq, int Lk, int& kt0,
                                              int& nkt) {
  int64_t lo = 0, hi = static_cast<int64_t>(Lk) - 1;
  if (masking(p)) {
    const int64_t off = static_cast<int64_t>(Lk) - Lq;
    const int wr = right_window(p);
    if (p.wl >= 0) lo = max(lo, off - p.wl);
    if (wr >= 0) hi = min(hi, static_cast<int64_t>(Lq) - 1 + off + wr);
  }
  if (Lq == 0 || lo > hi) {
    kt0 = 0;
    nkt = 0;
    return;
  }
  kt0 = static_cast<int>(lo / kKeys);
  nkt = static_cast<int>(hi / kKeys) - kt0 + 1;
}

// Under a mask whose admissible keys grow with the query (a right bound and
// no left bound: causal) the query tiles of a sequence are drawn last token
// block first, and under the mirror case the key tiles last tile first, so
// the longest tiles of a sequence start first.
__device__ __forceinline__ bool qtiles_reversed(const Params& p) {
  return p.wl < 0 && right_window(p) >= 0;
}
__device__ __forceinline__ bool ktiles_reversed(const Params& p) {
  return p.wl >= 0 && right_window(p) < 0;
}

// Largest r in [0, B) with pre[r] <= n.
__device__ __forceinline__ int sched_find(const int32_t* pre, int B, int n) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(pre + mid) <= n)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int qtile_count(const Params& p) { return __ldg(p.sched + 2 * p.B); }
__device__ __forceinline__ int ktile_count(const Params& p) {
  return __ldg(p.sched + 4 * p.B + 1);
}

// MASK: the call has a causal/window mask (kernels are instantiated for both
// cases, so the unmasked instance carries none of the span arithmetic).
template <bool MASK>
__device__ __forceinline__ void qtile_decode(const Params& p, int n, QTile& t) {
  const int32_t* ord = p.sched;
  const int32_t* pre = p.sched + p.B;
  int r = sched_find(pre, p.B, n);
  int b = __ldg(ord + r);
  int local = n - __ldg(pre + r);
  int ngroups = p.Hq / p.G;
  const int rows_tok = kRowsQ / p.G;
  t.b = b;
  t.q0 = __ldg(p.cu_q + b);
  t.k0 = __ldg(p.cu_k + b);
  t.Lq = __ldg(p.cu_q + b + 1) - t.q0;
  t.Lk = __ldg(p.cu_k + b + 1) - t.k0;
  int blk = local / ngroups;
  if (MASK && qtiles_reversed(p)) blk = (t.Lq + rows_tok - 1) / rows_tok - 1 - blk;
  t.tok = blk * rows_tok;
  t.hg = local % ngroups;
  if (MASK) {
    key_tile_span(p, t.Lq, t.Lk, t.tok, min(t.tok + rows_tok, t.Lq) - 1, t.kt0, t.nkt);
  } else {
    t.kt0 = 0;
    t.nkt = (t.Lk + kKeys - 1) / kKeys;
  }
}

template <bool MASK>
__device__ __forceinline__ void ktile_decode(const Params& p, int n, KTile& t) {
  const int32_t* ord = p.sched + 2 * p.B + 1;
  const int32_t* pre = p.sched + 3 * p.B + 1;
  int r = sched_find(pre, p.B, n);
  int b = __ldg(ord + r);
  t.b = b;
  t.q0 = __ldg(p.cu_q + b);
  t.k0 = __ldg(p.cu_k + b);
  t.Lq = __ldg(p.cu_q + b + 1) - t.q0;
  t.Lk = __ldg(p.cu_k + b + 1) - t.k0;
  int kt = n - __ldg(pre + r);
  if (MASK && ktiles_reversed(p)) kt = __ldg(pre + r + 1) - __ldg(pre + r) - 1 - kt;
  kt += __ldg(p.sched + 4 * p.B + 2 + r);  // the sequence's first scheduled key tile
  t.key = kt * kKeys;
  if (MASK) {
    query_block_span(p, t.Lq, t.Lk, t.key, min(t.key + kKeys, t.Lk) - 1, kRowsQ / p.G, t.tb0,
                     t.ntb);
  } else {
    const int blk = kRowsQ / p.G;
    t.tb0 = 0;
    t.ntb = (t.Lq + blk - 1) / blk;
  }
}

// Block (tb, hg, kt) of sequence b in this K/V head group's part of the
// stored keep mask (layout in attn_internal.h).
__device__ __forceinline__ uint64_t* drop_mask_block(const Params& p, int b, int Lk, int tb,
                                                     int hg, int kt) {
  const int32_t* pre = reinterpret_cast<const int32_t*>(p.drop_mask);
  const int64_t nkt = (Lk + kKeys - 1) / kKeys;
  const int64_t g = p.head0 / p.Hq;
  const int64_t blk = g * __ldg(pre + p.B) + __ldg(pre + b) +
                      (static_cast<int64_t>(tb) * (p.Hq / p.G) + hg) * nkt + kt;
  return reinterpret_cast<uint64_t*>(p.drop_mask + drop_mask_header(p.B)) +
         blk * kMaskBlockWords;
}

// Dynamic tile stream of a persistent CTA.  Warp 0 draws tile numbers from
// a global counter (so tiles start in the schedule's longest-first order)
// and publishes them through a four-deep ring in shared memory; every other
// role of the CTA reads the same sequence, which ends with -1.  What a tile
// computes never depends on which CTA computes it, so drawing tiles at run
// time keeps the results bitwise repeatable, while SMs that run faster take
// more tiles (the SMs of one GPU were measured to differ by up to ~10 %).
struct TileRing {
  int32_t item[4];
  uint64_t full[4], empty[4];
};

__device__ __forceinline__ void tile_ring_init(TileRing* r, uint32_t consumers) {
  for (int s = 0; s < 4; ++s) {
    mbar_init(&r->full[s], 1);
    mbar_init(&r->empty[s], consumers);
  }
}

// Whole warp: draw the next tile, publish it as entry k (or -1 when none is
// left) and return it in *out.  False if a wait gave up.
__device__ __forceinline__ bool tile_publish(TileRing* r, uint32_t& k, int32_t* counter,
                                             int ntiles, int* out, volatile int* abort) {
  const int slot = k & 3;
  if (k >= 4 && !mbar_wait_warp(&r->empty[slot], ((k >> 2) - 1) & 1, abort)) return false;
  int it = 0;
  if ((threadIdx.x & 31) == 0) {
    it = atomicAdd(counter, 1);
    if (it >= ntiles) it = -1;
    r->item[slot] = it;
  }
  it = __shfl_sync(0xffffffffu, it, 0);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&r->full[slot]);
  ++k;
  *out = it;
  return true;
}

// One thread: read entry k of the stream.
__device__ __forceinline__ bool tile_take(TileRing* r, uint32_t& k, int* out,
                                          volatile int* abort) {
  const int slot = k & 3;
  if (!mbar_wait(&r->full[slot], (k >> 2) & 1, abort)) return false;
  *out = *reinterpret_cast<volatile int32_t*>(&r->item[slot]);
  mbar_arrive(&r->empty[slot]);
  ++k;
  return true;
}

// Whole warp: read entry k of the stream (one arrival for the warp).
__device__ __forceinline__ bool tile_take_warp(TileRing* r, uint32_t& k, int* out,
                                               volatile int* abort) {
  const int slot = k & 3;
  if (!mbar_wait_warp(&r->full[slot], (k >> 2) & 1, abort)) return false;
  *out = *reinterpret_cast<volatile int32_t*>(&r->item[slot]);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&r->empty[slot]);
  ++k;
  return true;
}

// Key j of local query i is admissible under the causal/window mask.
__device__ __forceinline__ bool admissible(const Params& p, int Lq, int Lk, int i, int j) {
  int k0 = i + Lk - Lq;
  int wr = right_window(p);
  if (p.wl >= 0 && j < k0 - p.wl) return false;
  if (wr >= 0 && j > k0 + wr) return false;
  return true;
}

// Every key of local keys [ja, jb] is admissible for local query i.
__device__ __forceinline__ bool all_admissible(const Params& p, int Lq, int Lk, int i, int ja,
                                               int jb) {
  const int64_t k0 = static_cast<int64_t>(i) + Lk - Lq;
  const int wr = right_window(p);
  return (p.wl < 0 || ja >= k0 - p.wl) && (wr < 0 || jb <= k0 + wr);
}

}  // namespace attn
