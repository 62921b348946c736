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
};

// One dk/dv tile: kKeys keys of one sequence.
struct KTile {
  int b, key, Lq, Lk, q0, k0;
};

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

__device__ __forceinline__ void qtile_decode(const Params& p, int n, QTile& t) {
  const int32_t* ord = p.sched;
  const int32_t* pre = p.sched + p.B;
  int r = sched_find(pre, p.B, n);
  int b = __ldg(ord + r);
  int local = n - __ldg(pre + r);
  int ngroups = p.Hq / p.G;
  t.b = b;
  t.tok = (local / ngroups) * (kRowsQ / p.G);
  t.hg = local % ngroups;
  t.q0 = __ldg(p.cu_q + b);
  t.k0 = __ldg(p.cu_k + b);
  t.Lq = __ldg(p.cu_q + b + 1) - t.q0;
  t.Lk = __ldg(p.cu_k + b + 1) - t.k0;
}

__device__ __forceinline__ void ktile_decode(const Params& p, int n, KTile& t) {
  const int32_t* ord = p.sched + 2 * p.B + 1;
  const int32_t* pre = p.sched + 3 * p.B + 1;
  int r = sched_find(pre, p.B, n);
  int b = __ldg(ord + r);
  t.b = b;
  t.key = (n - __ldg(pre + r)) * kKeys;
  t.q0 = __ldg(p.cu_q + b);
  t.k0 = __ldg(p.cu_k + b);
  t.Lq = __ldg(p.cu_q + b + 1) - t.q0;
  t.Lk = __ldg(p.cu_k + b + 1) - t.k0;
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
  int wr = p.causal ? 0 : p.wr;
  if (p.wl >= 0 && j < k0 - p.wl) return false;
  if (wr >= 0 && j > k0 + wr) return false;
  return true;
}

__device__ __forceinline__ bool masking(const Params& p) {
  return p.causal || p.wl >= 0 || p.wr >= 0;
}

}  // namespace attn
