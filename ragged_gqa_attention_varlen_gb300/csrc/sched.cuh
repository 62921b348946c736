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
