// shard.cu -- one batch over several processes (one GPU each): the shard
// plan and the fixed-order sum of partial key gradients.
//
// Sequences are independent problems, so a batch shards by sequence with no
// exchange: each rank takes whole sequences, assigned longest processing
// time first on their work Hq * (admissible query-key pairs).  A sequence
// with more than 1/N of the batch's work would leave the other ranks idle,
// so its heads are split over several ranks.  With one K/V head every part
// holds a partial dk/dv of the sequence's keys (each part sums over its own
// query heads only); the parts are added in the order of their first head
// on the rank that holds part 0 -- the one exchange step of the sharded path.
// With several K/V heads a sequence is split only between K/V head groups,
// whose dk/dv rows are disjoint, so no partial sums arise.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/attn_varlen.h"

namespace {

// Admissible (query, key) pairs of one sequence under the mask: key j is
// admissible for query i when i + Lk - Lq - wl <= j <= i + Lk - Lq + wr
// (each bound only where its window is set; causal caps wr at 0).
double admissible_pairs(int64_t Lq, int64_t Lk, int causal, int wl, int wr_in) {
  const int wr = causal ? 0 : wr_in;
  if (wl < 0 && wr < 0) return static_cast<double>(Lq) * static_cast<double>(Lk);
  double n = 0;
  for (int64_t i = 0; i < Lq; ++i) {
    const int64_t k0 = i + Lk - Lq;
    const int64_t lo = wl >= 0 ? std::max<int64_t>(0, k0 - wl) : 0;
    const int64_t hi = wr >= 0 ? std::min<int64_t>(Lk - 1, k0 + wr) : Lk - 1;
    if (hi >= lo) n += static_cast<double>(hi - lo + 1);
  }
  return n;
}

struct Unit {
  int seq, h0, h1, part;  // part: index among the sequence's parts (0 if whole)
  double work;
  int rank;
};

template <bool BF16>
struct Cvt;
template <>
struct Cvt<true> {
  __device__ static float2 in(uint32_t v) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
  }
  __device__ static uint32_t out(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};
template <>
struct Cvt<false> {
  __device__ static float2 in(uint32_t v) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
  }
  __device__ static uint32_t out(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
};

constexpr int kMaxParts = 16;
struct Parts {
  const uint16_t* p[kMaxParts];
};

// out[r, :] = sum over parts in index order of part[r, :], accumulated in
// fp32 and rounded once; one thread per 8 features of a row.
template <bool BF16>
__global__ void sum_parts_kernel(Parts parts, int nparts, int64_t rows, int units_per_row,
                                 int64_t part_rs, uint16_t* out, int64_t out_rs) {
  const int64_t n = rows * units_per_row;
  for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < n;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = t / units_per_row;
    const int u = static_cast<int>(t % units_per_row);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int k = 0; k < nparts; ++k) {
      const uint4 w = *reinterpret_cast<const uint4*>(parts.p[k] + r * part_rs + u * 8);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = Cvt<BF16>::in(ws[e]);
        acc[2 * e] += f.x;
        acc[2 * e + 1] += f.y;
      }
    }
    uint4 o;
    o.x = Cvt<BF16>::out(acc[0], acc[1]);
    o.y = Cvt<BF16>::out(acc[2], acc[3]);
    o.z = Cvt<BF16>::out(acc[4], acc[5]);
    o.w = Cvt<BF16>::out(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(out + r * out_rs + u * 8) = o;
  }
}

}  // namespace

extern "C" int attn_varlen_shard_plan(int B, const int32_t* cu_q, const int32_t* cu_k, int Hq,
                                      int Hkv, int causal, int window_left, int window_right,
                                      int nranks, int max_units, int32_t* unit_seq,
                                      int32_t* unit_h0, int32_t* unit_h1, int32_t* unit_rank,
                                      double* rank_work) {
  if (B < 0 || Hq <= 0 || Hkv < 1 || Hq % Hkv || nranks < 1 || nranks > kMaxParts ||
      max_units < 0 || (B > 0 && (!cu_q || !cu_k)) || !unit_seq || !unit_h0 || !unit_h1 ||
      !unit_rank || !rank_work)
    return -1;
  for (int b = 0; b < B; ++b)
    if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return -1;
  std::vector<double> w(static_cast<size_t>(B));
  double total = 0;
  for (int b = 0; b < B; ++b) {
    w[b] = static_cast<double>(Hq) * admissible_pairs(cu_q[b + 1] - cu_q[b],
                                                      cu_k[b + 1] - cu_k[b], causal,
                                                      window_left, window_right);
    total += w[b];
  }
  const double target = total / nranks;
  const int R = Hq / Hkv;
  std::vector<Unit> units;
  for (int b = 0; b < B; ++b) {
    int k = 1;
    if (nranks > 1 && w[b] > target) {
      k = static_cast<int>(std::min<double>(nranks, std::ceil(w[b] / target)));
      k = std::min(k, Hkv > 1 ? Hkv : Hq);
    }
    for (int e = 0; e < k; ++e) {
      int h0, h1;
      if (Hkv > 1) {  // whole K/V head groups
        h0 = static_cast<int>(static_cast<int64_t>(e) * Hkv / k) * R;
        h1 = static_cast<int>(static_cast<int64_t>(e + 1) * Hkv / k) * R;
      } else {
        h0 = static_cast<int>(static_cast<int64_t>(e) * Hq / k);
        h1 = static_cast<int>(static_cast<int64_t>(e + 1) * Hq / k);
      }
      units.push_back(Unit{b, h0, h1, e, w[b] * (h1 - h0) / Hq, -1});
    }
  }
  if (static_cast<int>(units.size()) > max_units) return -1;
  // longest processing time first: the heaviest unit goes to the least
  // loaded rank (the lowest such rank on ties); parts of one sequence go to
  // different ranks while one is free of it
  std::vector<int> order(units.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = static_cast<int>(i);
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int c) { return units[a].work > units[c].work; });
  std::vector<double> load(static_cast<size_t>(nranks), 0.0);
  std::vector<std::vector<int>> holds(static_cast<size_t>(B));
  for (int i : order) {
    Unit& u = units[i];
    int best = -1;
    for (int pass = 0; pass < 2 && best < 0; ++pass)
      for (int r = 0; r < nranks; ++r) {
        const auto& hs = holds[u.seq];
        if (pass == 0 && std::find(hs.begin(), hs.end(), r) != hs.end()) continue;
        if (best < 0 || load[r] < load[best]) best = r;
      }
    u.rank = best;
    load[best] += u.work;
    holds[u.seq].push_back(best);
  }
  for (size_t i = 0; i < units.size(); ++i) {
    unit_seq[i] = units[i].seq;
    unit_h0[i] = units[i].h0;
    unit_h1[i] = units[i].h1;
    unit_rank[i] = units[i].rank;
  }
  for (int r = 0; r < nranks; ++r) rank_work[r] = load[r];
  return static_cast<int>(units.size());
}

extern "C" attn_status attn_varlen_sum_partials(attn_dtype dtype, int nparts,
                                                const void* const* parts, int64_t rows, int d,
                                                int64_t part_row_stride, void* out,
                                                int64_t out_row_stride, void* stream) {
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
  if (nparts < 1 || nparts > kMaxParts || !parts || rows < 0 || d <= 0 || !out)
    return ATTN_ERR_INVALID;
  if (d % 8 || part_row_stride % 8 || out_row_stride % 8 || part_row_stride < d ||
      out_row_stride < d || (reinterpret_cast<uintptr_t>(out) & 15u))
    return ATTN_ERR_ALIGNMENT;
  Parts ps = {};
  for (int k = 0; k < nparts; ++k) {
    if (!parts[k]) return ATTN_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(parts[k]) & 15u) return ATTN_ERR_ALIGNMENT;
    ps.p[k] = static_cast<const uint16_t*>(parts[k]);
  }
  if (rows == 0) return ATTN_OK;
  const int upr = d / 8;
  const int64_t n = rows * upr;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<int64_t>((n + threads - 1) / threads, 4096));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == ATTN_BF16)
    sum_parts_kernel<true><<<blocks, threads, 0, s>>>(ps, nparts, rows, upr, part_row_stride,
                                                      static_cast<uint16_t*>(out), out_row_stride);
  else
    sum_parts_kernel<false><<<blocks, threads, 0, s>>>(ps, nparts, rows, upr, part_row_stride,
                                                       static_cast<uint16_t*>(out), out_row_stride);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
