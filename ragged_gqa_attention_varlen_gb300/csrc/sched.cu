// sched.cu -- the ragged tile scheduler, the D = rowsum(dO * O) preprocess
// of the backward pass, and fill kernels for degenerate sizes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/attn_varlen.h"
#include "attn_internal.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

// One block.  Validates cu_q/cu_k, resets the status word and the tile
// counters, and builds both tile orders (see attn_internal.h for the array
// layout).  Sorting is by counting rank (descending work, ties by index), so
// the order is a deterministic function of the lengths.
__global__ void __launch_bounds__(1024) sched_kernel(Params p) {
  const int B = p.B;
  const int tid = threadIdx.x;
  __shared__ int bad;
  if (tid == 0) {
    bad = (p.cu_q[0] != 0 || p.cu_k[0] != 0 || p.cu_q[B] != p.total_q ||
           p.cu_k[B] != p.total_k);
  }
  __syncthreads();
  for (int b = tid; b < B; b += blockDim.x) {
    if (p.cu_q[b + 1] < p.cu_q[b] || p.cu_k[b + 1] < p.cu_k[b]) atomicOr(&bad, 1);
  }
  __syncthreads();
  int32_t* ord_f = p.sched;
  int32_t* pre_f = p.sched + B;
  int32_t* ord_b = p.sched + 2 * B + 1;
  int32_t* pre_b = p.sched + 3 * B + 1;
  int32_t* kt0_b = p.sched + 4 * B + 2;
  if (bad) {
    // No tiles: every later kernel finds nothing to do.
    for (int b = tid; b <= B; b += blockDim.x) {
      pre_f[b] = 0;
      pre_b[b] = 0;
      if (b < B) {
        ord_f[b] = 0;
        ord_b[b] = 0;
        kt0_b[b] = 0;
      }
    }
    if (tid == 0) *p.status = ATTN_DEV_BAD_CU;
    return;
  }
  if (tid == 0) {
    *p.status = 0;
    for (int i = 0; i < p.ncounters; ++i) p.counters[i] = 0;
  }
  // per-token dropout thresholds and scales
  if (p.drop_tab)
    for (int64_t t = tid; t < p.total_q; t += blockDim.x) {
      uint32_t T;
      float sc;
      drop_params(p.drop_rates[t], T, sc);
      p.drop_tab[t] = make_uint2(T, __float_as_uint(sc));
    }
  // The work of a sequence's longest forward/dq tile grows with the keys it
  // visits, of a dk/dv tile with the queries: the whole other length, or
  // under a window bounded on both sides about the window's span.
  const int wr = right_window(p);
  const bool banded = p.wl >= 0 && wr >= 0;
  const int64_t span_f = banded ? static_cast<int64_t>(p.wl) + wr + kRowsQ / p.G + kKeys : 0;
  const int64_t span_b = banded ? static_cast<int64_t>(p.wl) + wr + kKeys + kRowsQ / p.G : 0;
  auto work_f = [&](int c) -> int64_t {
    const int64_t lk = p.cu_k[c + 1] - p.cu_k[c];
    return banded ? min(lk, span_f) : lk;
  };
  auto work_b = [&](int c) -> int64_t {
    const int64_t lq = p.cu_q[c + 1] - p.cu_q[c];
    return banded ? min(lq, span_b) : lq;
  };
  for (int b = tid; b < B; b += blockDim.x) {
    const int64_t lk = work_f(b), lq = work_b(b);
    int rf = 0, rb = 0;
    for (int c = 0; c < B; ++c) {
      const int64_t lkc = work_f(c), lqc = work_b(c);
      rf += (lkc > lk) || (lkc == lk && c < b);
      rb += (lqc > lq) || (lqc == lq && c < b);
    }
    ord_f[rf] = b;
    ord_b[rb] = b;
  }
  __syncthreads();
  if (tid == 0) {
    const int rows_tok = kRowsQ / p.G;
    const int ngroups = p.Hq / p.G;
    int acc_f = 0, acc_b = 0;
    for (int r = 0; r < B; ++r) {
      pre_f[r] = acc_f;
      pre_b[r] = acc_b;
      int bf = ord_f[r], bb = ord_b[r];
      int lq = p.cu_q[bf + 1] - p.cu_q[bf];
      acc_f += ((lq + rows_tok - 1) / rows_tok) * ngroups;
      int kt0, nkt;
      dkdv_key_span(p, p.cu_q[bb + 1] - p.cu_q[bb], p.cu_k[bb + 1] - p.cu_k[bb], kt0, nkt);
      kt0_b[r] = kt0;
      acc_b += nkt;
    }
    pre_f[B] = acc_f;
    pre_b[B] = acc_b;
    // stored keep mask: the per-sequence block prefix (its header) and the
    // check that the caller's buffer holds every K/V head group's blocks
    if (p.drop_mask) {
      int32_t* mp = reinterpret_cast<int32_t*>(p.drop_mask);
      int64_t acc = 0;
      for (int b = 0; b < B; ++b) {
        mp[b] = static_cast<int32_t>(acc);
        const int64_t lq = p.cu_q[b + 1] - p.cu_q[b], lk = p.cu_k[b + 1] - p.cu_k[b];
        acc += (lq + rows_tok - 1) / rows_tok * ngroups * ((lk + kKeys - 1) / kKeys);
      }
      mp[B] = static_cast<int32_t>(acc);
      const uint64_t need = drop_mask_header(B) + static_cast<uint64_t>(acc) * p.Hkv *
                                                      (8ull * kMaskBlockWords);
      if (acc > INT32_MAX || need > p.drop_mask_bytes) *p.status = ATTN_DEV_MASK_SPACE;
    }
  }
}

cudaError_t launch_sched(const Params& p, cudaStream_t s) {
  sched_kernel<<<1, 1024, 0, s>>>(p);
  return cudaGetLastError();
}

// The stored keep mask of a dropout call: every block of every K/V head
// group (layout in attn_internal.h).  CTA c takes a contiguous run of blocks
// in layout order, so it decodes (group, sequence, token block, head group,
// key tile) once and then steps through them; thread w writes word w of each
// block -- query row r = w % 128 of the tile, keys 64 (w / 128) .. + 63 of
// the key tile -- from the counter-based hash the forward and backward
// kernels would otherwise evaluate, zero for rows past the sequence.
// Launched with group 0's parameters (Hq = heads per K/V head).
__global__ void __launch_bounds__(256) mask_kernel(Params p) {
  if (*p.status != 0) return;
  const int32_t* pre = reinterpret_cast<const int32_t*>(p.drop_mask);
  const int64_t per_group = pre[p.B];
  const int64_t total = per_group * p.Hkv;
  const int64_t chunk = (total + gridDim.x - 1) / gridDim.x;
  int64_t n = static_cast<int64_t>(blockIdx.x) * chunk;
  const int64_t n_end = min(total, n + chunk);
  if (n >= n_end) return;
  const int G = p.G;
  const int rows_tok = kRowsQ / G;
  const int ngroups = p.Hq / G;
  uint64_t* words = reinterpret_cast<uint64_t*>(p.drop_mask + drop_mask_header(p.B));
  const int w = threadIdx.x;
  const int kh = w / kRowsQ, r = w % kRowsQ;
  const int rtok = r / G, rhead = r % G;
  // decode the run's first block
  int g = static_cast<int>(n / per_group);
  const int local = static_cast<int>(n - static_cast<int64_t>(g) * per_group);
  int b = 0;
  {
    int lo = 0, hi = p.B - 1;  // largest b with pre[b] <= local
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= local)
        lo = mid;
      else
        hi = mid - 1;
    }
    b = lo;
  }
  int q0 = 0, Lq = 0, nkt = 1, ntb = 1;
  uint64_t dkb = 0;
  auto enter = [&]() {  // sequence b's lengths and hash key
    q0 = p.cu_q[b];
    Lq = p.cu_q[b + 1] - q0;
    nkt = (p.cu_k[b + 1] - p.cu_k[b] + kKeys - 1) / kKeys;
    ntb = (Lq + rows_tok - 1) / rows_tok;
    dkb = splitmix64(p.drop_seed ^ static_cast<uint64_t>(b));
  };
  enter();
  int blk = local - pre[b];
  int kt = blk % nkt;
  blk /= nkt;
  int hg = blk % ngroups;
  int tb = blk / ngroups;
  for (; n < n_end; ++n) {
    const int i = tb * rows_tok + rtok;
    uint64_t bits = 0;
    if (i < Lq) {
      uint32_t T;
      float sc;
      drop_row(p, static_cast<int64_t>(q0) + i, T, sc);
      const uint64_t dhi = drop_hi(g * p.Hq + hg * G + rhead, i);
      const int key0 = kt * kKeys + kh * 64;
#pragma unroll 4
      for (int c = 0; c < 64; c += 4)
        bits |= static_cast<uint64_t>(drop_keep4(drop_hash(dkb, dhi, (key0 + c) >> 2), T)) << c;
    }
    words[n * kMaskBlockWords + w] = bits;
    // the next block in layout order (sequences without blocks are skipped)
    if (++kt == nkt) {
      kt = 0;
      if (++hg == ngroups) {
        hg = 0;
        if (++tb == ntb) {
          tb = 0;
          do {
            if (++b == p.B) {
              b = 0;
              ++g;
            }
          } while (pre[b + 1] == pre[b] && n + 1 < n_end);
          enter();
        }
      }
    }
  }
}

cudaError_t launch_mask(const Params& p, cudaStream_t s) {
  mask_kernel<<<152 * 8, 256, 0, s>>>(p);
  return cudaGetLastError();
}

// D[t, h] = sum_f dO[t,h,f] * O[t,h,f] in fp32 over the stored (rounded)
// output, for every head of the call (D row stride = Hq = lse_rs).  One warp
// per (token, head) row; lanes 0..19 each take 8 features.
template <typename T>
__device__ __forceinline__ float dot8(uint4 a, uint4 b);

template <>
__device__ __forceinline__ float dot8<__half>(uint4 a, uint4 b) {
  const __half2* x = reinterpret_cast<const __half2*>(&a);
  const __half2* y = reinterpret_cast<const __half2*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 fx = __half22float2(x[i]), fy = __half22float2(y[i]);
    acc = fmaf(fx.x, fy.x, acc);
    acc = fmaf(fx.y, fy.y, acc);
  }
  return acc;
}

template <>
__device__ __forceinline__ float dot8<__nv_bfloat16>(uint4 a, uint4 b) {
  const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
  const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 fx = __bfloat1622float2(x[i]), fy = __bfloat1622float2(y[i]);
    acc = fmaf(fx.x, fy.x, acc);
    acc = fmaf(fx.y, fy.y, acc);
  }
  return acc;
}

template <typename T>
__global__ void __launch_bounds__(256) preprocess_kernel(Params p) {
  if (*p.status != 0) return;
  const int64_t rows = p.total_q * p.Hq;
  const int lane = threadIdx.x & 31;
  int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t stride_rows = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const T* o = static_cast<const T*>(p.outp);
  const T* d = static_cast<const T*>(p.dout);
  for (; row < rows; row += stride_rows) {
    const int64_t t = row / p.Hq;
    const int h = static_cast<int>(row - t * p.Hq);
    float acc = 0.f;
    if (lane < p.d / 8) {
      uint4 a = *reinterpret_cast<const uint4*>(o + t * p.out_ts + h * p.out_hs + lane * 8);
      uint4 b = *reinterpret_cast<const uint4*>(d + t * p.do_ts + h * p.do_hs + lane * 8);
      acc = dot8<T>(a, b);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) p.Dbuf[row] = acc;
  }
  // dk = dv = 0 (every K/V head) for the keys outside every scheduled dk/dv
  // tile: keys of sequences without queries and keys the mask leaves
  // unreached.  The dk/dv kernel writes every other key row.
  const int64_t kstride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t krow = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       krow < p.total_k; krow += kstride) {
    int lo = 0, hi = p.B - 1;  // the last sequence with cu_k[b] <= krow
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.cu_k[mid] <= krow)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int k0 = p.cu_k[lo];
    const int Lk = p.cu_k[lo + 1] - k0;
    const int j = static_cast<int>(krow - k0);
    int kt0, nkt;
    dkdv_key_span(p, p.cu_q[lo + 1] - p.cu_q[lo], Lk, kt0, nkt);
    if (j >= Lk || (nkt > 0 && j >= kt0 * kKeys && j < (kt0 + nkt) * kKeys)) continue;
    for (int g = 0; g < p.Hkv; ++g) {
      uint4* dk = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dk) + krow * p.dk_ts +
                                           g * p.dk_hs);
      uint4* dv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dv) + krow * p.dv_ts +
                                           g * p.dv_hs);
      for (int u = 0; u < p.d / 8; ++u) {
        dk[u] = make_uint4(0u, 0u, 0u, 0u);
        dv[u] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (p.dkg) {  // the gate's key projections (gated calls)
        uint4* dg = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dkg) + krow * p.dkg_ts +
                                             g * p.dkg_hs);
        for (int u = 0; u < p.R / 8; ++u) dg[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
}

cudaError_t launch_preprocess(const Params& p, cudaStream_t s) {
  const int64_t rows = p.total_q * p.Hq;
  if (rows == 0 && p.total_k == 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (p.dtype == 1)
    preprocess_kernel<__nv_bfloat16><<<static_cast<int>(blocks), 256, 0, s>>>(p);
  else
    preprocess_kernel<__half><<<static_cast<int>(blocks), 256, 0, s>>>(p);
  return cudaGetLastError();
}

// Zero a strided [T, H, d] 16-bit tensor, 16 bytes per thread.
__global__ void zero_fill_kernel(uint16_t* base, int64_t T, int H, int64_t ts, int64_t hs,
                                 int d) {
  const int per_row = d / 8;
  const int64_t units = T * H * per_row;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int64_t row = u / per_row;
    int c = static_cast<int>(u - row * per_row);
    int64_t t = row / H;
    int h = static_cast<int>(row - t * H);
    *reinterpret_cast<uint4*>(base + t * ts + h * hs + c * 8) = make_uint4(0, 0, 0, 0);
  }
}

cudaError_t launch_zero_fill(void* base, int64_t T, int H, int64_t ts, int64_t hs, int d,
                             cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  zero_fill_kernel<<<152 * 8, 256, 0, s>>>(static_cast<uint16_t*>(base), T, H, ts, hs, d);
  return cudaGetLastError();
}

__global__ void fill_f32_kernel(float* base, int64_t n, float value) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    base[i] = value;
}

cudaError_t launch_fill_f32(float* base, int64_t n, float value, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  fill_f32_kernel<<<152 * 4, 256, 0, s>>>(base, n, value);
  return cudaGetLastError();
}

}  // namespace attn
