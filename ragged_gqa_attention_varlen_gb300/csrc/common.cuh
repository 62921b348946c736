// common.cuh -- per-element arithmetic shared by the attention kernels:
// the logit map's constants, counter-based dropout and 16-bit packing.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_internal.h"
#include "sm103.cuh"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// SplitMix64's output function (Steele, Lea and Flood, OOPSLA 2014): a Weyl
// increment, two xor-shift-multiply rounds and a final xor-shift.
__host__ __device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Threshold and scale of a dropout rate: keep when an element's 16-bit draw
// is >= T (probability 1 - T / 2^16), and scale kept values by 1/(1 - rate).
__host__ __device__ __forceinline__ void drop_params(float rate, uint32_t& T, float& scale) {
  if (!(rate < 1.f)) {
    T = 1u << 16;
    scale = 0.f;
  } else if (!(rate > 0.f)) {
    T = 0u;
    scale = 1.f;
  } else {
    T = static_cast<uint32_t>(rate * 65536.0f);
    scale = 1.f / (1.f - rate);
  }
}

// The hash of the four keys 4m .. 4m + 3 of one row: `kb` =
// splitmix64(seed ^ b), `hi` = h << 48 | i << 24, `m` = key / 4.  Key 4m + f
// draws the 16-bit field f (bits 16 f and up).
__device__ __forceinline__ uint64_t drop_hash(uint64_t kb, uint64_t hi, int m) {
  return splitmix64(kb ^ (hi | static_cast<uint32_t>(m)));
}

// Keep bits of the four keys of one hash (bit f for key 4m + f).
__device__ __forceinline__ uint32_t drop_keep4(uint64_t x, uint32_t T) {
  return static_cast<uint32_t>((x & 0xFFFFu) >= T) |
         (static_cast<uint32_t>(((x >> 16) & 0xFFFFu) >= T) << 1) |
         (static_cast<uint32_t>(((x >> 32) & 0xFFFFu) >= T) << 2) |
         (static_cast<uint32_t>((x >> 48) >= T) << 3);
}
__device__ __forceinline__ uint64_t drop_hi(int h, int i) {
  return (static_cast<uint64_t>(h) << 48) | (static_cast<uint64_t>(static_cast<uint32_t>(i)) << 24);
}

// Transpose of a 32 x 32 bit matrix held one row per lane (bit k of lane l's
// word = element (l, k)): returns lane k's column, bit l = element (l, k).
// Five exchange rounds swap ever smaller off-diagonal blocks (16 x 16, then
// 8 x 8, ... 1 x 1): at width j the lanes with bit j set trade their words'
// low j-bit groups for their partners' high ones.
__device__ __forceinline__ uint32_t bit_transpose32(uint32_t x) {
  const int lane = threadIdx.x & 31;
  uint32_t m = 0x0000FFFFu;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1, m ^= m << j) {
    const uint32_t y = __shfl_xor_sync(0xffffffffu, x, j);
    x = (lane & j) ? ((x & ~m) | ((y >> j) & m)) : ((x & m) | ((y & m) << j));
  }
  return x;
}

// Threshold and scale of query token `tok` (packed index).
__device__ __forceinline__ void drop_row(const Params& p, int64_t tok, uint32_t& T, float& scale) {
  if (p.drop_tab) {
    const uint2 e = __ldg(p.drop_tab + tok);
    T = e.x;
    scale = __uint_as_float(e.y);
  } else {
    T = p.drop_T;
    scale = p.drop_scale;
  }
}

// Constants of the logit map z2 = log2(e) * (c*tanh(sigma*x/c) - slope*dist)
// (or log2(e) * (sigma*x - slope*dist) without a cap), where x is the raw
// q.k accumulator.
struct LogitMap {
  float in_scale;   // sigma / c   (or sigma*log2e without a cap)
  float out_scale;  // c * log2e
  bool capped;
};

__device__ __forceinline__ LogitMap make_logit_map(const Params& p) {
  LogitMap m;
  m.capped = p.softcap > 0.f;
  m.in_scale = m.capped ? p.sigma / p.softcap : p.sigma * kLog2e;
  m.out_scale = m.capped ? p.softcap * kLog2e : 1.f;
  return m;
}

template <bool BF16>
struct Pack;

template <>
struct Pack<true> {
  __device__ __forceinline__ static uint32_t two(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  // The two packed values back as an fp32 pair (f2_make order).
  __device__ __forceinline__ static uint64_t unpack(uint32_t v) {
    return f2_make(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
  }
};

template <>
struct Pack<false> {
  __device__ __forceinline__ static uint32_t two(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ __forceinline__ static uint64_t unpack(uint32_t v) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
    return f2_make(f.x, f.y);
  }
};

// Pack 8 floats (v[0..7]) to one 16-byte unit of 16-bit values.
template <bool BF16>
__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(Pack<BF16>::two(v[0], v[1]), Pack<BF16>::two(v[2], v[3]),
                    Pack<BF16>::two(v[4], v[5]), Pack<BF16>::two(v[6], v[7]));
}

}  // namespace attn
