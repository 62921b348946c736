// common.cuh -- per-element arithmetic shared by the attention kernels:
// logits with softcap and ALiBi in the base-2 domain, 16-bit packing, and
// swizzled shared-memory row writes.
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

// Threshold and scale of a dropout rate: keep when the hash's top 24 bits
// are >= T (probability 1 - T / 2^24), and scale kept values by 1/(1 - rate).
__host__ __device__ __forceinline__ void drop_params(float rate, uint32_t& T, float& scale) {
  if (!(rate < 1.f)) {
    T = 1u << 24;
    scale = 0.f;
  } else if (!(rate > 0.f)) {
    T = 0u;
    scale = 1.f;
  } else {
    T = static_cast<uint32_t>(rate * 16777216.0f);
    scale = 1.f / (1.f - rate);
  }
}

// Dropout of one element: `kb` = splitmix64(seed ^ b), `hi` = h << 48 | i << 24.
__device__ __forceinline__ bool drop_keep(uint64_t kb, uint64_t hi, int j, uint32_t T) {
  return static_cast<uint32_t>(splitmix64(kb ^ (hi | static_cast<uint32_t>(j))) >> 40) >= T;
}
__device__ __forceinline__ uint64_t drop_hi(int h, int i) {
  return (static_cast<uint64_t>(h) << 48) | (static_cast<uint64_t>(static_cast<uint32_t>(i)) << 24);
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

// tanh(x) = sign(x) * (1 - 2 / (exp(2|x|) + 1)).  Only the absolute error
// matters here (the logit is c * tanh), and it stays near 2e-7 on the whole
// line: the exponential's relative error scales a term that is at most 1.
// |x| is clamped at 15, where tanh already rounds to 1 in fp32.
__device__ __forceinline__ float tanh_acc(float x) {
  float ax = fminf(fabsf(x), 15.f);
  float e = ex2_approx(2.f * kLog2e * ax);
  return copysignf(1.f - __fdividef(2.f, e + 1.f), x);
}

// Base-2 logit and, through *th, the tanh value (for the chain rule).
__device__ __forceinline__ float logit2(const LogitMap& m, float acc, float slope2, float dist,
                                        float* th) {
  float z;
  if (m.capped) {
    float t = tanh_acc(acc * m.in_scale);
    *th = t;
    z = t * m.out_scale;
  } else {
    *th = 0.f;
    z = acc * m.in_scale;
  }
  return fmaf(-slope2, dist, z);
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

// Write 32 consecutive values v[0..31] of row r, starting at element col
// (a multiple of 32) of a K-major swizzled tile made of 64-wide chunks that
// are chunk_bytes apart.
template <bool BF16>
__device__ __forceinline__ void store_row32_sw128(uint8_t* tile, uint32_t chunk_bytes, int r,
                                                  int col, const float* v) {
  uint8_t* base = tile + (col >> 6) * chunk_bytes;
  const int u0 = (col & 63) >> 3;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint4 w = pack8<BF16>(v + 8 * u);
    *reinterpret_cast<uint4*>(base + sw128_offset(r, u0 + u)) = w;
  }
}

}  // namespace attn
