// fwd.cu -- forward pass: out and lse for every query row.
//
// "Noncausal Global Extreme-GQA Ragged Attention Full VJP" ("What You Have"):
// scaled logits, 3*tanh(s/3) softcap, ALiBi -slope*|i + Lk - Lq - j|, softmax,
// out = P V.  The softmax is the online (running max / running sum) form of
// "ragged flash attention gradient recompute" ("Root causes addressed"):
// only O and L = m + log l are stored.
//
// Tile: 128 query rows = (128/G tokens) x (G heads of one head group); every
// head shares the single K/V head, so the rows of one tile all read the same
// 128-key K and V tiles.  Per key tile:
//   S  = Q K^T            tcgen05.mma, M=128 N=128 K=160, fp32 in TMEM
//   P  = exp2(z - m)      registers, one thread per row (TMEM lane)
//   O  = alpha*O + P V    O rescaled in TMEM, then M=128 N=160 K=128
// Q, K, V are staged by TMA (128-byte swizzle, three 64-feature chunks; the
// tensor map's feature extent is 160 so chunk 2's upper half reads as zero).
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace fwd {
constexpr uint32_t kTile = 16384;  // one 64-feature chunk of a 128-row tile
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 3 * kTile;
constexpr uint32_t kOffV = 6 * kTile;
constexpr uint32_t kOffP = 9 * kTile;   // P: 2 chunks (128 keys)
constexpr uint32_t kOffBar = 11 * kTile;
constexpr uint32_t kSmem = kOffBar + 64 + 1024;  // + barriers + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;
}  // namespace fwd

// Wait with a time limit only (used to drain copies after an abort).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq,
               const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
  uint8_t* sP = sm + kOffP;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffBar);  // q, k, v, mma
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar + 4);
  int* s_item = reinterpret_cast<int*>(s_tmem + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int ntiles = qtile_count(p);

  // The status is read once, by one thread, so the whole CTA decides alike.
  if (tid == 0)
    *s_item = (*reinterpret_cast<volatile int32_t*>(p.status) != 0) ? ntiles
                                                                     : atomicAdd(p.counters + 0, 1);
  __syncthreads();
  int item = *s_item;
  if (item >= ntiles) return;  // uniform: nothing allocated yet

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
    fence_barrier_init();
    *s_abort = 0;
    prefetch_tensormap(&tq);
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tS = tmem + kColS;
  const uint32_t tO = tmem + kColO;

  uint32_t ph_q = 0, ph_k = 0, ph_v = 0, ph_m = 0;
  bool pend_q = false, pend_k = false, pend_v = false;  // TMA loads not yet observed
  bool pend_m = false;                                  // an MMA commit not yet observed
  const LogitMap lm = make_logit_map(p);
  const bool masked = masking(p);
  constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
  constexpr uint32_t kIdO = idesc_f16(128, kHeadDim, BF16, false, true);
  const int G = p.G;

  while (true) {
    QTile t;
    qtile_decode(p, item, t);
    const int r = tid;
    const int i_loc = t.tok + r / G;
    const int h = t.hg * G + r % G;
    const bool row_valid = i_loc < t.Lq;
    const float slope2 = p.slopes ? __ldg(p.slopes + t.b * p.slopes_bs + h) * kLog2e : 0.f;
    const int nkt = (t.Lk + kKeys - 1) / kKeys;
    const int pos_off = i_loc + t.Lk - t.Lq;  // dist = |pos_off - j|

    if (tid == 0) {
      mbar_arrive_expect_tx(&bar[0], 3 * kTile);
      for (int c = 0; c < 3; ++c)
        tma_load_3d(sQ + c * kTile, &tq, &bar[0], c * kChunk, t.hg * G, t.q0 + t.tok);
      pend_q = true;
    }

    float m2 = -INFINITY, l = 0.f;
    for (int kt = 0; kt < nkt; ++kt) {
      const int key0 = kt * kKeys;
      if (tid == 0) {
        mbar_arrive_expect_tx(&bar[1], 3 * kTile);
        for (int c = 0; c < 3; ++c)
          tma_load_2d(sK + c * kTile, &tk, &bar[1], c * kChunk, t.k0 + key0);
        mbar_arrive_expect_tx(&bar[2], 3 * kTile);
        for (int c = 0; c < 3; ++c)
          tma_load_2d(sV + c * kTile, &tv, &bar[2], c * kChunk, t.k0 + key0);
        pend_k = pend_v = true;
        bool ok = true;
        if (pend_q) {
          ok = mbar_wait(&bar[0], ph_q, s_abort);
          if (ok) {
            ph_q ^= 1;
            pend_q = false;
          }
        }
        ok = ok && mbar_wait(&bar[1], ph_k, s_abort);
        if (ok) {
          ph_k ^= 1;
          pend_k = false;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t off = (k >> 2) * kTile + (k & 3) * 32;
            umma_ss(tS, sdesc_sw128(smem_addr(sQ) + off, 16, 1024),
                    sdesc_sw128(smem_addr(sK) + off, 16, 1024), kIdS, k > 0);
          }
          umma_commit(&bar[3]);
          pend_m = true;
        }
      }
      __syncwarp();
      if (mbar_wait(&bar[3], ph_m, s_abort)) {
        ph_m ^= 1;
        pend_m = false;
      }
      __syncthreads();
      if (*s_abort) break;
      tc_fence_after();

      // ---- softmax on row r: 128 logits
      float s[kKeys];
#pragma unroll
      for (int c = 0; c < kKeys / 32; ++c)
        tmem_ld32(tS + lane + c * 32, *reinterpret_cast<float(*)[32]>(s + c * 32));
      tmem_wait_ld();
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kKeys; ++j) {
        const int jg = key0 + j;
        float th;
        float z = logit2(lm, s[j], slope2, fabsf(static_cast<float>(pos_off - jg)), &th);
        bool adm = jg < t.Lk;
        if (masked) adm = adm && admissible(p, t.Lq, t.Lk, i_loc, jg);
        s[j] = adm ? z : -INFINITY;
        mx = fmaxf(mx, s[j]);
      }
      const float m_new = fmaxf(m2, mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m2 - m_use);
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < kKeys; ++j) {
        s[j] = ex2_approx(s[j] - m_use);
        rs += s[j];
      }
      l = l * alpha + rs;
      m2 = m_new;
      if (kt > 0) {
        // O *= alpha (the previous P V is complete: its commit was awaited)
#pragma unroll
        for (int c = 0; c < kHeadDim / 32; ++c) {
          float o[32];
          tmem_ld32(tO + lane + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tO + lane + c * 32, o);
        }
        tmem_wait_st();
      }
#pragma unroll
      for (int c = 0; c < kKeys / 32; ++c) store_row32_sw128<BF16>(sP, kTile, r, c * 32, s + c * 32);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();

      if (tid == 0) {
        bool ok = mbar_wait(&bar[2], ph_v, s_abort);
        if (ok) {
          ph_v ^= 1;
          pend_v = false;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k) {
            umma_ss(tO, sdesc_sw128(smem_addr(sP) + (k >> 2) * kTile + (k & 3) * 32, 16, 1024),
                    sdesc_sw128(smem_addr(sV) + k * 2048, kTile, 1024), kIdO, (kt > 0 || k > 0));
          }
          umma_commit(&bar[3]);
          pend_m = true;
        }
      }
      __syncwarp();
      if (mbar_wait(&bar[3], ph_m, s_abort)) {
        ph_m ^= 1;
        pend_m = false;
      }
      __syncthreads();
      if (*s_abort) break;
    }
    if (*s_abort) break;
    if (tid == 0 && pend_q) {  // no key tile: the Q load was never awaited
      if (mbar_wait(&bar[0], ph_q, s_abort)) {
        ph_q ^= 1;
        pend_q = false;
      }
    }

    // ---- epilogue: out = O / l, lse = (m + log2 l) ln 2
    tc_fence_after();
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
    if (row_valid) {
      const float lse = (l > 0.f) ? (m2 + log2f(l)) * kLn2 : -INFINITY;
      p.lse[static_cast<int64_t>(t.q0 + i_loc) * p.Hq + h] = lse;
    }
    using T = uint16_t;
    T* orow = static_cast<T*>(p.out) + static_cast<int64_t>(t.q0 + i_loc) * p.out_ts +
              static_cast<int64_t>(h) * p.out_hs;
#pragma unroll
    for (int c = 0; c < kHeadDim / 32; ++c) {
      float o[32];
      tmem_ld32(tO + lane + c * 32, o);
      tmem_wait_ld();
      if (row_valid) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = nkt > 0 ? o[8 * u + i] * inv : 0.f;
          *reinterpret_cast<uint4*>(orow + c * 32 + u * 8) = pack8<BF16>(w);
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // TMEM O and the s_item slot are free again
    if (tid == 0) *s_item = atomicAdd(p.counters + 0, 1);
    __syncthreads();
    item = *s_item;
    if (item >= ntiles) break;
  }

  if (*s_abort) {
    if (tid == 0) {
      atomicOr(p.status, ATTN_DEV_TIMEOUT_FWD);
      if (pend_q) drain_wait(&bar[0], ph_q);
      if (pend_k) drain_wait(&bar[1], ph_k);
      if (pend_v) drain_wait(&bar[2], ph_v);
      if (pend_m) drain_wait(&bar[3], ph_m);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_fwd(const Params& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, int grid, cudaStream_t s) {
  if (p.dtype == 1) {
    auto k = fwd_kernel<true>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::kSmem);
    k<<<grid, kThreads, fwd::kSmem, s>>>(p, tq, tk, tv);
  } else {
    auto k = fwd_kernel<false>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::kSmem);
    k<<<grid, kThreads, fwd::kSmem, s>>>(p, tq, tk, tv);
  }
  return cudaGetLastError();
}

}  // namespace attn
