// fwd.cu -- forward pass: out and lse for every query row.
//
// "Noncausal Global Extreme-GQA Ragged Attention Full VJP" ("What You Have"):
// scaled logits, 3*tanh(s/3) softcap, ALiBi -slope*|i + Lk - Lq - j|, softmax,
// out = P V.  The softmax is the online (running max / running sum) form of
// "ragged flash attention gradient recompute" ("Root causes addressed"):
// only O and L = m + log l are stored.
//
// Tile: 128 query rows = (128/G tokens) x (G heads of one head group); all
// heads share the single K/V head, so every row of a tile reads the same
// 128-key K and V tiles.  Per key tile j:
//   S_j = Q K_j^T         tcgen05.mma (Q, K from shared memory), fp32 in TMEM
//   P_j = exp2(z - m)     softmax warps, one thread per row (TMEM lane); P_j
//                         is written back over S_j as 16-bit pairs
//   O  += P_j V_j         tcgen05.mma with P_j read from TMEM
//
// Warp roles (192 threads): warp 0 issues TMA loads (Q once per tile, K and
// V through a 3-slot ring), warp 1 issues the MMAs, warps 2-5 run the
// softmax and the epilogue.  S is double-buffered in TMEM so the tensor core
// computes S_{j+1} while the softmax works on S_j.
//
// Key tiles are visited starting with the one that holds the ALiBi peak of
// the tile's rows (the key aligned with the query, where the distance is 0),
// so the running max is (nearly) final after the first tile.  O is rescaled
// only when a row's max grows by more than 8 (base-2 units); until then P is
// taken relative to the stale max and stays below 2^8.  With the softcap
// (|t| <= c) and ALiBi (<= 0) no later tile can exceed the first tile's max
// by more than 2*c*log2(e) = 8.66, so rescales are rare.
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace fwd {
constexpr int kThreadsF = 192;
constexpr int kSlots = 3;
constexpr uint32_t kTile = 16384;        // one 64-feature chunk of a 128-row tile
constexpr uint32_t kTile3 = 3 * kTile;   // a whole 128 x 160 tile
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffSlot = kTile3;    // kSlots tiles of K or V
constexpr uint32_t kOffBar = kOffSlot + kSlots * kTile3;
constexpr uint32_t kSmem = kOffBar + 256 + 1024;  // + barriers + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;          // S0: [0,128), S1: [128,256), O: [256,416)
constexpr float kRescale = 8.f;          // lazy-rescale threshold (base 2)

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t slot_full[kSlots], slot_empty[kSlots];
  uint64_t s_full[2], s_free[2], p_full[2];
  uint64_t o_full, o_empty, drain;
};
}  // namespace fwd

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

// First key tile to visit and the tile count for a query tile.
__device__ __forceinline__ void key_order(const QTile& t, int& n, int& t0) {
  n = (t.Lk + kKeys - 1) / kKeys;
  int k0 = t.tok + t.Lk - t.Lq;  // key aligned with the tile's first query
  k0 = k0 < 0 ? 0 : (k0 >= t.Lk ? t.Lk - 1 : k0);
  t0 = n > 0 ? k0 / kKeys : 0;
}

template <bool BF16>
__global__ void __launch_bounds__(fwd::kThreadsF, 1)
    fwd_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq,
               const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using namespace fwd;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sSlot = sm + kOffSlot;
  Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_status = reinterpret_cast<int*>(s_tmem + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int ntiles = qtile_count(p);
  if (tid == 0) *s_status = *reinterpret_cast<volatile int32_t*>(p.status);
  __syncthreads();
  if (*s_status != 0 || static_cast<int>(blockIdx.x) >= ntiles) return;  // uniform

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars->slot_full[s], 1);
      mbar_init(&bars->slot_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], 1);
      mbar_init(&bars->p_full[b], 4);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 4);
    mbar_init(&bars->drain, 1);
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int G = p.G;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tq);
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tv);
      uint32_t fill = 0;
      int tcount = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < ntiles && ok; item += gridDim.x, ++tcount) {
        QTile t;
        qtile_decode(p, item, t);
        int n, t0;
        key_order(t, n, t0);
        if (tcount > 0 && !(ok = mbar_wait(&bars->q_empty, (tcount - 1) & 1, s_abort))) break;
        mbar_arrive_expect_tx(&bars->q_full, kTile3);
        for (int c = 0; c < 3; ++c)
          tma_load_3d(sQ + c * kTile, &tq, &bars->q_full, c * kChunk, t.hg * G, t.q0 + t.tok);
        for (int jj = 0; jj < n && ok; ++jj) {
          const int kt = (t0 + jj) % n;
          for (int kv = 0; kv < 2; ++kv, ++fill) {
            const int s = fill % kSlots;
            if (fill >= kSlots &&
                !(ok = mbar_wait(&bars->slot_empty[s], (fill / kSlots - 1) & 1, s_abort)))
              break;
            mbar_arrive_expect_tx(&bars->slot_full[s], kTile3);
            uint8_t* dst = sSlot + s * kTile3;
            for (int c = 0; c < 3; ++c)
              tma_load_2d(dst + c * kTile, kv ? &tv : &tk, &bars->slot_full[s], c * kChunk,
                          t.k0 + kt * kKeys);
          }
        }
      }
      if (*s_abort) {
        // let every load this thread started land before the CTA exits
        if (tcount > 0) drain_wait(&bars->q_full, (tcount - 1) & 1);
        for (uint32_t f = fill > kSlots ? fill - kSlots : 0; f < fill; ++f)
          drain_wait(&bars->slot_full[f % kSlots], (f / kSlots) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t kIdO = idesc_f16(128, kHeadDim, BF16, false, true);
      uint32_t g = 0;  // global key-step counter of this CTA
      int tcount = 0;
      bool ok = true;
      auto issue_s = [&](uint32_t gs) -> bool {
        const uint32_t f = 2 * gs;  // K fill index of step gs
        if (!mbar_wait(&bars->slot_full[f % kSlots], (f / kSlots) & 1, s_abort)) return false;
        if (gs >= 2 && !mbar_wait(&bars->s_free[gs & 1], ((gs - 2) >> 1) & 1, s_abort))
          return false;
        tc_fence_after();
        const uint32_t kb = smem_addr(sSlot + (f % kSlots) * kTile3);
        const uint32_t qb = smem_addr(sQ);
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k) {
          const uint32_t off = (k >> 2) * kTile + (k & 3) * 32;
          umma_ss(tmem + (gs & 1) * 128, sdesc_sw128(qb + off, 16, 1024),
                  sdesc_sw128(kb + off, 16, 1024), kIdS, k > 0);
        }
        umma_commit(&bars->s_full[gs & 1]);
        umma_commit(&bars->slot_empty[f % kSlots]);
        return true;
      };
      for (int item = blockIdx.x; item < ntiles && ok; item += gridDim.x, ++tcount) {
        QTile t;
        qtile_decode(p, item, t);
        int n, t0;
        key_order(t, n, t0);
        if (!(ok = mbar_wait(&bars->q_full, tcount & 1, s_abort))) break;
        if (n == 0) {  // no keys: nothing to multiply; keep every phase count
          mbar_arrive(&bars->q_empty);
          if (tcount > 0 && !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort))) break;
          mbar_arrive(&bars->o_full);
          continue;
        }
        if (!(ok = issue_s(g))) break;
        if (n == 1) umma_commit(&bars->q_empty);
        for (int jj = 0; jj < n; ++jj) {
          const uint32_t gg = g + jj;
          if (jj + 1 < n) {
            if (!(ok = issue_s(gg + 1))) break;
            if (jj + 1 == n - 1) umma_commit(&bars->q_empty);
          }
          if (!(ok = mbar_wait(&bars->p_full[gg & 1], (gg >> 1) & 1, s_abort))) break;
          if (jj == 0 && tcount > 0 &&
              !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort)))
            break;
          const uint32_t f = 2 * gg + 1;  // V fill index
          if (!(ok = mbar_wait(&bars->slot_full[f % kSlots], (f / kSlots) & 1, s_abort))) break;
          tc_fence_after();
          const uint32_t vb = smem_addr(sSlot + (f % kSlots) * kTile3);
          const uint32_t pa = tmem + (gg & 1) * 128;
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k)
            umma_ts(tmem + kColO, pa + k * 8, sdesc_sw128(vb + k * 2048, kTile, 1024), kIdO,
                    (jj > 0 || k > 0));
          umma_commit(&bars->s_free[gg & 1]);
          umma_commit(&bars->slot_empty[f % kSlots]);
          if (jj == n - 1) umma_commit(&bars->o_full);
        }
        g += n;
      }
      // every MMA this thread issued completes before the CTA moves on
      umma_commit(&bars->drain);
      drain_wait(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const LogitMap lm = make_logit_map(p);
    const bool masked = masking(p);
    uint32_t g = 0;
    int tcount = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < ntiles && ok; item += gridDim.x, ++tcount) {
      QTile t;
      qtile_decode(p, item, t);
      int n, t0;
      key_order(t, n, t0);
      const int i_loc = t.tok + r / G;
      const int h = t.hg * G + r % G;
      const bool row_valid = i_loc < t.Lq;
      const float slope2 = p.slopes ? __ldg(p.slopes + t.b * p.slopes_bs + h) * kLog2e : 0.f;
      const int pos_off = i_loc + t.Lk - t.Lq;  // dist(j) = |pos_off - j|
      float m_run = -INFINITY, l = 0.f;
      for (int jj = 0; jj < n; ++jj) {
        const uint32_t gg = g + jj;
        const int key0 = ((t0 + jj) % n) * kKeys;
        const uint32_t sb = tmem + (gg & 1) * 128 + lane_addr;
        if (!(ok = mbar_wait_warp(&bars->s_full[gg & 1], (gg >> 1) & 1, s_abort))) break;
        tc_fence_after();
        float x[kKeys];
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c)
          tmem_ld32(sb + c * 32, *reinterpret_cast<float(*)[32]>(x + c * 32));
        tmem_wait_ld();
        const float pos0 = static_cast<float>(pos_off - key0);
        const bool edge = masked || key0 + kKeys > t.Lk;
        float mx = -INFINITY;
        if (lm.capped) {
#pragma unroll
          for (int j = 0; j < kKeys; ++j) {
            const float th = tanh_approx(x[j] * lm.in_scale);
            x[j] = fmaf(th, lm.out_scale, -slope2 * fabsf(pos0 - static_cast<float>(j)));
          }
        } else {
#pragma unroll
          for (int j = 0; j < kKeys; ++j)
            x[j] = fmaf(x[j], lm.in_scale, -slope2 * fabsf(pos0 - static_cast<float>(j)));
        }
        if (edge) {
#pragma unroll
          for (int j = 0; j < kKeys; ++j) {
            const int jg = key0 + j;
            bool adm = jg < t.Lk;
            if (masked) adm = adm && admissible(p, t.Lq, t.Lk, i_loc, jg);
            x[j] = adm ? x[j] : -INFINITY;
          }
        }
#pragma unroll
        for (int j = 0; j < kKeys; ++j) mx = fmaxf(mx, x[j]);
        const float m_new = fmaxf(m_run, mx);
        const bool need = m_new > m_run + kRescale;
        const float alpha = need ? ex2_approx(m_run - m_new) : 1.f;
        if (jj > 0 && __any_sync(0xffffffffu, need)) {
          // O must absorb the new max: wait for the previous P V, then scale
          const uint32_t gp = gg - 1;
          if (!(ok = mbar_wait_warp(&bars->s_free[gp & 1], (gp >> 1) & 1, s_abort))) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kHeadDim / 32; ++c) {
            float o[32];
            tmem_ld32(tmem + kColO + lane_addr + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tmem + kColO + lane_addr + c * 32, o);
          }
          tmem_wait_st();
        }
        if (need) {
          l *= alpha;
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        uint32_t pk[kKeys / 2];
#pragma unroll
        for (int j = 0; j < kKeys; j += 2) {
          const float p0 = ex2_approx(x[j] - m_use);
          const float p1 = ex2_approx(x[j + 1] - m_use);
          l += p0 + p1;
          pk[j >> 1] = Pack<BF16>::two(p0, p1);
        }
#pragma unroll
        for (int c = 0; c < kKeys / 32; ++c)
          tmem_st16(sb + c * 16, *reinterpret_cast<uint32_t(*)[16]>(pk + c * 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[gg & 1]);
      }
      if (!ok) break;
      g += n;
      // ---- epilogue: out = O / l, lse = (m + log2 l) ln 2
      if (!(ok = mbar_wait_warp(&bars->o_full, tcount & 1, s_abort))) break;
      tc_fence_after();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      if (row_valid)
        p.lse[static_cast<int64_t>(t.q0 + i_loc) * p.Hq + h] =
            (l > 0.f) ? (m_run + log2f(l)) * kLn2 : -INFINITY;
      uint16_t* orow = static_cast<uint16_t*>(p.out) +
                       static_cast<int64_t>(t.q0 + i_loc) * p.out_ts +
                       static_cast<int64_t>(h) * p.out_hs;
#pragma unroll 1
      for (int c = 0; c < kHeadDim / 32; ++c) {
        float o[32];
        tmem_ld32(tmem + kColO + lane_addr + c * 32, o);
        tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = n > 0 ? o[8 * u + i] * inv : 0.f;
            *reinterpret_cast<uint4*>(orow + c * 32 + u * 8) = pack8<BF16>(w);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty);
    }
  }

  __syncthreads();
  if (tid == 0 && *s_abort) atomicOr(p.status, ATTN_DEV_TIMEOUT_FWD);
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_fwd(const Params& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, int grid, cudaStream_t s) {
  if (p.dtype == 1) {
    auto k = fwd_kernel<true>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::kSmem);
    k<<<grid, fwd::kThreadsF, fwd::kSmem, s>>>(p, tq, tk, tv);
  } else {
    auto k = fwd_kernel<false>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::kSmem);
    k<<<grid, fwd::kThreadsF, fwd::kSmem, s>>>(p, tq, tk, tv);
  }
  return cudaGetLastError();
}

}  // namespace attn
