// bwd_dq.cu -- backward pass, dq.
//
// dq_i = sigma * sum_j dS_ij k_j with dS_ij = P_ij (dP_ij - D_i)(1 - tanh^2),
// P_ij = exp(z_ij - lse_i) recomputed from the stored lse ("ragged flash
// attention gradient recompute", "Root causes addressed": no P is stored; the
// backward recomputes each tile from L).  dq has its own pass over the key
// tiles so that every dq row is written once, by one CTA, with no atomics:
// repeated calls are bitwise identical.
//
// Tile: the forward's 128 query rows.  Per key tile:
//   S  = Q K^T, dP = dO V^T     two M=128 N=128 K=160 MMAs into TMEM
//   dS                          registers, one thread per row, 16-bit to smem
//   dQ += dS K                  M=128 N=160 K=128 into TMEM
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace dqk {
constexpr uint32_t kTile = 16384;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffDO = 3 * kTile;
constexpr uint32_t kOffK = 6 * kTile;
constexpr uint32_t kOffV = 9 * kTile;
constexpr uint32_t kOffDS = 12 * kTile;  // 2 chunks
constexpr uint32_t kOffBar = 14 * kTile;
constexpr uint32_t kSmem = kOffBar + 64 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColP = 128;
constexpr uint32_t kColQ = 256;
}  // namespace dqk

__device__ __forceinline__ void drain_wait_dq(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    dq_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq,
              const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv) {
  using namespace dqk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sDO = sm + kOffDO;
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
  uint8_t* sDS = sm + kOffDS;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffBar);  // q+do, k, v, mma
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar + 4);
  int* s_item = reinterpret_cast<int*>(s_tmem + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int ntiles = qtile_count(p);
  if (tid == 0)
    *s_item = (*reinterpret_cast<volatile int32_t*>(p.status) != 0) ? ntiles
                                                                     : atomicAdd(p.counters + 2, 1);
  __syncthreads();
  int item = *s_item;
  if (item >= ntiles) return;

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
    fence_barrier_init();
    *s_abort = 0;
    prefetch_tensormap(&tq);
    prefetch_tensormap(&tdo);
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
  const uint32_t tS = tmem + kColS, tP = tmem + kColP, tQ = tmem + kColQ;

  uint32_t ph_q = 0, ph_k = 0, ph_v = 0, ph_m = 0;
  bool pend_q = false, pend_k = false, pend_v = false, pend_m = false;
  const LogitMap lm = make_logit_map(p);
  const bool masked = masking(p);
  constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
  constexpr uint32_t kIdQ = idesc_f16(128, kHeadDim, BF16, false, true);
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
    const int pos_off = i_loc + t.Lk - t.Lq;
    float lse2 = INFINITY, Drow = 0.f;  // rows outside the sequence get P = 0
    if (row_valid) {
      const int64_t ri = static_cast<int64_t>(t.q0 + i_loc) * p.Hq + h;
      const float lse = p.lse[ri];
      lse2 = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
      Drow = p.Dbuf[ri];
    }

    if (tid == 0) {
      mbar_arrive_expect_tx(&bar[0], 6 * kTile);
      for (int c = 0; c < 3; ++c) {
        tma_load_3d(sQ + c * kTile, &tq, &bar[0], c * kChunk, t.hg * G, t.q0 + t.tok);
        tma_load_3d(sDO + c * kTile, &tdo, &bar[0], c * kChunk, t.hg * G, t.q0 + t.tok);
      }
      pend_q = true;
    }

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
        }
        ok = ok && mbar_wait(&bar[2], ph_v, s_abort);
        if (ok) {
          ph_v ^= 1;
          pend_v = false;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t off = (k >> 2) * kTile + (k & 3) * 32;
            umma_ss(tS, sdesc_sw128(smem_addr(sQ) + off, 16, 1024),
                    sdesc_sw128(smem_addr(sK) + off, 16, 1024), kIdS, k > 0);
          }
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t off = (k >> 2) * kTile + (k & 3) * 32;
            umma_ss(tP, sdesc_sw128(smem_addr(sDO) + off, 16, 1024),
                    sdesc_sw128(smem_addr(sV) + off, 16, 1024), kIdS, k > 0);
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

      // ---- dS for row r, 32 keys at a time
#pragma unroll 1
      for (int c = 0; c < kKeys / 32; ++c) {
        float sv[32], pv[32];
        tmem_ld32(tS + lane + c * 32, sv);
        tmem_ld32(tP + lane + c * 32, pv);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int jg = key0 + c * 32 + j;
          float th;
          float z = logit2(lm, sv[j], slope2, fabsf(static_cast<float>(pos_off - jg)), &th);
          bool adm = jg < t.Lk;
          if (masked) adm = adm && admissible(p, t.Lq, t.Lk, i_loc, jg);
          const float P = adm ? ex2_approx(z - lse2) : 0.f;
          const float g = lm.capped ? fmaf(-th, th, 1.f) : 1.f;
          sv[j] = P * (pv[j] - Drow) * g;
        }
        store_row32_sw128<BF16>(sDS, kTile, r, c * 32, sv);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();

      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kKeys / 16; ++k) {
          umma_ss(tQ, sdesc_sw128(smem_addr(sDS) + (k >> 2) * kTile + (k & 3) * 32, 16, 1024),
                  sdesc_sw128(smem_addr(sK) + k * 2048, kTile, 1024), kIdQ, (kt > 0 || k > 0));
        }
        umma_commit(&bar[3]);
        pend_m = true;
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
    if (tid == 0 && pend_q) {
      if (mbar_wait(&bar[0], ph_q, s_abort)) {
        ph_q ^= 1;
        pend_q = false;
      }
    }

    // ---- epilogue: dq = sigma * dQ
    tc_fence_after();
    uint16_t* qrow = static_cast<uint16_t*>(p.dq) + static_cast<int64_t>(t.q0 + i_loc) * p.dq_ts +
                     static_cast<int64_t>(h) * p.dq_hs;
#pragma unroll
    for (int c = 0; c < kHeadDim / 32; ++c) {
      float o[32];
      tmem_ld32(tQ + lane + c * 32, o);
      tmem_wait_ld();
      if (row_valid) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = nkt > 0 ? o[8 * u + i] * p.sigma : 0.f;
          *reinterpret_cast<uint4*>(qrow + c * 32 + u * 8) = pack8<BF16>(w);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) *s_item = atomicAdd(p.counters + 2, 1);
    __syncthreads();
    item = *s_item;
    if (item >= ntiles) break;
  }

  if (*s_abort) {
    if (tid == 0) {
      atomicOr(p.status, ATTN_DEV_TIMEOUT_DQ);
      if (pend_q) drain_wait_dq(&bar[0], ph_q);
      if (pend_k) drain_wait_dq(&bar[1], ph_k);
      if (pend_v) drain_wait_dq(&bar[2], ph_v);
      if (pend_m) drain_wait_dq(&bar[3], ph_m);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_dq(const Params& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                      const CUtensorMap& tk, const CUtensorMap& tv, int grid, cudaStream_t s) {
  if (p.dtype == 1) {
    auto k = dq_kernel<true>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dqk::kSmem);
    k<<<grid, kThreads, dqk::kSmem, s>>>(p, tq, tdo, tk, tv);
  } else {
    auto k = dq_kernel<false>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dqk::kSmem);
    k<<<grid, kThreads, dqk::kSmem, s>>>(p, tq, tdo, tk, tv);
  }
  return cudaGetLastError();
}

}  // namespace attn
