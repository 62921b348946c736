// bwd_dkdv.cu -- backward pass, dk and dv.
//
// dv_j = sum_h sum_i P_ij dO_i and dk_j = sigma * sum_h sum_i dS_ij q_i, the
// sums running over every query head that shares the single K/V head
// ("Noncausal Global Extreme-GQA Ragged Attention Full VJP", "Hard
// Constraints") and every query of the sequence.  P is recomputed from the
// stored lse ("ragged flash attention gradient recompute", "Root causes
// addressed").
//
// One CTA owns 128 keys of one sequence and keeps their dK and dV
// accumulators in TMEM (2 x 160 fp32 columns) while it walks every 64-row
// query step (64/G tokens x G heads) of the sequence in a fixed order, so the
// reduction order over heads and queries never changes: no atomics, bitwise
// repeatable.  Per query step, with keys in the MMA M dimension:
//   S^T  = K Q^T, dP^T = V dO^T      M=128 N=64 K=160
//   P^T, dS^T                        registers (thread = key), 16-bit to smem
//   dV  += P^T dO, dK += dS^T Q      M=128 N=160 K=64
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace kv {
constexpr uint32_t kTile = 16384;   // 64-feature chunk of a 128-key tile
constexpr uint32_t kTileQ = 8192;   // 64-feature chunk of a 64-row query step
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = 3 * kTile;
constexpr uint32_t kOffQ = 6 * kTile;
constexpr uint32_t kOffDO = kOffQ + 3 * kTileQ;
constexpr uint32_t kOffPt = kOffDO + 3 * kTileQ;  // 128 keys x 64 query rows
constexpr uint32_t kOffDSt = kOffPt + kTile;
constexpr uint32_t kOffCol = kOffDSt + kTile;     // per-column scalars
constexpr uint32_t kOffBar = kOffCol + 4 * 64 * 4;
constexpr uint32_t kSmem = kOffBar + 64 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDV = 0;
constexpr uint32_t kColDK = 160;
constexpr uint32_t kColS = 320;
constexpr uint32_t kColP = 384;
}  // namespace kv

__device__ __forceinline__ void drain_wait_kv(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq,
                const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv) {
  using namespace kv;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sDO = sm + kOffDO;
  uint8_t* sPt = sm + kOffPt;
  uint8_t* sDSt = sm + kOffDSt;
  float* cLse = reinterpret_cast<float*>(sm + kOffCol);  // lse * log2e, +inf if no P
  float* cD = cLse + 64;
  float* cSlope = cD + 64;                               // slope * log2e
  int* cPos = reinterpret_cast<int*>(cSlope + 64);        // local query position
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffBar);  // k+v, q+do, mma
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar + 4);
  int* s_item = reinterpret_cast<int*>(s_tmem + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int ntiles = ktile_count(p);
  if (tid == 0)
    *s_item = (*reinterpret_cast<volatile int32_t*>(p.status) != 0) ? ntiles
                                                                     : atomicAdd(p.counters + 1, 1);
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
  const uint32_t tDV = tmem + kColDV, tDK = tmem + kColDK, tS = tmem + kColS, tP = tmem + kColP;

  uint32_t ph_kv = 0, ph_q = 0, ph_m = 0;
  bool pend_kv = false, pend_q = false, pend_m = false;
  const LogitMap lm = make_logit_map(p);
  const bool masked = masking(p);
  constexpr uint32_t kIdS = idesc_f16(128, 64, BF16, false, false);
  constexpr uint32_t kIdG = idesc_f16(128, kHeadDim, BF16, false, true);
  const int G = p.G;
  const int step_tok = kRowsKV / G;
  const int ngroups = p.Hq / G;

  while (true) {
    KTile t;
    ktile_decode(p, item, t);
    const int j = t.key + tid;  // this thread's key (TMEM lane)
    const bool key_valid = j < t.Lk;
    const int nsteps = ((t.Lq + step_tok - 1) / step_tok) * ngroups;

    if (tid == 0) {
      mbar_arrive_expect_tx(&bar[0], 6 * kTile);
      for (int c = 0; c < 3; ++c) {
        tma_load_2d(sK + c * kTile, &tk, &bar[0], c * kChunk, t.k0 + t.key);
        tma_load_2d(sV + c * kTile, &tv, &bar[0], c * kChunk, t.k0 + t.key);
      }
      pend_kv = true;
    }

    for (int st = 0; st < nsteps; ++st) {
      const int tok0 = (st / ngroups) * step_tok;
      const int hg = st % ngroups;
      // per-column scalars of this query step (column c = token*G + head)
      if (tid < kRowsKV) {
        const int c = tid;
        const int i = tok0 + c / G;
        const int h = hg * G + c % G;
        float l2 = INFINITY, dv = 0.f;
        if (i < t.Lq) {
          const int64_t ri = static_cast<int64_t>(t.q0 + i) * p.Hq + h;
          const float lse = p.lse[ri];
          l2 = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
          dv = p.Dbuf[ri];
        }
        cLse[c] = l2;
        cD[c] = dv;
        cSlope[c] = p.slopes ? __ldg(p.slopes + t.b * p.slopes_bs + h) * kLog2e : 0.f;
        cPos[c] = i;
      }
      if (tid == 0) {
        mbar_arrive_expect_tx(&bar[1], 6 * kTileQ);
        for (int c = 0; c < 3; ++c) {
          tma_load_3d(sQ + c * kTileQ, &tq, &bar[1], c * kChunk, hg * G, t.q0 + tok0);
          tma_load_3d(sDO + c * kTileQ, &tdo, &bar[1], c * kChunk, hg * G, t.q0 + tok0);
        }
        pend_q = true;
        bool ok = true;
        if (pend_kv) {
          ok = mbar_wait(&bar[0], ph_kv, s_abort);
          if (ok) {
            ph_kv ^= 1;
            pend_kv = false;
          }
        }
        ok = ok && mbar_wait(&bar[1], ph_q, s_abort);
        if (ok) {
          ph_q ^= 1;
          pend_q = false;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t offa = (k >> 2) * kTile + (k & 3) * 32;
            const uint32_t offb = (k >> 2) * kTileQ + (k & 3) * 32;
            umma_ss(tS, sdesc_sw128(smem_addr(sK) + offa, 16, 1024),
                    sdesc_sw128(smem_addr(sQ) + offb, 16, 1024), kIdS, k > 0);
          }
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k) {
            const uint32_t offa = (k >> 2) * kTile + (k & 3) * 32;
            const uint32_t offb = (k >> 2) * kTileQ + (k & 3) * 32;
            umma_ss(tP, sdesc_sw128(smem_addr(sV) + offa, 16, 1024),
                    sdesc_sw128(smem_addr(sDO) + offb, 16, 1024), kIdS, k > 0);
          }
          umma_commit(&bar[2]);
          pend_m = true;
        }
      }
      __syncwarp();
      if (mbar_wait(&bar[2], ph_m, s_abort)) {
        ph_m ^= 1;
        pend_m = false;
      }
      __syncthreads();  // also publishes the column scalars
      if (*s_abort) break;
      tc_fence_after();

      // ---- P^T and dS^T for key j over the step's 64 query rows
#pragma unroll 1
      for (int cc = 0; cc < kRowsKV / 32; ++cc) {
        float sv[32], pv[32];
        tmem_ld32(tS + lane + cc * 32, sv);
        tmem_ld32(tP + lane + cc * 32, pv);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int c = cc * 32 + q;
          const int i = cPos[c];
          float th;
          float z = logit2(lm, sv[q], cSlope[c],
                           fabsf(static_cast<float>(i + t.Lk - t.Lq - j)), &th);
          bool adm = !masked || admissible(p, t.Lq, t.Lk, i, j);
          const float P = adm ? ex2_approx(z - cLse[c]) : 0.f;
          const float g = lm.capped ? fmaf(-th, th, 1.f) : 1.f;
          sv[q] = P;
          pv[q] = P * (pv[q] - cD[c]) * g;
        }
        store_row32_sw128<BF16>(sPt, kTile, tid, cc * 32, sv);
        store_row32_sw128<BF16>(sDSt, kTile, tid, cc * 32, pv);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();

      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kRowsKV / 16; ++k) {
          umma_ss(tDV, sdesc_sw128(smem_addr(sPt) + k * 32, 16, 1024),
                  sdesc_sw128(smem_addr(sDO) + k * 2048, kTileQ, 1024), kIdG, (st > 0 || k > 0));
        }
#pragma unroll
        for (int k = 0; k < kRowsKV / 16; ++k) {
          umma_ss(tDK, sdesc_sw128(smem_addr(sDSt) + k * 32, 16, 1024),
                  sdesc_sw128(smem_addr(sQ) + k * 2048, kTileQ, 1024), kIdG, (st > 0 || k > 0));
        }
        umma_commit(&bar[2]);
        pend_m = true;
      }
      __syncwarp();
      if (mbar_wait(&bar[2], ph_m, s_abort)) {
        ph_m ^= 1;
        pend_m = false;
      }
      __syncthreads();
      if (*s_abort) break;
    }
    if (*s_abort) break;
    if (tid == 0 && pend_kv) {
      if (mbar_wait(&bar[0], ph_kv, s_abort)) {
        ph_kv ^= 1;
        pend_kv = false;
      }
    }

    // ---- epilogue: dv = dV, dk = sigma * dK
    tc_fence_after();
    uint16_t* vrow = static_cast<uint16_t*>(p.dv) + static_cast<int64_t>(t.k0 + j) * p.dv_ts;
    uint16_t* krow = static_cast<uint16_t*>(p.dk) + static_cast<int64_t>(t.k0 + j) * p.dk_ts;
#pragma unroll
    for (int c = 0; c < kHeadDim / 32; ++c) {
      float a[32], b[32];
      tmem_ld32(tDV + lane + c * 32, a);
      tmem_ld32(tDK + lane + c * 32, b);
      tmem_wait_ld();
      if (key_valid) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float w[8], x[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            w[i] = nsteps > 0 ? a[8 * u + i] : 0.f;
            x[i] = nsteps > 0 ? b[8 * u + i] * p.sigma : 0.f;
          }
          *reinterpret_cast<uint4*>(vrow + c * 32 + u * 8) = pack8<BF16>(w);
          *reinterpret_cast<uint4*>(krow + c * 32 + u * 8) = pack8<BF16>(x);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) *s_item = atomicAdd(p.counters + 1, 1);
    __syncthreads();
    item = *s_item;
    if (item >= ntiles) break;
  }

  if (*s_abort) {
    if (tid == 0) {
      atomicOr(p.status, ATTN_DEV_TIMEOUT_DKDV);
      if (pend_kv) drain_wait_kv(&bar[0], ph_kv);
      if (pend_q) drain_wait_kv(&bar[1], ph_q);
      if (pend_m) drain_wait_kv(&bar[2], ph_m);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_dkdv(const Params& p, const CUtensorMap& tq64, const CUtensorMap& tdo64,
                        const CUtensorMap& tk, const CUtensorMap& tv, int grid, cudaStream_t s) {
  if (p.dtype == 1) {
    auto k = dkdv_kernel<true>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kSmem);
    k<<<grid, kThreads, kv::kSmem, s>>>(p, tq64, tdo64, tk, tv);
  } else {
    auto k = dkdv_kernel<false>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kSmem);
    k<<<grid, kThreads, kv::kSmem, s>>>(p, tq64, tdo64, tk, tv);
  }
  return cudaGetLastError();
}

}  // namespace attn
