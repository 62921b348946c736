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
// repeatable.  Per query step, keys in the MMA M dimension:
//   S^T  = K Q^T, dP^T = V dO^T      M=128 N=64 K=160, shared-memory operands
//   P^T, dS^T                        elementwise warps (thread = key), written
//                                    back into TMEM as 16-bit pairs
//   dV  += P^T dO, dK += dS^T Q      M=128 N=160 K=64, A operand from TMEM
//
// Warp roles (320 threads): warp 0 loads (K, V once per key tile; Q and dO
// through a 3-stage ring), warp 1 issues the MMAs, warps 2-9 compute P^T and
// dS^T and write dk/dv -- two warps per TMEM lane quadrant, each taking half
// of the step's 64 query columns, so every SM sub-partition has two warps to
// hide MUFU and load latency.  They also fetch the next step's per-column
// scalars (lse, D, slope, aligned key position) while the current step runs.  S^T is
// double-buffered so S^T of the next step runs while this step's elementwise
// work is in flight.  K and V keep their last 32 features in a 64-byte-
// swizzled chunk (they are only K-major A operands here), which leaves room
// for the third Q/dO stage.
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace kv {
constexpr int kThreadsKV = 320;
constexpr int kStages = 3;
constexpr uint32_t kTile = 16384;   // 64-feature chunk of a 128-key tile
constexpr uint32_t kTail = 8192;    // features 128..159 of a 128-key tile (64 B rows)
constexpr uint32_t kKV = 2 * kTile + kTail;
constexpr uint32_t kTileQ = 8192;   // 64-feature chunk of a 64-row query step
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kKV;
constexpr uint32_t kOffStage = 2 * kKV;             // stages of (Q, dO)
constexpr uint32_t kStage = 6 * kTileQ;             // Q 3 chunks + dO 3 chunks
constexpr uint32_t kOffCol = kOffStage + kStages * kStage;  // 2 buffers of scalars
constexpr uint32_t kColBytes = 4 * 64 * 4;
constexpr uint32_t kOffBar = kOffCol + 2 * kColBytes;
constexpr uint32_t kSmem = kOffBar + 256;  // the dynamic base is checked to be 1024-aligned
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDV = 0;
constexpr uint32_t kColDK = 160;
constexpr uint32_t kColS = 320;    // two 64-column S^T buffers: [320,384), [384,448)
constexpr uint32_t kColP = 448;    // dP^T: [448, 512)

struct Cols {  // per-column scalars of one query step
  float lse2[64];   // lse * log2(e); +inf where no P exists (row outside / empty)
  float D[64];
  float slope2[64];  // slope * log2(e)
  float pos[64];     // i + Lk - Lq (the key aligned with query row i)
};

struct Bars {
  uint64_t kv_full, kv_empty;
  uint64_t st_full[kStages], st_empty[kStages];
  uint64_t s_full[2], s_free[2];
  uint64_t dp_full, dp_free, p_full;
  uint64_t acc_full, acc_empty, drain;
  uint64_t cols_x[2];  // per-step scalars published (one arrival per elementwise warp)
};
}  // namespace kv

__device__ __forceinline__ void drain_wait_kv(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

template <bool BF16>
__global__ void __launch_bounds__(kv::kThreadsKV, 1)
    dkdv_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq,
                const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tkt,
                const __grid_constant__ CUtensorMap tvt) {
  using namespace kv;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
  uint8_t* sStage = sm + kOffStage;
  Cols* cols = reinterpret_cast<Cols*>(sm + kOffCol);
  Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_status = reinterpret_cast<int*>(s_tmem + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int ntiles = ktile_count(p);
  if (tid == 0) {
    *s_status = *reinterpret_cast<volatile int32_t*>(p.status);
    // every tile here needs a 1024-byte-aligned base (swizzle atoms)
    if (smem_addr(sm) & 1023u) {
      atomicOr(p.status, ATTN_DEV_SMEM_ALIGN);
      *s_status = 1;
    }
  }
  __syncthreads();
  if (*s_status != 0 || static_cast<int>(blockIdx.x) >= ntiles) return;

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->st_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], 1);
    }
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_free, 1);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->cols_x[0], 8);
    mbar_init(&bars->cols_x[1], 8);
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
  const int step_tok = kRowsKV / G;
  const int ngroups = p.Hq / G;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tq);
      prefetch_tensormap(&tdo);
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tv);
      prefetch_tensormap(&tkt);
      prefetch_tensormap(&tvt);
      uint32_t armed = 0;  // stage fills armed
      int tcount = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < ntiles && ok; item += gridDim.x, ++tcount) {
        KTile t;
        ktile_decode(p, item, t);
        const int nsteps = ((t.Lq + step_tok - 1) / step_tok) * ngroups;
        if (tcount > 0 && !(ok = mbar_wait(&bars->kv_empty, (tcount - 1) & 1, s_abort))) break;
        mbar_arrive_expect_tx(&bars->kv_full, 2 * kKV);
        for (int c = 0; c < 2; ++c) {
          tma_load_2d(sK + c * kTile, &tk, &bars->kv_full, c * kChunk, t.k0 + t.key);
          tma_load_2d(sV + c * kTile, &tv, &bars->kv_full, c * kChunk, t.k0 + t.key);
        }
        tma_load_2d(sK + 2 * kTile, &tkt, &bars->kv_full, 2 * kChunk, t.k0 + t.key);
        tma_load_2d(sV + 2 * kTile, &tvt, &bars->kv_full, 2 * kChunk, t.k0 + t.key);
        for (int st = 0; st < nsteps; ++st, ++armed) {
          const int s = armed % kStages;
          const int tok0 = (st / ngroups) * step_tok;
          const int hg = st % ngroups;
          if (armed >= kStages &&
              !(ok = mbar_wait(&bars->st_empty[s], (armed / kStages - 1) & 1, s_abort)))
            break;
          mbar_arrive_expect_tx(&bars->st_full[s], 6 * kTileQ);
          uint8_t* dst = sStage + s * kStage;
          for (int c = 0; c < 3; ++c) {
            tma_load_3d(dst + c * kTileQ, &tq, &bars->st_full[s], c * kChunk, hg * G, t.q0 + tok0);
            tma_load_3d(dst + (3 + c) * kTileQ, &tdo, &bars->st_full[s], c * kChunk, hg * G,
                        t.q0 + tok0);
          }
        }
      }
      if (*s_abort) {
        if (tcount > 0) drain_wait_kv(&bars->kv_full, (tcount - 1) & 1);
        for (uint32_t f = armed > kStages ? armed - kStages : 0; f < armed; ++f)
          drain_wait_kv(&bars->st_full[f % kStages], (f / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 64, BF16, false, false);
      constexpr uint32_t kIdG = idesc_f16(128, kHeadDim, BF16, false, true);
      const uint32_t kb = smem_addr(sK), vb = smem_addr(sV);
      uint32_t g = 0;
      int tcount = 0;
      bool ok = true;
      // A = K or V (features 0..127 in 128-byte-swizzled chunks, 128..159 in
      // a 64-byte-swizzled chunk); B = the step's Q or dO chunks.
      auto a_desc = [&](uint32_t base, int k) -> uint64_t {
        return k < 8 ? sdesc_sw128(base + (k >> 2) * kTile + (k & 3) * 32, 16, 1024)
                     : sdesc_sw64(base + 2 * kTile + (k - 8) * 32);
      };
      auto issue_st = [&](uint32_t gs) -> bool {  // S^T = K Q^T for step gs
        if (!mbar_wait(&bars->st_full[gs % kStages], (gs / kStages) & 1, s_abort)) return false;
        if (gs >= 2 && !mbar_wait(&bars->s_free[gs & 1], ((gs - 2) >> 1) & 1, s_abort))
          return false;
        tc_fence_after();
        const uint32_t qb = smem_addr(sStage + (gs % kStages) * kStage);
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          umma_ss(tmem + kColS + (gs & 1) * 64, a_desc(kb, k),
                  sdesc_sw128(qb + (k >> 2) * kTileQ + (k & 3) * 32, 16, 1024), kIdS, k > 0);
        umma_commit(&bars->s_full[gs & 1]);
        return true;
      };
      auto issue_dpt = [&](uint32_t gs) -> bool {  // dP^T = V dO^T for step gs
        if (gs >= 1 && !mbar_wait(&bars->dp_free, (gs - 1) & 1, s_abort)) return false;
        tc_fence_after();
        const uint32_t db = smem_addr(sStage + (gs % kStages) * kStage + 3 * kTileQ);
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k)
          umma_ss(tmem + kColP, a_desc(vb, k),
                  sdesc_sw128(db + (k >> 2) * kTileQ + (k & 3) * 32, 16, 1024), kIdS, k > 0);
        umma_commit(&bars->dp_full);
        return true;
      };
      for (int item = blockIdx.x; item < ntiles && ok; item += gridDim.x, ++tcount) {
        KTile t;
        ktile_decode(p, item, t);
        const int nsteps = ((t.Lq + step_tok - 1) / step_tok) * ngroups;
        if (!(ok = mbar_wait(&bars->kv_full, tcount & 1, s_abort))) break;
        if (nsteps == 0) {  // no queries: dk = dv = 0; keep every phase count
          mbar_arrive(&bars->kv_empty);
          if (tcount > 0 && !(ok = mbar_wait(&bars->acc_empty, (tcount - 1) & 1, s_abort))) break;
          mbar_arrive(&bars->acc_full);
          continue;
        }
        if (!(ok = issue_st(g)) || !(ok = issue_dpt(g))) break;
        for (int st = 0; st < nsteps; ++st) {
          const uint32_t gg = g + st;
          if (st + 1 < nsteps && !(ok = issue_st(gg + 1))) break;
          if (!(ok = mbar_wait(&bars->p_full, gg & 1, s_abort))) break;
          if (st == 0 && tcount > 0 &&
              !(ok = mbar_wait(&bars->acc_empty, (tcount - 1) & 1, s_abort)))
            break;
          tc_fence_after();
          const uint32_t sb = smem_addr(sStage + (gg % kStages) * kStage);
          const uint32_t pa = tmem + kColS + (gg & 1) * 64;
          // query rows 16k..16k+15 of the step: half k/2, pair column 8*(k%2)
#pragma unroll
          for (int k = 0; k < kRowsKV / 16; ++k)  // dV += P^T dO
            umma_ts(tmem + kColDV, pa + (k >> 1) * 32 + (k & 1) * 8,
                    sdesc_sw128(sb + 3 * kTileQ + k * 2048, kTileQ, 1024), kIdG,
                    (st > 0 || k > 0));
#pragma unroll
          for (int k = 0; k < kRowsKV / 16; ++k)  // dK += dS^T Q
            umma_ts(tmem + kColDK, tmem + kColP + (k >> 1) * 32 + (k & 1) * 8,
                    sdesc_sw128(sb + k * 2048, kTileQ, 1024), kIdG, (st > 0 || k > 0));
          umma_commit(&bars->s_free[gg & 1]);
          umma_commit(&bars->dp_free);
          umma_commit(&bars->st_empty[gg % kStages]);
          if (st == nsteps - 1) {
            umma_commit(&bars->acc_full);
            umma_commit(&bars->kv_empty);
          } else if (!(ok = issue_dpt(gg + 1))) {
            break;
          }
        }
        g += nsteps;
      }
      umma_commit(&bars->drain);
      drain_wait_kv(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;  // which 32 of the step's 64 query columns
    const int r = quad * 32 + lane;    // key within the tile (TMEM lane)
    const int e = (warp - 2) * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const LogitMap lm = make_logit_map(p);
    const bool masked = masking(p);
    const int wr = p.causal ? 0 : p.wr;
    // Threads 0..127 of this role also fetch one scalar column of a query
    // step: 0..63 the lse, slope and aligned position of column e, 64..127
    // the D of column e - 64.
    const int lc = e & 63;
    const bool fetcher = e < 128;
    const bool loads_d = e >= 64;
    auto fetch = [&](const KTile& t, int st, float& a, float& b, float& c) {
      if (!fetcher) return;
      const int i = (st / ngroups) * step_tok + lc / G;
      const int h = (st % ngroups) * G + lc % G;
      const int64_t ri = static_cast<int64_t>(t.q0 + i) * p.Hq + h;
      if (loads_d) {
        a = i < t.Lq ? __ldg(p.Dbuf + ri) : 0.f;
      } else {
        const float lse = i < t.Lq ? __ldg(p.lse + ri) : -INFINITY;
        a = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
        b = p.slopes ? __ldg(p.slopes + t.b * p.slopes_bs + h) * kLog2e : 0.f;
        c = static_cast<float>(i + t.Lk - t.Lq);
      }
    };
    auto publish = [&](Cols* cs, float a, float b, float c) {
      if (!fetcher) return;
      if (loads_d) {
        cs->D[lc] = a;
      } else {
        cs->lse2[lc] = a;
        cs->slope2[lc] = b;
        cs->pos[lc] = c;
      }
    };
    uint32_t g = 0;
    int tcount = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < ntiles && ok; item += gridDim.x, ++tcount) {
      KTile t;
      ktile_decode(p, item, t);
      const int nsteps = ((t.Lq + step_tok - 1) / step_tok) * ngroups;
      const int j = t.key + r;
      const float jf = static_cast<float>(j);
      if (nsteps > 0) {
        float a = 0.f, b = 0.f, c = 0.f;
        fetch(t, 0, a, b, c);
        publish(cols + (g & 1), a, b, c);
        if (!(ok = warp_exchange(&bars->cols_x[g & 1], (g >> 1) & 1, s_abort))) break;
      }
      for (int st = 0; st < nsteps; ++st) {
        const uint32_t gg = g + st;
        const Cols* cs = cols + (gg & 1);
        const bool more = st + 1 < nsteps;
        float na = 0.f, nb = 0.f, nc = 0.f;
        if (more) fetch(t, st + 1, na, nb, nc);  // lands while this step runs
        const uint32_t sbuf = tmem + kColS + (gg & 1) * 64 + half * 32 + lane_addr;
        const uint32_t pbuf = tmem + kColP + half * 32 + lane_addr;
        // this half's 32 columns of the per-column scalars
        const float4* s_l2 = reinterpret_cast<const float4*>(cs->lse2 + half * 32);
        const float4* s_sl = reinterpret_cast<const float4*>(cs->slope2 + half * 32);
        const float4* s_ps = reinterpret_cast<const float4*>(cs->pos + half * 32);
        const float4* s_d = reinterpret_cast<const float4*>(cs->D + half * 32);
        if (!(ok = mbar_wait_warp(&bars->s_full[gg & 1], (gg >> 1) & 1, s_abort))) break;
        tc_fence_after();
        float x[32];
        tmem_ld32(sbuf, x);
        tmem_wait_ld();
        // Batched so that dependent MUFU results are 32 instructions apart:
        // all tanh, then all biases and exponent arguments, then all exp2.
        float th[32], z[32];
        if (lm.capped) {
#pragma unroll
          for (int c = 0; c < 32; ++c) th[c] = tanh_approx(x[c] * lm.in_scale);
        }
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 l2 = s_l2[q4], sl = s_sl[q4], ps = s_ps[q4];
          const float l2v[4] = {l2.x, l2.y, l2.z, l2.w};
          const float slv[4] = {sl.x, sl.y, sl.z, sl.w};
          const float psv[4] = {ps.x, ps.y, ps.z, ps.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = q4 * 4 + u;
            // base-2 logit minus lse: t*c*log2e - slope2*|pos - j| - lse2
            const float bias = fmaf(-slv[u], fabsf(psv[u] - jf), -l2v[u]);
            z[c] = lm.capped ? fmaf(th[c], lm.out_scale, bias) : fmaf(x[c], lm.in_scale, bias);
            if (masked) {
              const bool adm = (p.wl < 0 || jf >= psv[u] - static_cast<float>(p.wl)) &&
                               (wr < 0 || jf <= psv[u] + static_cast<float>(wr));
              z[c] = adm ? z[c] : -INFINITY;
            }
          }
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) z[c] = ex2_approx(z[c]);  // P
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          pk[c >> 1] = Pack<BF16>::two(z[c], z[c + 1]);
          // P * (1 - tanh^2): dS = this * (dP - D)
          x[c] = lm.capped ? z[c] * fmaf(-th[c], th[c], 1.f) : z[c];
          x[c + 1] = lm.capped ? z[c + 1] * fmaf(-th[c + 1], th[c + 1], 1.f) : z[c + 1];
        }
        tmem_st16(sbuf, pk);  // P^T pairs over this half's own (already read) columns
        if (!(ok = mbar_wait_warp(&bars->dp_full, gg & 1, s_abort))) break;
        tc_fence_after();
        float d[32];
        tmem_ld32(pbuf, d);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 dd = s_d[q4];
          pk[q4 * 2] = Pack<BF16>::two(x[q4 * 4] * (d[q4 * 4] - dd.x),
                                       x[q4 * 4 + 1] * (d[q4 * 4 + 1] - dd.y));
          pk[q4 * 2 + 1] = Pack<BF16>::two(x[q4 * 4 + 2] * (d[q4 * 4 + 2] - dd.z),
                                           x[q4 * 4 + 3] * (d[q4 * 4 + 3] - dd.w));
        }
        tmem_st16(pbuf, pk);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
        if (more) {
          publish(cols + ((gg + 1) & 1), na, nb, nc);
          if (!(ok = warp_exchange(&bars->cols_x[(gg + 1) & 1], ((gg + 1) >> 1) & 1, s_abort)))
            break;
        }
      }
      if (!ok) break;
      g += nsteps;
      // ---- epilogue: half 0 writes dv = dV, half 1 writes dk = sigma * dK
      if (!(ok = mbar_wait_warp(&bars->acc_full, tcount & 1, s_abort))) break;
      tc_fence_after();
      const bool key_valid = j < t.Lk;
      const float scale = half ? p.sigma : 1.f;
      uint16_t* row = half ? static_cast<uint16_t*>(p.dk) + static_cast<int64_t>(t.k0 + j) * p.dk_ts
                           : static_cast<uint16_t*>(p.dv) + static_cast<int64_t>(t.k0 + j) * p.dv_ts;
      const uint32_t acc = tmem + (half ? kColDK : kColDV) + lane_addr;
#pragma unroll 1
      for (int c = 0; c < kHeadDim / 32; ++c) {
        float a[32];
        tmem_ld32(acc + c * 32, a);
        tmem_wait_ld();
        if (key_valid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = nsteps > 0 ? a[8 * u + i] * scale : 0.f;
            *reinterpret_cast<uint4*>(row + c * 32 + u * 8) = pack8<BF16>(w);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty);
    }
  }

  __syncthreads();
  if (tid == 0 && *s_abort) atomicOr(p.status, ATTN_DEV_TIMEOUT_DKDV);
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_dkdv(const Params& p, const CUtensorMap& tq64, const CUtensorMap& tdo64,
                        const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tkt,
                        const CUtensorMap& tvt, int grid, cudaStream_t s) {
  if (p.dtype == 1) {
    auto k = dkdv_kernel<true>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kSmem);
    k<<<grid, kv::kThreadsKV, kv::kSmem, s>>>(p, tq64, tdo64, tk, tv, tkt, tvt);
  } else {
    auto k = dkdv_kernel<false>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kSmem);
    k<<<grid, kv::kThreadsKV, kv::kSmem, s>>>(p, tq64, tdo64, tk, tv, tkt, tvt);
  }
  return cudaGetLastError();
}

}  // namespace attn
