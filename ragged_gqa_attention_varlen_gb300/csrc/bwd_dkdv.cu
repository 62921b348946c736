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
// accumulators in TMEM (2 x 160 fp32 columns) while it walks every 128-row
// query step (128/G tokens x G heads, the forward's query tile) of the
// sequence in a fixed order, so the reduction order over heads and queries
// never changes: no atomics, bitwise repeatable.  Per query step, keys in the
// MMA M dimension (every MMA has N >= 128, which keeps the shared-memory
// operand traffic within what the tensor core can consume at full rate):
//   S^T  = K Q^T        M=128 N=128 K=160 -> TMEM columns [320, 448)
//   P^T                 elementwise warps; 16-bit pairs over read S^T columns
//   dP^T = V dO^T       M=128 N=128 K=160 -> TMEM columns [384, 512), issued as
//                       soon as S^T has been read (it overlaps S^T's upper half)
//   dS^T                elementwise warps; 16-bit pairs over read dP^T columns
//   dV  += P^T dO, dK += dS^T Q      M=128 N=160 K=128, A operand from TMEM
//
// Warp roles (384 threads, 12 warps): warp 0 loads (K, V once per key tile; Q through
// two slots, dO through one), warp 1 issues the MMAs, warps 4-11 compute P^T
// and dS^T and write dk/dv -- two warps per TMEM lane quadrant, each taking
// 64 of the step's 128 query columns.  They also fetch the next step's
// per-column scalars (lse, D, slope, aligned key position) while the current
// step runs.  K and V are only K-major operands here and keep their last 32
// features in a 64-byte-swizzled chunk; Q and dO are also MN-major operands
// (of dK and dV) and stay in three 128-byte-swizzled chunks.
// Warps 2-3 only complete warpgroup 0, which hands most of its registers to
// the elementwise warpgroups (setmaxnreg), so those can keep every column's
// MUFU/FMA chain of a batch in flight.
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace kv {
constexpr int kThreadsKV = kThreads;  // 12 warps
constexpr uint32_t kTile = 16384;   // 64-feature chunk of 128 rows
constexpr uint32_t kTail = 8192;    // features 128..159 of 128 rows (64-byte rows)
constexpr uint32_t kKV = 2 * kTile + kTail;
constexpr uint32_t kTile3 = 3 * kTile;
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kKV;
constexpr uint32_t kOffQ = 2 * kKV;              // two Q slots
constexpr uint32_t kOffDO = kOffQ + 2 * kTile3;  // one dO slot
constexpr uint32_t kOffCol = kOffDO + kTile3;    // the step's column scalars
constexpr uint32_t kOffBar = kOffCol + 4 * 128 * 4;
constexpr uint32_t kSmem = kOffBar + 256;  // the dynamic base is checked to be 1024-aligned
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDV = 0;
constexpr uint32_t kColDK = 160;
constexpr uint32_t kColS = 320;  // S^T: [320, 448); P^T pairs: [320, 384)
constexpr uint32_t kColP = 384;  // dP^T: [384, 512); dS^T pairs: [384,416) and [448,480)

struct Cols {  // per-column scalars of one query step (column = token * G + head)
  float lse2[128];    // lse * log2(e); +inf where no P exists (row outside / empty)
  float D[128];
  float slope2[128];  // slope * log2(e)
  float pos[128];     // i + Lk - Lq (the key aligned with query row i)
};

struct Bars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2], do_full, do_empty;
  uint64_t s_full, s_read, dp_full, p_full, ds_full, dk_done;
  uint64_t acc_full, acc_empty, cols_x, drain;
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
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sDO = sm + kOffDO;
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
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 1);
    }
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->do_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_read, 8);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->cols_x, 8);
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
  const int step_tok = kRowsQ / G;
  const int ngroups = p.Hq / G;

  // Each role runs inside the branch that set its register budget, so the
  // compiler allocates each branch against its own budget.
  if (warp < 4) {
  warpgroup_reg_dealloc<kRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tq);
      prefetch_tensormap(&tdo);
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tv);
      prefetch_tensormap(&tkt);
      prefetch_tensormap(&tvt);
      uint32_t g = 0;                  // query steps armed
      uint32_t dfill = 0;              // dO fills armed
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
        for (int st = 0; st < nsteps; ++st) {
          const int tok = t.q0 + (st / ngroups) * step_tok;
          const int hg = st % ngroups;
          const int s = g & 1;
          // Q of step g (its slot was last read by dK of step g - 2)
          if (g >= 2 && !(ok = mbar_wait(&bars->q_empty[s], ((g - 2) >> 1) & 1, s_abort))) break;
          mbar_arrive_expect_tx(&bars->q_full[s], kTile3);
          for (int c = 0; c < 3; ++c)
            tma_load_3d(sQ + s * kTile3 + c * kTile, &tq, &bars->q_full[s], c * kChunk, hg * G, tok);
          ++g;
          // dO of the step (its slot was last read by dV of the previous step)
          if (dfill >= 1 && !(ok = mbar_wait(&bars->do_empty, (dfill - 1) & 1, s_abort))) break;
          mbar_arrive_expect_tx(&bars->do_full, kTile3);
          for (int c = 0; c < 3; ++c)
            tma_load_3d(sDO + c * kTile, &tdo, &bars->do_full, c * kChunk, hg * G, tok);
          ++dfill;
        }
      }
      if (*s_abort) {
        if (tcount > 0) drain_wait_kv(&bars->kv_full, (tcount - 1) & 1);
        for (uint32_t f = g > 2 ? g - 2 : 0; f < g; ++f)
          drain_wait_kv(&bars->q_full[f & 1], (f >> 1) & 1);
        if (dfill > 0) drain_wait_kv(&bars->do_full, (dfill - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t kIdG = idesc_f16(128, kHeadDim, BF16, false, true);
      const uint32_t kb = smem_addr(sK), vb = smem_addr(sV), db = smem_addr(sDO);
      // A = K or V: features 0..127 in 128-byte-swizzled chunks, 128..159 in a
      // 64-byte-swizzled chunk.  B = the step's Q or dO (three 128-byte chunks).
      auto a_desc = [&](uint32_t base, int k) -> uint64_t {
        return k < 8 ? sdesc_sw128(base + (k >> 2) * kTile + (k & 3) * 32, 16, 1024)
                     : sdesc_sw64(base + 2 * kTile + (k - 8) * 32);
      };
      auto b_desc = [&](uint32_t base, int k) -> uint64_t {
        return sdesc_sw128(base + (k >> 2) * kTile + (k & 3) * 32, 16, 1024);
      };
      uint32_t g = 0;
      int tcount = 0;
      bool ok = true;
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
        for (int st = 0; st < nsteps; ++st) {
          const uint32_t gg = g + st;
          const uint32_t qb = smem_addr(sQ + (gg & 1) * kTile3);
          // S^T = K Q^T, once the previous step's dK (last reader of the
          // region) is done
          if (!(ok = mbar_wait(&bars->q_full[gg & 1], (gg >> 1) & 1, s_abort))) break;
          if (gg >= 1 && !(ok = mbar_wait(&bars->dk_done, (gg - 1) & 1, s_abort))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k)
            umma_ss(tmem + kColS, a_desc(kb, k), b_desc(qb, k), kIdS, k > 0);
          umma_commit(&bars->s_full);
          // dP^T = V dO^T over S^T's upper half once S^T has been read
          if (!(ok = mbar_wait(&bars->s_read, gg & 1, s_abort))) break;
          if (!(ok = mbar_wait(&bars->do_full, gg & 1, s_abort))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k)
            umma_ss(tmem + kColP, a_desc(vb, k), b_desc(db, k), kIdS, k > 0);
          umma_commit(&bars->dp_full);
          // dV += P^T dO; query rows 16k..16k+15 are pair columns
          // 320 + 32*(k/4) + 8*(k%4)
          if (!(ok = mbar_wait(&bars->p_full, gg & 1, s_abort))) break;
          if (st == 0 && tcount > 0 &&
              !(ok = mbar_wait(&bars->acc_empty, (tcount - 1) & 1, s_abort)))
            break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kRowsQ / 16; ++k)
            umma_ts(tmem + kColDV, tmem + kColS + (k >> 2) * 32 + (k & 3) * 8,
                    sdesc_sw128(db + k * 2048, kTile, 1024), kIdG, (st > 0 || k > 0));
          umma_commit(&bars->do_empty);
          // dK += dS^T Q; query rows 16k..16k+15 are pair columns
          // 384 + 64*(k/4) + 8*(k%4)
          if (!(ok = mbar_wait(&bars->ds_full, gg & 1, s_abort))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kRowsQ / 16; ++k)
            umma_ts(tmem + kColDK, tmem + kColP + (k >> 2) * 64 + (k & 3) * 8,
                    sdesc_sw128(qb + k * 2048, kTile, 1024), kIdG, (st > 0 || k > 0));
          umma_commit(&bars->dk_done);
          umma_commit(&bars->q_empty[gg & 1]);
          if (st == nsteps - 1) {
            umma_commit(&bars->acc_full);
            umma_commit(&bars->kv_empty);
          }
        }
        g += nsteps;
      }
      umma_commit(&bars->drain);
      drain_wait_kv(&bars->drain, 0);
    }
  }
  } else {
  warpgroup_reg_alloc<kRegsHigh>();
  {
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;  // query columns [64*half, 64*half + 64)
    const int r = quad * 32 + lane;    // key within the tile (TMEM lane)
    const int e = (warp - 4) * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const LogitMap lm = make_logit_map(p);
    const bool masked = masking(p);
    const int wr = p.causal ? 0 : p.wr;
    // Each thread also fetches one scalar column of a query step: threads
    // 0..127 the lse, slope and aligned position of column e, 128..255 the D
    // of column e - 128.
    const int lc = e & 127;
    const bool loads_d = e >= 128;
    auto fetch = [&](const KTile& t, int st, float& a, float& b, float& c) {
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
    auto publish = [&](float a, float b, float c) {
      if (loads_d) {
        cols->D[lc] = a;
      } else {
        cols->lse2[lc] = a;
        cols->slope2[lc] = b;
        cols->pos[lc] = c;
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
      float na = 0.f, nb = 0.f, nc = 0.f;
      if (nsteps > 0) fetch(t, 0, na, nb, nc);
      for (int st = 0; st < nsteps; ++st) {
        const uint32_t gg = g + st;
        // publish this step's scalars into the single scalar buffer once every
        // warp is done with the previous step's (its dS^T, the last use, is
        // signalled by ds_full of that step)
        if (gg >= 1 && !(ok = mbar_wait_warp(&bars->ds_full, (gg - 1) & 1, s_abort))) break;
        publish(na, nb, nc);
        if (!(ok = warp_exchange(&bars->cols_x, gg & 1, s_abort))) break;
        if (st + 1 < nsteps) fetch(t, st + 1, na, nb, nc);  // lands while this step runs
        const float4* s_l2 = reinterpret_cast<const float4*>(cols->lse2 + half * 64);
        const float4* s_sl = reinterpret_cast<const float4*>(cols->slope2 + half * 64);
        const float4* s_ps = reinterpret_cast<const float4*>(cols->pos + half * 64);
        const float4* s_d = reinterpret_cast<const float4*>(cols->D + half * 64);
        // Everything that does not depend on S^T first, while S^T is being
        // computed: the base-2 bias -slope2*|pos - j| - lse2 of each column.
        float bias[64];
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 l2 = s_l2[q4], sl = s_sl[q4], ps = s_ps[q4];
          const float l2v[4] = {l2.x, l2.y, l2.z, l2.w};
          const float slv[4] = {sl.x, sl.y, sl.z, sl.w};
          const float psv[4] = {ps.x, ps.y, ps.z, ps.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float bv = fmaf(-slv[u], fabsf(psv[u] - jf), -l2v[u]);
            if (masked) {
              const bool adm = (p.wl < 0 || jf >= psv[u] - static_cast<float>(p.wl)) &&
                               (wr < 0 || jf <= psv[u] + static_cast<float>(wr));
              bv = adm ? bv : -INFINITY;
            }
            bias[q4 * 4 + u] = bv;
          }
        }
        if (!(ok = mbar_wait_warp(&bars->s_full, gg & 1, s_abort))) break;
        tc_fence_after();
        float x[64];
        const uint32_t sbuf = tmem + kColS + half * 64 + lane_addr;
        tmem_ld32(sbuf, *reinterpret_cast<float(*)[32]>(x));
        tmem_ld32(sbuf + 32, *reinterpret_cast<float(*)[32]>(x + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_read);
        // P = exp2(t*c*log2e + bias) and P (1 - tanh^2), in two batches of 32:
        // all tanh (in place of S), then all exp2 (in place of the bias)
        uint32_t pk[32];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float* xb = x + b * 32;
          float* zb = bias + b * 32;
          if (lm.capped) {
#pragma unroll
            for (int c = 0; c < 32; ++c) xb[c] = tanh_approx(xb[c] * lm.in_scale);
#pragma unroll
            for (int c = 0; c < 32; ++c) zb[c] = fmaf(xb[c], lm.out_scale, zb[c]);
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) zb[c] = fmaf(xb[c], lm.in_scale, zb[c]);
          }
#pragma unroll
          for (int c = 0; c < 32; ++c) zb[c] = ex2_approx(zb[c]);  // P
#pragma unroll
          for (int c = 0; c < 32; c += 2) pk[b * 16 + (c >> 1)] = Pack<BF16>::two(zb[c], zb[c + 1]);
#pragma unroll
          for (int c = 0; c < 32; ++c)  // P (1 - tanh^2): dS = this * (dP - D)
            xb[c] = lm.capped ? zb[c] * fmaf(-xb[c], xb[c], 1.f) : zb[c];
        }
        // P^T pairs: this half's 64 columns -> 32 pair columns at 320 + 32*half,
        // which may still hold S^T of the other half until every warp has read it
        if (!(ok = mbar_wait_warp(&bars->s_read, gg & 1, s_abort))) break;
        const uint32_t pdst = tmem + kColS + half * 32 + lane_addr;
        tmem_st16(pdst, *reinterpret_cast<uint32_t(*)[16]>(pk));
        tmem_st16(pdst + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
        // D of each column into the (now free) bias registers before dP^T lands
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
          const float4 dd = s_d[q4];
          bias[q4 * 4] = dd.x;
          bias[q4 * 4 + 1] = dd.y;
          bias[q4 * 4 + 2] = dd.z;
          bias[q4 * 4 + 3] = dd.w;
        }
        // dS^T = P (1 - tanh^2) (dP - D), written over this half's own dP^T columns
        if (!(ok = mbar_wait_warp(&bars->dp_full, gg & 1, s_abort))) break;
        tc_fence_after();
        const uint32_t pbuf = tmem + kColP + half * 64 + lane_addr;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float d[32];
          tmem_ld32(pbuf + cc * 32, d);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            pk[cc * 16 + (c >> 1)] =
                Pack<BF16>::two(x[cc * 32 + c] * (d[c] - bias[cc * 32 + c]),
                                x[cc * 32 + c + 1] * (d[c + 1] - bias[cc * 32 + c + 1]));
        }
        tmem_st16(pbuf, *reinterpret_cast<uint32_t(*)[16]>(pk));
        tmem_st16(pbuf + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->ds_full);
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

  }
  __syncthreads();
  if (tid == 0 && *s_abort) atomicOr(p.status, ATTN_DEV_TIMEOUT_DKDV);
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

cudaError_t launch_dkdv(const Params& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                        const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tkt,
                        const CUtensorMap& tvt, int grid, cudaStream_t s) {
  if (p.dtype == 1) {
    auto k = dkdv_kernel<true>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kSmem);
    k<<<grid, kv::kThreadsKV, kv::kSmem, s>>>(p, tq, tdo, tk, tv, tkt, tvt);
  } else {
    auto k = dkdv_kernel<false>;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kSmem);
    k<<<grid, kv::kThreadsKV, kv::kSmem, s>>>(p, tq, tdo, tk, tv, tkt, tvt);
  }
  return cudaGetLastError();
}

}  // namespace attn
