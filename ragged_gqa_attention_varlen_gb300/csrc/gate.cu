// gate.cu -- the sigmoid-gated variant: forward, dq and dk/dv kernels.
//
// "Pairwise-Gated Attention Engine" ("Why it is hard") gives the operation
//   O = (softmax(Q K^T / sqrt(D)) o sigmoid(Q_g K_g^T / sqrt(R))) V
// with a gate from separate projections q_g, k_g of width R that scales each
// normalised weight: the gate sits outside the softmax normalisation, so lse
// stays the ungated one and out_i = sum_j P_ij G_ij v_j.  The backward pass
// (the chain rule of that definition) is, with W = P o G and dW = dO V^T:
//   D_i   = dO_i . out_i               (as without the gate)
//   dS_ij = P_ij (G_ij dW_ij - D_i) = W_ij dW_ij - P_ij D_i
//   dg_ij = dW_ij W_ij (1 - G_ij)      (gradient at the gate logit)
//   dq = sigma dS K,  dk = sigma dS^T Q,  dv = W^T dO,
//   dq_g = dg K_g / sqrt(R),  dk_g = dg^T Q_g / sqrt(R).
// The page's attention is the plain softmax, so these kernels take no
// softcap; ALiBi, causal/window masks and grouped K/V heads are those of the
// rest of the library.  G = sigmoid(x) is taken as 1/2 + tanh(x/2)/2.
//
// Head dimension 64 or 128 (the page's sizes): tiles are 128 rows of one or
// two 64-feature chunks in the 128-byte swizzle, and the gate projections are
// staged as one 64-wide chunk (a width of 32 is zero-filled by the tensor
// map, which adds nothing to any product).
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace gt {
constexpr uint32_t kChunkB = 16384;  // 128 rows x 64 16-bit values, 128-byte swizzle
template <int HD>
struct Dim {
  static constexpr int NC = HD / 64;                  // feature chunks of a tile
  static constexpr uint32_t kTileB = NC * kChunkB;    // a 128-row tile of HD features
};

__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

// Operand descriptors of a tile of 64-wide chunks, as a base descriptor plus
// the byte offset of K step k: K-major (16 elements of the contraction per
// step, 32 bytes within a chunk, chunks kChunkB apart) or MN-major (16 rows
// of the contraction per step, N running along the chunk's 64 values).
__device__ __forceinline__ SDesc kbase(uint32_t base) {
  return sdesc_split(sdesc_sw128(base, 16, 1024));
}
__device__ __forceinline__ SDesc mbase(uint32_t base) {
  return sdesc_split(sdesc_sw128(base, kChunkB, 1024));
}
__device__ __forceinline__ constexpr uint32_t koff(int k) {
  return (k >> 2) * kChunkB + (k & 3) * 32;
}
__device__ __forceinline__ constexpr uint32_t moff(int k) { return k * 2048; }

// sigmoid(x * scale) as 1/2 + tanh(x * scale / 2) / 2
__device__ __forceinline__ float gate_of(float x, float half_scale) {
  return fmaf(0.5f, tanh_approx(x * half_scale), 0.5f);
}
}  // namespace gt

// ============================================================== forward

namespace gf {
template <int HD>
struct Lay {
  static constexpr uint32_t T = gt::Dim<HD>::kTileB;
  static constexpr uint32_t offQ = 0;
  static constexpr uint32_t offQg = offQ + T;
  static constexpr uint32_t slotK = T + gt::kChunkB;  // K, then K_g, of one slot
  static constexpr uint32_t offK = offQg + gt::kChunkB;
  static constexpr uint32_t offV = offK + 2 * slotK;
  static constexpr uint32_t offMax = offV + 2 * T;   // [2 steps][2 halves][128] fp32
  static constexpr uint32_t offSum = offMax + 2 * 2 * 128 * 4;
  static constexpr uint32_t offBar = offSum + 2 * 2 * 128 * 4;
};
constexpr uint32_t kColS = 0;    // S = Q K^T
constexpr uint32_t kColG = 128;  // gate logits Q_g K_g^T
constexpr uint32_t kColP = 256;  // P o G as 16-bit pairs (64 columns)
constexpr uint32_t kColO = 320;  // O accumulator (HD columns)
constexpr float kRescale = 8.f;  // lazy-rescale threshold (base 2)

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full, s_read, p_full, pv_done;
  uint64_t o_full, o_empty, drain;
  uint64_t mx_x[2], l_x[2];
  TileRing ring;
};
template <int HD>
constexpr uint32_t smem_bytes() {
  return Lay<HD>::offBar + sizeof(Bars) + 16;
}
static_assert(smem_bytes<128>() <= 232448, "shared memory");
}  // namespace gf

// One CTA per SM, persistent; each tile is 128 query rows (128/G tokens x G
// heads of one group) against every key tile its rows may attend to.  Per
// key tile: S and the gate logits on the tensor core (warp 1), then per row
// P = 2^(z - m) with the running max m exchanged between the two warps of a
// lane quadrant (each takes 64 keys), W = P G into TMEM, and O += W V (warp
// 2).  l sums the ungated P, so out = O / l is the gated output of the
// normalised weights.  S and the gate logits have one TMEM buffer each: the
// softmax warps copy both to registers at once and release them.
template <bool BF16, bool MASK, int HD>
__global__ void __launch_bounds__(kThreads, 1)
    gate_fwd_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq,
                    const __grid_constant__ CUtensorMap tqg, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tkg,
                    const __grid_constant__ CUtensorMap tv) {
  using Ly = gf::Lay<HD>;
  using namespace gf;
  constexpr uint32_t T = Ly::T;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sQ = sm + Ly::offQ;
  uint8_t* sQg = sm + Ly::offQg;
  uint8_t* sK = sm + Ly::offK;
  uint8_t* sV = sm + Ly::offV;
  float* sMax = reinterpret_cast<float*>(sm + Ly::offMax);
  float* sSum = reinterpret_cast<float*>(sm + Ly::offSum);
  Bars* bars = reinterpret_cast<Bars*>(sm + Ly::offBar);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_status = reinterpret_cast<int*>(s_tmem + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int ntiles = qtile_count(p);
  if (tid == 0) {
    *s_status = *reinterpret_cast<volatile int32_t*>(p.status);
    if (smem_addr(sm) & 1023u) {
      atomicOr(p.status, ATTN_DEV_SMEM_ALIGN);
      *s_status = 1;
    }
  }
  __syncthreads();
  if (*s_status != 0 || static_cast<int>(blockIdx.x) >= ntiles) return;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->k_full[b], 1);
      mbar_init(&bars->k_empty[b], 1);
      mbar_init(&bars->v_full[b], 1);
      mbar_init(&bars->v_empty[b], 1);
      mbar_init(&bars->mx_x[b], 8);
      mbar_init(&bars->l_x[b], 8);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_read, 8);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 8);
    mbar_init(&bars->drain, 2);
    // readers: the Q/K and the V load lanes, the two MMA threads, 8 softmax warps
    tile_ring_init(&bars->ring, 12);
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int G = p.G;

  if (warp < 4) {
  warpgroup_reg_dealloc<kRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // lane 0: Q and K (+ the gate projections of both), lane 1: V
    if (lane < 2) {
      const bool kq = lane == 0;
      if (kq) {
        prefetch_tensormap(&tq);
        prefetch_tensormap(&tqg);
        prefetch_tensormap(&tk);
        prefetch_tensormap(&tkg);
      } else {
        prefetch_tensormap(&tv);
      }
      uint32_t g = 0;
      int tcount = 0;
      bool ok = true;
      uint32_t ktake = 0;
      int item = -1;
      for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        if (kq) {
          if (tcount > 0 && !(ok = mbar_wait(&bars->q_empty, (tcount - 1) & 1, s_abort))) break;
          mbar_arrive_expect_tx(&bars->q_full, T + gt::kChunkB);
          if (HD == 128)
            tma_load_4d(sQ, &tq, &bars->q_full, 0, t.hg * G, t.q0 + t.tok, 0);
          else
            tma_load_3d(sQ, &tq, &bars->q_full, 0, t.hg * G, t.q0 + t.tok);
          tma_load_3d(sQg, &tqg, &bars->q_full, 0, t.hg * G, t.q0 + t.tok);
        }
        for (int jj = 0; jj < t.nkt; ++jj, ++g) {
          const int key = t.k0 + (t.kt0 + jj) * kKeys;
          const int s = g & 1;
          if (g >= 2 && !(ok = mbar_wait(kq ? &bars->k_empty[s] : &bars->v_empty[s],
                                         ((g - 2) >> 1) & 1, s_abort)))
            break;
          if (kq) {
            uint8_t* dst = sK + s * Ly::slotK;
            mbar_arrive_expect_tx(&bars->k_full[s], Ly::slotK);
            if (HD == 128)
              tma_load_3d(dst, &tk, &bars->k_full[s], 0, key, 0);
            else
              tma_load_2d(dst, &tk, &bars->k_full[s], 0, key);
            tma_load_2d(dst + T, &tkg, &bars->k_full[s], 0, key);
          } else {
            uint8_t* dst = sV + s * T;
            mbar_arrive_expect_tx(&bars->v_full[s], T);
            if (HD == 128)
              tma_load_3d(dst, &tv, &bars->v_full[s], 0, key, 0);
            else
              tma_load_2d(dst, &tv, &bars->v_full[s], 0, key);
          }
        }
        if (!ok) break;
      }
      if (*s_abort) {
        if (kq && tcount > 0) gt::drain(&bars->q_full, (tcount - 1) & 1);
        for (uint32_t f = g > 2 ? g - 2 : 0; f < g; ++f)
          gt::drain(kq ? &bars->k_full[f & 1] : &bars->v_full[f & 1], (f >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S and gate logits
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
      uint32_t g = 0;
      int tcount = 0;
      bool ok = true;
      uint32_t ktake = 0;
      int item = -1;
      const SDesc qd = gt::kbase(smem_addr(sQ)), qgd = gt::kbase(smem_addr(sQg));
      for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        if (!(ok = mbar_wait(&bars->q_full, tcount & 1, s_abort))) break;
        if (t.nkt == 0) {
          mbar_arrive(&bars->q_empty);
          continue;
        }
        for (int jj = 0; jj < t.nkt; ++jj) {
          const uint32_t gs = g + jj;
          if (!(ok = mbar_wait(&bars->k_full[gs & 1], (gs >> 1) & 1, s_abort))) break;
          // the previous S and gate logits have been copied out by the softmax
          if (gs >= 1 && !(ok = mbar_wait(&bars->s_read, (gs - 1) & 1, s_abort))) break;
          tc_fence_after();
          const uint32_t kb = smem_addr(sK + (gs & 1) * Ly::slotK);
          const SDesc kd = gt::kbase(kb), kgd = gt::kbase(kb + T);
#pragma unroll
          for (int k = 0; k < HD / 16; ++k)
            umma_ss_off(tmem + kColS, qd, gt::koff(k), kd, gt::koff(k), kIdS, k > 0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_ss_off(tmem + kColG, qgd, gt::koff(k), kgd, gt::koff(k), kIdS, k > 0);
          umma_commit(&bars->s_full);
          umma_commit(&bars->k_empty[gs & 1]);
          if (jj == t.nkt - 1) umma_commit(&bars->q_empty);
        }
        if (!ok) break;
        g += t.nkt;
      }
      umma_commit(&bars->drain);
      gt::drain(&bars->drain, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ O += W V
    if (lane == 0) {
      constexpr uint32_t kIdO = idesc_f16(128, HD, BF16, false, true);
      uint32_t g = 0;
      int tcount = 0;
      bool ok = true;
      uint32_t ktake = 0;
      int item = -1;
      for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        if (t.nkt == 0) {
          if (tcount > 0 && !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort))) break;
          mbar_arrive(&bars->o_full);
          continue;
        }
        for (int jj = 0; jj < t.nkt; ++jj) {
          const uint32_t gg = g + jj;
          if (!(ok = mbar_wait(&bars->p_full, gg & 1, s_abort))) break;
          if (jj == 0 && tcount > 0 &&
              !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort)))
            break;
          if (!(ok = mbar_wait(&bars->v_full[gg & 1], (gg >> 1) & 1, s_abort))) break;
          tc_fence_after();
          const SDesc vd = gt::mbase(smem_addr(sV + (gg & 1) * T));
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k)
            umma_ts_off(tmem + kColO, tmem + kColP + k * 8, vd, gt::moff(k), kIdO,
                        (jj > 0 || k > 0));
          umma_commit(&bars->pv_done);
          umma_commit(&bars->v_empty[gg & 1]);
          if (jj == t.nkt - 1) umma_commit(&bars->o_full);
        }
        if (!ok) break;
        g += t.nkt;
      }
      umma_commit(&bars->drain);
      gt::drain(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ tile stream
    uint32_t kpub = 0;
    int it = 0;
    bool ok = true;
    while (ok && it >= 0) ok = tile_publish(&bars->ring, kpub, p.counters, ntiles, &it, s_abort);
  }
  } else {
  warpgroup_reg_alloc<kRegsHigh>();
  {
    // ------------------------------------------------------------ softmax
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;  // keys [64*half, 64*half + 64) of each key tile
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const float zscale = p.sigma * kLog2e;
    const float ghalf = 0.5f * p.gscale;
    uint32_t g = 0;
    int tcount = 0;
    bool ok = true;
    uint32_t ktake = 0;
    int item = -1;
    for (; (ok = tile_take_warp(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
      QTile t;
      qtile_decode<MASK>(p, item, t);
      const int i_loc = t.tok + r / G;
      const int h = t.hg * G + r % G;
      const bool row_valid = i_loc < t.Lq;
      const float slope2 = p.slopes ? __ldg(p.slopes + t.b * p.slopes_bs + h) * kLog2e : 0.f;
      const int pos_off = i_loc + t.Lk - t.Lq;
      float m_run = -INFINITY, l = 0.f;
      for (int jj = 0; jj < t.nkt; ++jj) {
        const uint32_t gg = g + jj;
        const int key0 = (t.kt0 + jj) * kKeys + half * 64;
        if (!(ok = mbar_wait_warp(&bars->s_full, gg & 1, s_abort))) break;
        tc_fence_after();
        float x[64], gv[64];
        const uint32_t sb = tmem + kColS + half * 64 + lane_addr;
        const uint32_t gb = tmem + kColG + half * 64 + lane_addr;
        tmem_ld32(sb, *reinterpret_cast<float(*)[32]>(x));
        tmem_ld32(sb + 32, *reinterpret_cast<float(*)[32]>(x + 32));
        tmem_ld32(gb, *reinterpret_cast<float(*)[32]>(gv));
        tmem_ld32(gb + 32, *reinterpret_cast<float(*)[32]>(gv + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_read);
        const float pos0 = static_cast<float>(pos_off - key0);
        // the gates as 16-bit pairs (W = P G is rounded to 16 bits anyway)
        uint32_t gp[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2)
          gp[c >> 1] = Pack<BF16>::two(gt::gate_of(gv[c], ghalf), gt::gate_of(gv[c + 1], ghalf));
#pragma unroll
        for (int c = 0; c < 64; ++c)
          x[c] = fmaf(x[c], zscale, -slope2 * fabsf(pos0 - static_cast<float>(c)));
        const bool edge =
            key0 + 64 > t.Lk ||
            (MASK && !__all_sync(0xffffffffu, !row_valid ||
                                                  all_admissible(p, t.Lq, t.Lk, i_loc, key0,
                                                                 key0 + 63)));
        if (edge) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int jg = key0 + c;
            bool adm = jg < t.Lk;
            if (MASK) adm = adm && admissible(p, t.Lq, t.Lk, i_loc, jg);
            x[c] = adm ? x[c] : -INFINITY;
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) mx = fmaxf(mx, x[c]);
        float* mxs = sMax + (gg & 1) * 256;
        mxs[half * 128 + r] = mx;
        if (!(ok = warp_exchange(&bars->mx_x[gg & 1], (gg >> 1) & 1, s_abort))) break;
        mx = fmaxf(mx, mxs[(half ^ 1) * 128 + r]);
        const float m_new = fmaxf(m_run, mx);
        const bool need = m_new > m_run + kRescale;
        const float alpha = need ? ex2_approx(m_run - m_new) : 1.f;
        // the previous W V has finished reading the P region (and adding to O)
        if (gg >= 1 && !(ok = mbar_wait_warp(&bars->pv_done, (gg - 1) & 1, s_abort))) break;
        tc_fence_after();
        if (jj > 0 && __any_sync(0xffffffffu, need)) {
          // O absorbs the new max: this half scales its HD/2 columns
          const uint32_t ob = tmem + kColO + half * (HD / 2) + lane_addr;
#pragma unroll 1
          for (int c = 0; c < HD / 64; ++c) {
            float o[32];
            tmem_ld32(ob + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(ob + c * 32, o);
            tmem_wait_st();
          }
        }
        if (need) {
          l *= alpha;
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float p0 = ex2_approx(x[c] - m_use), p1 = ex2_approx(x[c + 1] - m_use);
          l += p0 + p1;
          const uint64_t w = f2_mul(f2_make(p0, p1), Pack<BF16>::unpack(gp[c >> 1]));
          pk[c >> 1] = Pack<BF16>::two(f2_lo(w), f2_hi(w));
        }
        const uint32_t pb = tmem + kColP + half * 32 + lane_addr;
        tmem_st16(pb, *reinterpret_cast<uint32_t(*)[16]>(pk));
        tmem_st16(pb + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
      }
      if (!ok) break;
      g += t.nkt;
      // ---- epilogue: out = O / l with l the ungated sum, lse = m + log l
      float* ls = sSum + (tcount & 1) * 256;
      ls[half * 128 + r] = l;
      if (!(ok = warp_exchange(&bars->l_x[tcount & 1], (tcount >> 1) & 1, s_abort))) break;
      const float lt = l + ls[(half ^ 1) * 128 + r];
      if (!(ok = mbar_wait_warp(&bars->o_full, tcount & 1, s_abort))) break;
      tc_fence_after();
      const float inv = (lt > 0.f) ? 1.f / lt : 0.f;
      if (row_valid && half == 0)
        p.lse[static_cast<int64_t>(t.q0 + i_loc) * p.lse_rs + h] =
            (lt > 0.f) ? (m_run + log2f(lt)) * kLn2 : -INFINITY;
      const uint32_t ob = tmem + kColO + half * (HD / 2) + lane_addr;
      float o[HD / 2];
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) tmem_ld32(ob + c * 32, *reinterpret_cast<float(*)[32]>(o + 32 * c));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty);
      if (row_valid) {
        uint16_t* orow = static_cast<uint16_t*>(p.out) +
                         static_cast<int64_t>(t.q0 + i_loc) * p.out_ts +
                         static_cast<int64_t>(h) * p.out_hs + half * (HD / 2);
#pragma unroll
        for (int u = 0; u < HD / 16; ++u) {
          float w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = t.nkt > 0 ? o[8 * u + i] * inv : 0.f;
          *reinterpret_cast<uint4*>(orow + u * 8) = pack8<BF16>(w);
        }
      }
    }
  }
  }
  __syncthreads();
  if (tid == 0 && *s_abort) atomicOr(p.status, ATTN_DEV_TIMEOUT_FWD);
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <bool B, bool M>
auto gate_fwd_for_d(int d) {
  return d == 128 ? gate_fwd_kernel<B, M, 128> : gate_fwd_kernel<B, M, 64>;
}

cudaError_t launch_gate_fwd(const Params& p, const CUtensorMap& tq, const CUtensorMap& tqg,
                            const CUtensorMap& tk, const CUtensorMap& tkg, const CUtensorMap& tv,
                            int grid, cudaStream_t s) {
  const bool m = masked_call(p);
  auto k = p.dtype == 1 ? (m ? gate_fwd_for_d<true, true>(p.d) : gate_fwd_for_d<true, false>(p.d))
                        : (m ? gate_fwd_for_d<false, true>(p.d) : gate_fwd_for_d<false, false>(p.d));
  const uint32_t smem = p.d == 128 ? gf::smem_bytes<128>() : gf::smem_bytes<64>();
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k<<<grid, kThreads, smem, s>>>(p, tq, tqg, tk, tkg, tv);
  return cudaGetLastError();
}

}  // namespace attn

namespace attn {

// ============================================================== dq, dq_g

namespace gq {
template <int HD>
struct Lay {
  static constexpr uint32_t T = gt::Dim<HD>::kTileB;
  static constexpr uint32_t offQ = 0;
  static constexpr uint32_t offQg = offQ + T;
  static constexpr uint32_t offDO = offQg + gt::kChunkB;
  static constexpr uint32_t slotK = T + gt::kChunkB;  // K, then K_g, of one slot
  static constexpr uint32_t offK = offDO + T;
  static constexpr uint32_t offV = offK + 2 * slotK;
  static constexpr uint32_t offBar = offV + T;
};
constexpr uint32_t kColSG = 0;    // S, then (once S is read) the gate logits
constexpr uint32_t kColDP = 128;  // dP, then dS | dg pairs (32 + 32 columns per half)
constexpr uint32_t kColQ = 256;   // dQ (HD columns)
constexpr uint32_t kColQg = 384;  // dQ_g (64 columns)

struct Bars {
  uint64_t q_full, q_empty, k_full[2], k_empty[2], v_full, v_empty;
  uint64_t s_full, s_read, g_full, g_read, dp_full, p_full, acc_done;
  uint64_t o_full, o_empty, drain;
  TileRing ring;
};
template <int HD>
constexpr uint32_t smem_bytes() {
  return Lay<HD>::offBar + sizeof(Bars) + 16;
}
static_assert(smem_bytes<128>() <= 232448, "shared memory");
}  // namespace gq

// One CTA per SM, persistent; each tile is the forward's 128 query rows,
// walking every key tile they may attend to.  Per key tile: S into the SG
// region; dP (once dQ of the previous key tile has read the dS pairs); the
// gate logits into SG once S is read.  The elementwise warps form
// P = exp2(z - lse), a = P dP and b = P D, then per 16-key chunk of the gate
// logits dS = G a - b and dg = a G (1 - G), written as 16-bit pairs over the
// dP columns; dQ += dS K and dQ_g += dg K_g follow (warp 2).
template <bool BF16, bool MASK, int HD>
__global__ void __launch_bounds__(kThreads, 1)
    gate_dq_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tqg, const __grid_constant__ CUtensorMap tdo,
                   const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tkg,
                   const __grid_constant__ CUtensorMap tv) {
  using Ly = gq::Lay<HD>;
  using namespace gq;
  constexpr uint32_t T = Ly::T;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sQ = sm + Ly::offQ;
  uint8_t* sQg = sm + Ly::offQg;
  uint8_t* sDO = sm + Ly::offDO;
  uint8_t* sK = sm + Ly::offK;
  uint8_t* sV = sm + Ly::offV;
  Bars* bars = reinterpret_cast<Bars*>(sm + Ly::offBar);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_status = reinterpret_cast<int*>(s_tmem + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int ntiles = qtile_count(p);
  if (tid == 0) {
    *s_status = *reinterpret_cast<volatile int32_t*>(p.status);
    if (smem_addr(sm) & 1023u) {
      atomicOr(p.status, ATTN_DEV_SMEM_ALIGN);
      *s_status = 1;
    }
  }
  __syncthreads();
  if (*s_status != 0 || static_cast<int>(blockIdx.x) >= ntiles) return;

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->v_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_read, 8);
    mbar_init(&bars->g_full, 1);
    mbar_init(&bars->g_read, 8);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->acc_done, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 8);
    mbar_init(&bars->drain, 2);
    tile_ring_init(&bars->ring, 10);  // the two MMA threads, the 8 elementwise warps
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int G = p.G;

  if (warp < 4) {
  warpgroup_reg_dealloc<kRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // lane 0: the query tile (Q, Q_g, dO) and K + K_g; lane 1: V.  Lane 0
    // publishes the tile stream.
    if (lane == 0) {
      prefetch_tensormap(&tq);
      prefetch_tensormap(&tqg);
      prefetch_tensormap(&tdo);
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tkg);
    } else if (lane == 1) {
      prefetch_tensormap(&tv);
    }
    uint32_t g = 0;
    int tcount = 0;
    bool ok = true;
    uint32_t kpub = 0;
    int item = -1, item_next = -1;
    ok = tile_publish(&bars->ring, kpub, p.counters + 2, ntiles, &item, s_abort);
    if (ok && item >= 0)
      ok = tile_publish(&bars->ring, kpub, p.counters + 2, ntiles, &item_next, s_abort);
    for (; item >= 0 && ok; item = item_next, ++tcount,
         ok = ok && (item < 0 || tile_publish(&bars->ring, kpub, p.counters + 2, ntiles,
                                              &item_next, s_abort))) {
      QTile t;
      qtile_decode<MASK>(p, item, t);
      const int h0 = t.hg * G, tok = t.q0 + t.tok;
      if (tcount > 0 && !(ok = mbar_wait_warp(&bars->q_empty, (tcount - 1) & 1, s_abort))) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->q_full, 2 * T + gt::kChunkB);
        if (HD == 128) {
          tma_load_4d(sQ, &tq, &bars->q_full, 0, h0, tok, 0);
          tma_load_4d(sDO, &tdo, &bars->q_full, 0, h0, tok, 0);
        } else {
          tma_load_3d(sQ, &tq, &bars->q_full, 0, h0, tok);
          tma_load_3d(sDO, &tdo, &bars->q_full, 0, h0, tok);
        }
        tma_load_3d(sQg, &tqg, &bars->q_full, 0, h0, tok);
      }
      __syncwarp();
      for (int j = 0; j < t.nkt && ok; ++j, ++g) {
        const int key = t.k0 + (t.kt0 + j) * kKeys;
        const int s = g & 1;
        if (g >= 2 && !(ok = mbar_wait_warp(&bars->k_empty[s], ((g - 2) >> 1) & 1, s_abort)))
          break;
        if (lane == 0) {
          uint8_t* dst = sK + s * Ly::slotK;
          mbar_arrive_expect_tx(&bars->k_full[s], Ly::slotK);
          if (HD == 128)
            tma_load_3d(dst, &tk, &bars->k_full[s], 0, key, 0);
          else
            tma_load_2d(dst, &tk, &bars->k_full[s], 0, key);
          tma_load_2d(dst + T, &tkg, &bars->k_full[s], 0, key);
        }
        __syncwarp();
        if (g >= 1 && !(ok = mbar_wait_warp(&bars->v_empty, (g - 1) & 1, s_abort))) {
          ++g;  // the K fill above is armed
          break;
        }
        if (lane == 1) {
          mbar_arrive_expect_tx(&bars->v_full, T);
          if (HD == 128)
            tma_load_3d(sV, &tv, &bars->v_full, 0, key, 0);
          else
            tma_load_2d(sV, &tv, &bars->v_full, 0, key);
        }
        __syncwarp();
      }
    }
    if (*s_abort && lane == 0) {
      if (tcount > 0) gt::drain(&bars->q_full, (tcount - 1) & 1);
      for (uint32_t f = g > 2 ? g - 2 : 0; f < g; ++f) gt::drain(&bars->k_full[f & 1], (f >> 1) & 1);
      if (g > 0) gt::drain(&bars->v_full, (g - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S, dP, gate logits
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
      const SDesc qd = gt::kbase(smem_addr(sQ)), qgd = gt::kbase(smem_addr(sQg)),
                  dd = gt::kbase(smem_addr(sDO)), vd = gt::kbase(smem_addr(sV));
      uint32_t g = 0;
      int tcount = 0;
      bool ok = true;
      uint32_t ktake = 0;
      int item = -1;
      for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        if (!(ok = mbar_wait(&bars->q_full, tcount & 1, s_abort))) break;
        if (t.nkt == 0) {
          mbar_arrive(&bars->q_empty);
          continue;
        }
        for (int j = 0; j < t.nkt; ++j) {
          const uint32_t gs = g + j;
          if (!(ok = mbar_wait(&bars->k_full[gs & 1], (gs >> 1) & 1, s_abort))) break;
          const uint32_t kb = smem_addr(sK + (gs & 1) * Ly::slotK);
          const SDesc kd = gt::kbase(kb), kgd = gt::kbase(kb + T);
          // S into SG once the previous gate logits have been read
          if (gs >= 1 && !(ok = mbar_wait(&bars->g_read, (gs - 1) & 1, s_abort))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < HD / 16; ++k)
            umma_ss_off(tmem + kColSG, qd, gt::koff(k), kd, gt::koff(k), kIdS, k > 0);
          umma_commit(&bars->s_full);
          // dP once dQ and dQ_g of the previous key tile have read the pairs
          if (gs >= 1 && !(ok = mbar_wait(&bars->acc_done, (gs - 1) & 1, s_abort))) break;
          if (!(ok = mbar_wait(&bars->v_full, gs & 1, s_abort))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < HD / 16; ++k)
            umma_ss_off(tmem + kColDP, dd, gt::koff(k), vd, gt::koff(k), kIdS, k > 0);
          umma_commit(&bars->dp_full);
          umma_commit(&bars->v_empty);
          // the gate logits into SG once S has been read
          if (!(ok = mbar_wait(&bars->s_read, gs & 1, s_abort))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_ss_off(tmem + kColSG, qgd, gt::koff(k), kgd, gt::koff(k), kIdS, k > 0);
          umma_commit(&bars->g_full);
          if (j + 1 == t.nkt) umma_commit(&bars->q_empty);
        }
        if (!ok) break;
        g += t.nkt;
      }
      umma_commit(&bars->drain);
      gt::drain(&bars->drain, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ dQ, dQ_g
    if (lane == 0) {
      constexpr uint32_t kIdQ = idesc_f16(128, HD, BF16, false, true);
      constexpr uint32_t kIdG = idesc_f16(128, 64, BF16, false, true);
      uint32_t g = 0;
      int tcount = 0;
      bool ok = true;
      uint32_t ktake = 0;
      int item = -1;
      for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        if (t.nkt == 0) {
          if (tcount > 0 && !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort))) break;
          mbar_arrive(&bars->o_full);
          continue;
        }
        for (int j = 0; j < t.nkt; ++j) {
          const uint32_t gg = g + j;
          if (!(ok = mbar_wait(&bars->p_full, gg & 1, s_abort))) break;
          if (j == 0 && tcount > 0 &&
              !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort)))
            break;
          tc_fence_after();
          const uint32_t kb = smem_addr(sK + (gg & 1) * Ly::slotK);
          const SDesc kd = gt::mbase(kb), kgd = gt::mbase(kb + T);
          // keys 16k..16k+15: half k/4, pair column 8 (k % 4) of that half's dS
          // (dg: 32 columns further)
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k) {
            const uint32_t a = tmem + kColDP + (k >> 2) * 64 + (k & 3) * 8;
            umma_ts_off(tmem + kColQ, a, kd, gt::moff(k), kIdQ, (j > 0 || k > 0));
            umma_ts_off(tmem + kColQg, a + 32, kgd, gt::moff(k), kIdG, (j > 0 || k > 0));
          }
          umma_commit(&bars->acc_done);
          umma_commit(&bars->k_empty[gg & 1]);
          if (j + 1 == t.nkt) umma_commit(&bars->o_full);
        }
        if (!ok) break;
        g += t.nkt;
      }
      umma_commit(&bars->drain);
      gt::drain(&bars->drain, 0);
    }
  }
  } else {
  warpgroup_reg_alloc<kRegsHigh>();
  {
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;  // keys [64*half, 64*half + 64) of each key tile
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const float zscale = p.sigma * kLog2e;
    const float ghalf = 0.5f * p.gscale;
    uint32_t g = 0;
    int tcount = 0;
    bool ok = true;
    uint32_t ktake = 0;
    int item = -1;
    for (; (ok = tile_take_warp(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
      QTile t;
      qtile_decode<MASK>(p, item, t);
      const int i_loc = t.tok + r / G;
      const int h = t.hg * G + r % G;
      const bool row_valid = i_loc < t.Lq;
      const float slope2 = p.slopes ? __ldg(p.slopes + t.b * p.slopes_bs + h) * kLog2e : 0.f;
      const int pos_off = i_loc + t.Lk - t.Lq;
      float lse2 = INFINITY, Drow = 0.f;  // rows outside the sequence get P = 0
      if (row_valid) {
        const int64_t ri = static_cast<int64_t>(t.q0 + i_loc) * p.lse_rs + h;
        const float lse = p.lse[ri];
        lse2 = (lse == -INFINITY) ? INFINITY : lse * kLog2e;
        Drow = p.Dbuf[ri];
      }
      for (int j = 0; j < t.nkt; ++j) {
        const uint32_t gg = g + j;
        const int key0 = (t.kt0 + j) * kKeys + half * 64;
        const float pos0 = static_cast<float>(pos_off - key0);
        // P from S
        if (!(ok = mbar_wait_warp(&bars->s_full, gg & 1, s_abort))) break;
        tc_fence_after();
        float x[64];
        const uint32_t sgb = tmem + kColSG + half * 64 + lane_addr;
        tmem_ld32(sgb, *reinterpret_cast<float(*)[32]>(x));
        tmem_ld32(sgb + 32, *reinterpret_cast<float(*)[32]>(x + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_read);
        const bool edge =
            key0 + 64 > t.Lk ||
            (MASK && !__all_sync(0xffffffffu, !row_valid ||
                                                  all_admissible(p, t.Lq, t.Lk, i_loc, key0,
                                                                 key0 + 63)));
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float z = fmaf(x[c], zscale, fmaf(-slope2, fabsf(pos0 - static_cast<float>(c)), -lse2));
          if (edge) {
            const int jg = key0 + c;
            bool adm = jg < t.Lk;
            if (MASK) adm = adm && admissible(p, t.Lq, t.Lk, i_loc, jg);
            z = adm ? z : -INFINITY;
          }
          x[c] = ex2_approx(z);  // P
        }
        // a = P dP (over the dP values), b = P D (over P)
        if (!(ok = mbar_wait_warp(&bars->dp_full, gg & 1, s_abort))) break;
        tc_fence_after();
        float a[64];
        const uint32_t dpb = tmem + kColDP + half * 64 + lane_addr;
        tmem_ld32(dpb, *reinterpret_cast<float(*)[32]>(a));
        tmem_ld32(dpb + 32, *reinterpret_cast<float(*)[32]>(a + 32));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          a[c] *= x[c];
          x[c] *= Drow;
        }
        // gate logits, 16 keys at a time: dS = G a - b, dg = a G (1 - G),
        // both as pairs over this half's dP columns (read in full above)
        if (!(ok = mbar_wait_warp(&bars->g_full, gg & 1, s_abort))) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float gl[16];
          tmem_ld16(sgb + cc * 16, gl);
          tmem_wait_ld();
          uint32_t ds[8], dg[8];
#pragma unroll
          for (int c = 0; c < 16; c += 2) {
            const int k = cc * 16 + c;
            const float g0 = gt::gate_of(gl[c], ghalf), g1 = gt::gate_of(gl[c + 1], ghalf);
            ds[c >> 1] = Pack<BF16>::two(fmaf(g0, a[k], -x[k]), fmaf(g1, a[k + 1], -x[k + 1]));
            dg[c >> 1] =
                Pack<BF16>::two(a[k] * g0 * (1.f - g0), a[k + 1] * g1 * (1.f - g1));
          }
          tmem_st8(dpb + cc * 8, ds);
          tmem_st8(dpb + 32 + cc * 8, dg);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->g_read);
          mbar_arrive(&bars->p_full);
        }
      }
      if (!ok) break;
      g += t.nkt;
      // ---- epilogue: dq = sigma dQ (HD/2 features per half), dq_g = dQ_g / sqrt(R)
      if (!(ok = mbar_wait_warp(&bars->o_full, tcount & 1, s_abort))) break;
      tc_fence_after();
      float o[HD / 2], og[32];
      const uint32_t qa = tmem + kColQ + half * (HD / 2) + lane_addr;
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) tmem_ld32(qa + c * 32, *reinterpret_cast<float(*)[32]>(o + 32 * c));
      tmem_ld32(tmem + kColQg + half * 32 + lane_addr, og);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty);
      if (row_valid) {
        uint16_t* qrow = static_cast<uint16_t*>(p.dq) + static_cast<int64_t>(t.q0 + i_loc) * p.dq_ts +
                         static_cast<int64_t>(h) * p.dq_hs + half * (HD / 2);
#pragma unroll
        for (int u = 0; u < HD / 16; ++u) {
          float w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = t.nkt > 0 ? o[8 * u + i] * p.sigma : 0.f;
          *reinterpret_cast<uint4*>(qrow + u * 8) = pack8<BF16>(w);
        }
        uint16_t* grow = static_cast<uint16_t*>(p.dqg) +
                         static_cast<int64_t>(t.q0 + i_loc) * p.dqg_ts +
                         static_cast<int64_t>(h) * p.dqg_hs + half * 32;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = t.nkt > 0 ? og[8 * u + i] * p.gscale : 0.f;
          if (half * 32 + u * 8 < p.R) *reinterpret_cast<uint4*>(grow + u * 8) = pack8<BF16>(w);
        }
      }
    }
  }
  }
  __syncthreads();
  if (tid == 0 && *s_abort) atomicOr(p.status, ATTN_DEV_TIMEOUT_DQ);
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <bool B, bool M>
auto gate_dq_for_d(int d) {
  return d == 128 ? gate_dq_kernel<B, M, 128> : gate_dq_kernel<B, M, 64>;
}

cudaError_t launch_gate_dq(const Params& p, const CUtensorMap& tq, const CUtensorMap& tqg,
                           const CUtensorMap& tdo, const CUtensorMap& tk, const CUtensorMap& tkg,
                           const CUtensorMap& tv, int grid, cudaStream_t s) {
  const bool m = masked_call(p);
  auto k = p.dtype == 1 ? (m ? gate_dq_for_d<true, true>(p.d) : gate_dq_for_d<true, false>(p.d))
                        : (m ? gate_dq_for_d<false, true>(p.d) : gate_dq_for_d<false, false>(p.d));
  const uint32_t smem = p.d == 128 ? gq::smem_bytes<128>() : gq::smem_bytes<64>();
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k<<<grid, kThreads, smem, s>>>(p, tq, tqg, tdo, tk, tkg, tv);
  return cudaGetLastError();
}

}  // namespace attn

namespace attn {

// ============================================================== dk, dv, dk_g

namespace gk {
template <int HD>
struct Lay {
  static constexpr uint32_t T = gt::Dim<HD>::kTileB;
  static constexpr uint32_t offK = 0;
  static constexpr uint32_t offV = offK + T;
  static constexpr uint32_t offKg = offV + T;
  static constexpr uint32_t slotQ = T + gt::kChunkB;  // Q, then Q_g, of one slot
  static constexpr uint32_t offQ = offKg + gt::kChunkB;
  static constexpr uint32_t offDO = offQ + 2 * slotQ;
  static constexpr uint32_t offCol = offDO + T;
  // TMEM: dV, dK, dK_g accumulators, then SP (S^T, gate logits^T, dP^T in
  // turn) and X (W^T, dS^T, dg^T pairs in turn)
  static constexpr uint32_t colDV = 0, colDK = HD, colDKg = 2 * HD;
  static constexpr uint32_t colSP = 2 * HD + 64, colX = 2 * HD + 192;
};

struct Cols {       // per-column scalars of a query step (column = token * G + head)
  float a[2][128];  // base-2 bias at key r = a + m * r (one-sided steps), lse included
  float m[2][128];
  float D[128];
  int general[2][2];
};

struct Bars {
  uint64_t kv_full, kv_empty, q_full[2], q_empty[2], do_full, do_empty;
  uint64_t s_full, s_read, gl_full, gl_read, dp_full;
  uint64_t w_full, dv_done, ds_full, dk_done, dg_full, dkg_done;
  uint64_t acc_full, acc_empty, am_full[2], am_empty[2], d_full, d_empty, drain;
  TileRing ring;
};
template <int HD>
constexpr uint32_t smem_bytes() {
  return Lay<HD>::offCol + sizeof(Cols) + sizeof(Bars) + 16;
}
static_assert(smem_bytes<128>() <= 232448, "shared memory");
}  // namespace gk

// One CTA owns 128 keys of one sequence (and one K/V head group) and walks
// every query step (the forward's 128-row query tile) that may attend to
// them in a fixed order, so dV, dK and dK_g accumulate in TMEM with no
// atomics.  Per step: S^T, then the gate logits^T, then dP^T pass through SP
// (warp 1); the elementwise warps form P^T from S^T and the staged per-column
// bias (which holds -lse), W^T = P^T G^T into X for dV += W^T dO, then, 16
// columns of dP^T at a time (with W^T read back from X),
// dg^T = W^T dP^T (1 - G^T) as pairs over the SP columns just read, for
// dK_g += dg^T Q_g, and dS^T = W^T dP^T - P^T D, written over X once dV is
// done, for dK += dS^T Q (warp 3).  S^T of the next step follows dK_g into
// SP.  Warp 2 stages the per-column scalars.
template <bool BF16, bool MASK, int HD>
__global__ void __launch_bounds__(kThreads, 1)
    gate_dkdv_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq,
                     const __grid_constant__ CUtensorMap tqg,
                     const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk,
                     const __grid_constant__ CUtensorMap tkg,
                     const __grid_constant__ CUtensorMap tv) {
  using Ly = gk::Lay<HD>;
  using namespace gk;
  constexpr uint32_t T = Ly::T;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sK = sm + Ly::offK;
  uint8_t* sV = sm + Ly::offV;
  uint8_t* sKg = sm + Ly::offKg;
  uint8_t* sQ = sm + Ly::offQ;
  uint8_t* sDO = sm + Ly::offDO;
  Cols* cols = reinterpret_cast<Cols*>(sm + Ly::offCol);
  Bars* bars = reinterpret_cast<Bars*>(cols + 1);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* s_status = reinterpret_cast<int*>(s_tmem + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int ntiles = ktile_count(p);
  if (tid == 0) {
    *s_status = *reinterpret_cast<volatile int32_t*>(p.status);
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
      mbar_init(&bars->am_full[s], 1);
      mbar_init(&bars->am_empty[s], 8);
    }
    mbar_init(&bars->do_full, 1);
    mbar_init(&bars->do_empty, 2);  // read by dP^T (warp 1) and dV (warp 3)
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_read, 8);
    mbar_init(&bars->gl_full, 1);
    mbar_init(&bars->gl_read, 8);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->w_full, 8);
    mbar_init(&bars->dv_done, 1);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->dg_full, 8);
    mbar_init(&bars->dkg_done, 1);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->d_full, 1);
    mbar_init(&bars->d_empty, 8);
    mbar_init(&bars->drain, 2);
    // readers: the two MMA threads, the staging warp, the 8 elementwise warps
    tile_ring_init(&bars->ring, 11);
    fence_barrier_init();
    *s_abort = 0;
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int G = p.G;
  const int step_tok = kRowsQ / G;
  const int ngroups = p.Hq / G;
  auto step_count = [&](const KTile& t) { return t.ntb * ngroups; };

  if (warp < 4) {
  warpgroup_reg_dealloc<kRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // lanes 0-2: K, K_g, V of a key tile; then per query step Q (lane 0),
    // Q_g (lane 1) into slot g & 1 and dO (lane 2).  The warp publishes the
    // tile stream one tile ahead.
    if (lane == 0) {
      prefetch_tensormap(&tk);
      prefetch_tensormap(&tq);
    } else if (lane == 1) {
      prefetch_tensormap(&tkg);
      prefetch_tensormap(&tqg);
    } else if (lane == 2) {
      prefetch_tensormap(&tv);
      prefetch_tensormap(&tdo);
    }
    uint32_t nkv = 0, nq0 = 0, nq1 = 0, ndo = 0;
    bool ok = true;
    uint32_t kpub = 0;
    int item = -1, item_next = -1;
    ok = tile_publish(&bars->ring, kpub, p.counters + 1, ntiles, &item, s_abort);
    if (ok && item >= 0)
      ok = tile_publish(&bars->ring, kpub, p.counters + 1, ntiles, &item_next, s_abort);
    for (; item >= 0 && ok; item = item_next,
         ok = ok && (item < 0 || tile_publish(&bars->ring, kpub, p.counters + 1, ntiles,
                                              &item_next, s_abort))) {
      KTile t;
      ktile_decode<MASK>(p, item, t);
      const int nsteps = step_count(t);
      const int key = t.k0 + t.key;
      if (nkv > 0 && !(ok = mbar_wait_warp(&bars->kv_empty, (nkv - 1) & 1, s_abort))) break;
      if (lane == 0) mbar_arrive_expect_tx(&bars->kv_full, 2 * T + gt::kChunkB);
      __syncwarp();
      if (lane == 0) {
        if (HD == 128)
          tma_load_3d(sK, &tk, &bars->kv_full, 0, key, 0);
        else
          tma_load_2d(sK, &tk, &bars->kv_full, 0, key);
      } else if (lane == 1) {
        tma_load_2d(sKg, &tkg, &bars->kv_full, 0, key);
      } else if (lane == 2) {
        if (HD == 128)
          tma_load_3d(sV, &tv, &bars->kv_full, 0, key, 0);
        else
          tma_load_2d(sV, &tv, &bars->kv_full, 0, key);
      }
      ++nkv;
      int stb = t.tb0, shg = 0;
      for (int st = 0; st < nsteps; ++st, ++ndo) {
        const int tok = t.q0 + stb * step_tok;
        const int h0 = shg * G;
        if (++shg == ngroups) {
          shg = 0;
          ++stb;
        }
        const int s = (nq0 + nq1) & 1;
        const uint32_t n = s ? nq1++ : nq0++;
        if (n > 0 && !(ok = mbar_wait_warp(&bars->q_empty[s], (n - 1) & 1, s_abort))) break;
        if (lane == 0) mbar_arrive_expect_tx(&bars->q_full[s], Ly::slotQ);
        __syncwarp();
        uint8_t* dq = sQ + s * Ly::slotQ;
        if (lane == 0) {
          if (HD == 128)
            tma_load_4d(dq, &tq, &bars->q_full[s], 0, h0, tok, 0);
          else
            tma_load_3d(dq, &tq, &bars->q_full[s], 0, h0, tok);
        } else if (lane == 1) {
          tma_load_3d(dq + T, &tqg, &bars->q_full[s], 0, h0, tok);
        }
        if (ndo > 0 && !(ok = mbar_wait_warp(&bars->do_empty, (ndo - 1) & 1, s_abort))) break;
        if (lane == 0) mbar_arrive_expect_tx(&bars->do_full, T);
        __syncwarp();
        if (lane == 2) {
          if (HD == 128)
            tma_load_4d(sDO, &tdo, &bars->do_full, 0, h0, tok, 0);
          else
            tma_load_3d(sDO, &tdo, &bars->do_full, 0, h0, tok);
        }
      }
    }
    if (*s_abort && lane == 0) {
      if (nkv > 0) gt::drain(&bars->kv_full, (nkv - 1) & 1);
      if (nq0 > 0) gt::drain(&bars->q_full[0], (nq0 - 1) & 1);
      if (nq1 > 0) gt::drain(&bars->q_full[1], (nq1 - 1) & 1);
      if (ndo > 0) gt::drain(&bars->do_full, (ndo - 1) & 1);
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t kIdD = idesc_f16(128, HD, BF16, false, true);
      constexpr uint32_t kIdG = idesc_f16(128, 64, BF16, false, true);
      const SDesc kd = gt::kbase(smem_addr(sK)), vd = gt::kbase(smem_addr(sV)),
                  kgd = gt::kbase(smem_addr(sKg)), dkd = gt::kbase(smem_addr(sDO)),
                  dmd = gt::mbase(smem_addr(sDO));
      const uint32_t qb0 = smem_addr(sQ);
      auto qslot = [&](uint32_t gg) { return qb0 + (gg & 1) * Ly::slotQ; };
      uint32_t g = 0;
      int tcount = 0;
      bool ok = true;
      uint32_t ktake = 0;
      int item = -1;
      if (warp == 1) {
        // S^T, gate logits^T and dP^T through SP (dK_g of the step before
        // reads its dg^T pairs from SP)
        auto issue_s = [&](uint32_t gg) -> bool {
          if (gg >= 1 && !mbar_wait(&bars->dkg_done, (gg - 1) & 1, s_abort)) return false;
          if (!mbar_wait(&bars->q_full[gg & 1], (gg >> 1) & 1, s_abort)) return false;
          tc_fence_after();
          const SDesc qd = gt::kbase(qslot(gg));
#pragma unroll
          for (int k = 0; k < HD / 16; ++k)
            umma_ss_off(tmem + Ly::colSP, kd, gt::koff(k), qd, gt::koff(k), kIdS, k > 0);
          umma_commit(&bars->s_full);
          return true;
        };
        for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
          KTile t;
          ktile_decode<MASK>(p, item, t);
          const int nsteps = step_count(t);
          if (!(ok = mbar_wait(&bars->kv_full, tcount & 1, s_abort))) break;
          if (nsteps == 0) {
            mbar_arrive(&bars->kv_empty);
            continue;
          }
          if (!(ok = issue_s(g))) break;
          for (int st = 0; st < nsteps && ok; ++st) {
            const uint32_t gg = g + st;
            // gate logits^T once S^T has been read
            if (!(ok = mbar_wait(&bars->s_read, gg & 1, s_abort))) break;
            tc_fence_after();
            const SDesc qgd = gt::kbase(qslot(gg) + T);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_ss_off(tmem + Ly::colSP, kgd, gt::koff(k), qgd, gt::koff(k), kIdS, k > 0);
            umma_commit(&bars->gl_full);
            // dP^T once the gate logits have been read
            if (!(ok = mbar_wait(&bars->gl_read, gg & 1, s_abort))) break;
            if (!(ok = mbar_wait(&bars->do_full, gg & 1, s_abort))) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < HD / 16; ++k)
              umma_ss_off(tmem + Ly::colSP, vd, gt::koff(k), dkd, gt::koff(k), kIdS, k > 0);
            umma_commit(&bars->dp_full);
            umma_commit(&bars->do_empty);
            if (st + 1 < nsteps && !(ok = issue_s(gg + 1))) break;
          }
          if (!ok) break;
          umma_commit(&bars->kv_empty);  // K, V and K_g are read by this thread's MMAs only
          g += nsteps;
        }
      } else {
        // dV += W^T dO and dK += dS^T Q (A operands: pairs in X, query rows
        // 16k.. at column 32 (k / 4) + 8 (k % 4)), dK_g += dg^T Q_g (pairs in
        // SP at column 64 (k / 4) + 16 (k % 4))
        auto mma_x = [&](uint32_t d, SDesc b, uint32_t id, bool acc) {
#pragma unroll
          for (int k = 0; k < kRowsQ / 16; ++k)
            umma_ts_off(d, tmem + Ly::colX + (k >> 2) * 32 + (k & 3) * 8, b, gt::moff(k), id,
                        (acc || k > 0) ? 1u : 0u);
        };
        auto mma_sp = [&](uint32_t d, SDesc b, uint32_t id, bool acc) {
#pragma unroll
          for (int k = 0; k < kRowsQ / 16; ++k)
            umma_ts_off(d, tmem + Ly::colSP + (k >> 2) * 64 + (k & 3) * 16, b, gt::moff(k), id,
                        (acc || k > 0) ? 1u : 0u);
        };
        for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
          KTile t;
          ktile_decode<MASK>(p, item, t);
          const int nsteps = step_count(t);
          if (nsteps == 0) {
            if (tcount > 0 && !(ok = mbar_wait(&bars->acc_empty, (tcount - 1) & 1, s_abort)))
              break;
            mbar_arrive(&bars->acc_full);
            continue;
          }
          for (int st = 0; st < nsteps && ok; ++st) {
            const uint32_t gg = g + st;
            if (!(ok = mbar_wait(&bars->w_full, gg & 1, s_abort))) break;
            if (!(ok = mbar_wait(&bars->do_full, gg & 1, s_abort))) break;
            if (st == 0 && tcount > 0 &&
                !(ok = mbar_wait(&bars->acc_empty, (tcount - 1) & 1, s_abort)))
              break;
            tc_fence_after();
            mma_x(tmem + Ly::colDV, dmd, kIdD, st > 0);
            umma_commit(&bars->dv_done);
            umma_commit(&bars->do_empty);
            if (!(ok = mbar_wait(&bars->dg_full, gg & 1, s_abort))) break;
            tc_fence_after();
            mma_sp(tmem + Ly::colDKg, gt::mbase(qslot(gg) + T), kIdG, st > 0);
            umma_commit(&bars->dkg_done);
            if (!(ok = mbar_wait(&bars->ds_full, gg & 1, s_abort))) break;
            tc_fence_after();
            mma_x(tmem + Ly::colDK, gt::mbase(qslot(gg)), kIdD, st > 0);
            umma_commit(&bars->dk_done);
            umma_commit(&bars->q_empty[gg & 1]);
          }
          if (!ok) break;
          umma_commit(&bars->acc_full);
          g += nsteps;
        }
      }
      umma_commit(&bars->drain);
      gt::drain(&bars->drain, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ column scalars
    // Lane u stages columns u, u + 32, u + 64, u + 96 of every query step:
    // the base-2 bias line (-slope2 |i + Lk - Lq - j| - lse2 = a + m j on
    // steps that lie on one side of every column's aligned key) into a
    // two-deep ring, D into one buffer; global loads run two steps ahead.
    const int u = lane;
    const int lgGs = __ffs(G) - 1;
    struct Pos {
      int item, st, tb, hg, nsteps;
      KTile t;
    };
    struct Vals {
      float lse[4], sl2[4], D[4];
    };
    uint32_t ktake = 0;
    bool sok = true;
    auto take = [&]() -> int {
      int it = -1;
      if (sok) sok = tile_take_warp(&bars->ring, ktake, &it, s_abort);
      return (sok && it >= 0) ? it : ntiles;
    };
    auto seek = [&](Pos& q) {
      while (q.item < ntiles) {
        ktile_decode<MASK>(p, q.item, q.t);
        q.nsteps = step_count(q.t);
        q.tb = q.t.tb0;
        if (q.nsteps > 0) return;
        q.item = take();
      }
    };
    auto next = [&](const Pos& q) {
      Pos n = q;
      if (q.item >= ntiles) return n;
      if (++n.st < n.nsteps) {
        if (++n.hg == ngroups) {
          n.hg = 0;
          ++n.tb;
        }
        return n;
      }
      n.item = take();
      n.st = n.tb = n.hg = 0;
      seek(n);
      return n;
    };
    auto fetch = [&](const Pos& q, Vals& v) {
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const int lc = u + 32 * hh;
        const int i = q.tb * step_tok + (lc >> lgGs);
        const int h = q.hg * G + (lc & (G - 1));
        const bool live = q.item < ntiles;
        const bool valid = live && i < q.t.Lq;
        const int64_t ri = static_cast<int64_t>(q.t.q0 + i) * p.lse_rs + h;
        v.lse[hh] = valid ? __ldg(p.lse + ri) : -INFINITY;
        v.sl2[hh] = (live && p.slopes) ? __ldg(p.slopes + q.t.b * p.slopes_bs + h) : 0.f;
        v.D[hh] = valid ? __ldg(p.Dbuf + ri) : 0.f;
      }
    };
    Pos q0;
    q0.item = take();
    q0.st = q0.tb = q0.hg = 0;
    q0.t = KTile{};
    seek(q0);
    Pos q1 = next(q0);
    Vals v0, v1;
    fetch(q0, v0);
    fetch(q1, v1);
    bool ok = true;
    for (uint32_t gg = 0; q0.item < ntiles; ++gg) {
      const Pos q2 = next(q1);
      Vals v2;
      fetch(q2, v2);
      const int b = gg & 1;
      if (gg >= 2 && !(ok = mbar_wait_warp(&bars->am_empty[b], ((gg - 2) >> 1) & 1, s_abort)))
        break;
      bool straddle = false;
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        const int lc = u + 32 * hh;
        const int i = q0.tb * step_tok + (lc >> lgGs);
        const float nl2 = v0.lse[hh] == -INFINITY ? -INFINITY : -v0.lse[hh] * kLog2e;
        const float sl2 = v0.sl2[hh] * kLog2e;
        const float prel = static_cast<float>(i + q0.t.Lk - q0.t.Lq - q0.t.key);
        const bool right = prel <= 0.f;
        const float m = right ? -sl2 : sl2;
        cols->a[b][lc] = fmaf(-m, prel, nl2);
        cols->m[b][lc] = m;
        straddle |= !right && prel < static_cast<float>(kKeys - 1) && i < q0.t.Lq;
        if (MASK && i < q0.t.Lq)
          straddle |= !all_admissible(p, q0.t.Lq, q0.t.Lk, i, q0.t.key,
                                      min(q0.t.key + kKeys, q0.t.Lk) - 1);
      }
      const bool gen = __any_sync(0xffffffffu, straddle);
      if (lane == 0) {
        cols->general[b][0] = gen ? 1 : 0;
        cols->general[b][1] = 0;
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->am_full[b]);
      if (gg >= 1 && !(ok = mbar_wait_warp(&bars->d_empty, (gg - 1) & 1, s_abort))) break;
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) cols->D[u + 32 * hh] = v0.D[hh];
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->d_full);
      q0 = q1;
      v0 = v1;
      q1 = q2;
      v1 = v2;
    }
  }
  } else {
  warpgroup_reg_alloc<kRegsHigh>();
  {
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;  // query columns [64*half, 64*half + 64)
    const int r = quad * 32 + lane;    // key within the tile (TMEM lane)
    const float rf = static_cast<float>(r);
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const float zscale = p.sigma * kLog2e;
    const float ghalf = 0.5f * p.gscale;
    const int wl = p.wl;
    const int wr = right_window(p);
    const int lgG = __ffs(G) - 1;
    const uint32_t spbuf = tmem + Ly::colSP + half * 64 + lane_addr;
    const uint32_t xbuf = tmem + Ly::colX + half * 32 + lane_addr;
    uint32_t g = 0;
    int tcount = 0;
    bool ok = true;
    uint32_t ktake = 0;
    int item = -1;
    for (; (ok = tile_take_warp(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
      KTile t;
      ktile_decode<MASK>(p, item, t);
      const int nsteps = step_count(t);
      for (int st = 0; st < nsteps; ++st) {
        const uint32_t gg = g + st;
        const int b = gg & 1;
        // ---- P^T from S^T and the staged bias
        if (!(ok = mbar_wait_warp(&bars->s_full, gg & 1, s_abort))) break;
        tc_fence_after();
        float x[64];
        tmem_ld32(spbuf, *reinterpret_cast<float(*)[32]>(x));
        tmem_ld32(spbuf + 32, *reinterpret_cast<float(*)[32]>(x + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_read);
        if (!(ok = mbar_wait_warp(&bars->am_full[b], (gg >> 1) & 1, s_abort))) break;
        const float4* pa = reinterpret_cast<const float4*>(cols->a[b] + half * 64);
        const float4* pm = reinterpret_cast<const float4*>(cols->m[b] + half * 64);
        if ((cols->general[b][0] | cols->general[b][1]) == 0) {
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const float4 a4 = pa[q4], m4 = pm[q4];
            x[4 * q4] = ex2_approx(fmaf(x[4 * q4], zscale, fmaf(m4.x, rf, a4.x)));
            x[4 * q4 + 1] = ex2_approx(fmaf(x[4 * q4 + 1], zscale, fmaf(m4.y, rf, a4.y)));
            x[4 * q4 + 2] = ex2_approx(fmaf(x[4 * q4 + 2], zscale, fmaf(m4.z, rf, a4.z)));
            x[4 * q4 + 3] = ex2_approx(fmaf(x[4 * q4 + 3], zscale, fmaf(m4.w, rf, a4.w)));
          }
        } else {
          // some column's aligned key lies inside the tile, or a mask applies
          const int tok0 = (t.tb0 + st / ngroups) * step_tok;
          const int off = t.Lk - t.Lq - t.key;
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const float4 a4 = pa[q4], m4 = pm[q4];
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int c = half * 64 + q4 * 4 + v;
              const float prel = static_cast<float>(tok0 + (c >> lgG) + off);
              const float sl = prel <= 0.f ? -mv[v] : mv[v];
              float bv = fmaf(-sl, fabsf(prel - rf), fmaf(mv[v], prel, av[v]));
              if (MASK) {
                const bool adm = (wl < 0 || rf >= prel - static_cast<float>(wl)) &&
                                 (wr < 0 || rf <= prel + static_cast<float>(wr));
                bv = adm ? bv : -INFINITY;
              }
              x[4 * q4 + v] = ex2_approx(fmaf(x[4 * q4 + v], zscale, bv));
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->am_empty[b]);
        // ---- gate: W^T = P^T G^T (pairs), P D and 1 - G kept for dS and dg
        if (!(ok = mbar_wait_warp(&bars->d_full, gg & 1, s_abort))) break;
        if (!(ok = mbar_wait_warp(&bars->gl_full, gg & 1, s_abort))) break;
        tc_fence_after();
        uint32_t wpk[32], omg[32], pdp[32];  // W, 1 - G, P D as 16-bit pairs
        {
          const float4* pd = reinterpret_cast<const float4*>(cols->D + half * 64);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            float gl[16];
            tmem_ld16(spbuf + cc * 16, gl);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; c += 4) {
              const int k = cc * 16 + c;
              const float4 d4 = pd[k >> 2];
              const float g0 = gt::gate_of(gl[c], ghalf), g1 = gt::gate_of(gl[c + 1], ghalf);
              const float g2 = gt::gate_of(gl[c + 2], ghalf), g3 = gt::gate_of(gl[c + 3], ghalf);
              wpk[k >> 1] = Pack<BF16>::two(x[k] * g0, x[k + 1] * g1);
              wpk[(k >> 1) + 1] = Pack<BF16>::two(x[k + 2] * g2, x[k + 3] * g3);
              omg[k >> 1] = Pack<BF16>::two(1.f - g0, 1.f - g1);
              omg[(k >> 1) + 1] = Pack<BF16>::two(1.f - g2, 1.f - g3);
              pdp[k >> 1] = Pack<BF16>::two(x[k] * d4.x, x[k + 1] * d4.y);
              pdp[(k >> 1) + 1] = Pack<BF16>::two(x[k + 2] * d4.z, x[k + 3] * d4.w);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->gl_read);
          mbar_arrive(&bars->d_empty);
        }
        // W^T into X once dK of the previous step has read it
        if (gg >= 1 && !(ok = mbar_wait_warp(&bars->dk_done, (gg - 1) & 1, s_abort))) break;
        tc_fence_after();
        tmem_st16(xbuf, *reinterpret_cast<uint32_t(*)[16]>(wpk));
        tmem_st16(xbuf + 16, *reinterpret_cast<uint32_t(*)[16]>(wpk + 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->w_full);
        // ---- 16 columns of dP^T at a time: dg^T = W^T dP^T (1 - G^T) as
        // pairs over the columns just read, dS^T = W^T dP^T - P^T D kept
        if (!(ok = mbar_wait_warp(&bars->dp_full, gg & 1, s_abort))) break;
        tc_fence_after();
        uint32_t dsp[32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          float dp[16];
          uint32_t wv[8], dgp[8];
          tmem_ld16(spbuf + cc * 16, dp);
          tmem_ld8(xbuf + cc * 8, wv);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 16; c += 2) {
            const int k = cc * 16 + c;
            const uint64_t w2 = Pack<BF16>::unpack(wv[c >> 1]);
            const uint64_t o2 = Pack<BF16>::unpack(omg[k >> 1]);
            const uint64_t wdp = f2_mul(w2, f2_make(dp[c], dp[c + 1]));
            const uint64_t ds = f2_fma(Pack<BF16>::unpack(pdp[k >> 1]), f2_make(-1.f, -1.f), wdp);
            const uint64_t dg = f2_mul(wdp, o2);
            dsp[k >> 1] = Pack<BF16>::two(f2_lo(ds), f2_hi(ds));
            dgp[c >> 1] = Pack<BF16>::two(f2_lo(dg), f2_hi(dg));
          }
          tmem_st8(spbuf + cc * 16, dgp);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dg_full);
        // dS^T over X once dV has read W^T
        if (!(ok = mbar_wait_warp(&bars->dv_done, gg & 1, s_abort))) break;
        tc_fence_after();
        tmem_st16(xbuf, *reinterpret_cast<uint32_t(*)[16]>(dsp));
        tmem_st16(xbuf + 16, *reinterpret_cast<uint32_t(*)[16]>(dsp + 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->ds_full);
      }
      if (!ok) break;
      g += nsteps;
      // ---- epilogue: half 0 writes dv and dk_g, half 1 dk = sigma dK
      if (!(ok = mbar_wait_warp(&bars->acc_full, tcount & 1, s_abort))) break;
      tc_fence_after();
      const int j = t.key + r;
      const bool key_valid = j < t.Lk;
      const int64_t krow = t.k0 + j;
      if (half == 0) {
        uint16_t* row = static_cast<uint16_t*>(p.dv) + krow * p.dv_ts;
        uint16_t* grow = static_cast<uint16_t*>(p.dkg) + krow * p.dkg_ts;
#pragma unroll 1
        for (int c = 0; c < HD / 32 + 2; ++c) {
          const bool gate_part = c >= HD / 32;
          const int cg = c - HD / 32;
          float a[32];
          tmem_ld32(tmem + (gate_part ? Ly::colDKg + cg * 32 : Ly::colDV + c * 32) + lane_addr, a);
          tmem_wait_ld();
          if (key_valid) {
            const float sc = gate_part ? p.gscale : 1.f;
            uint16_t* dst = gate_part ? grow + cg * 32 : row + c * 32;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float w8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) w8[i] = nsteps > 0 ? a[8 * v + i] * sc : 0.f;
              if (!gate_part || cg * 32 + v * 8 < p.R)
                *reinterpret_cast<uint4*>(dst + v * 8) = pack8<BF16>(w8);
            }
          }
        }
      } else {
        uint16_t* row = static_cast<uint16_t*>(p.dk) + krow * p.dk_ts;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          float a[32];
          tmem_ld32(tmem + Ly::colDK + c * 32 + lane_addr, a);
          tmem_wait_ld();
          if (key_valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              float w8[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) w8[i] = nsteps > 0 ? a[8 * v + i] * p.sigma : 0.f;
              *reinterpret_cast<uint4*>(row + c * 32 + v * 8) = pack8<BF16>(w8);
            }
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
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <bool B, bool M>
auto gate_dkdv_for_d(int d) {
  return d == 128 ? gate_dkdv_kernel<B, M, 128> : gate_dkdv_kernel<B, M, 64>;
}

cudaError_t launch_gate_dkdv(const Params& p, const CUtensorMap& tq, const CUtensorMap& tqg,
                             const CUtensorMap& tdo, const CUtensorMap& tk, const CUtensorMap& tkg,
                             const CUtensorMap& tv, int grid, cudaStream_t s) {
  const bool m = masked_call(p);
  auto k = p.dtype == 1
               ? (m ? gate_dkdv_for_d<true, true>(p.d) : gate_dkdv_for_d<true, false>(p.d))
               : (m ? gate_dkdv_for_d<false, true>(p.d) : gate_dkdv_for_d<false, false>(p.d));
  const uint32_t smem = p.d == 128 ? gk::smem_bytes<128>() : gk::smem_bytes<64>();
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  k<<<grid, kThreads, smem, s>>>(p, tq, tqg, tdo, tk, tkg, tv);
  return cudaGetLastError();
}

}  // namespace attn
