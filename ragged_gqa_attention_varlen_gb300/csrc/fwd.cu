// fwd.cu -- forward pass: out and lse for every query row.
//
// "Noncausal Global Extreme-GQA Ragged Attention Full VJP" ("What You Have"):
// scaled logits, 3*tanh(s/3) softcap, ALiBi -slope*|i + Lk - Lq - j|, softmax,
// out = P V.  The softmax is the online (running max / running sum) form of
// "ragged flash attention gradient recompute" ("Root causes addressed"):
// only O and L = m + log l are stored.
//
// Tile: 128 query rows = (128/G tokens) x (G heads of one head group); all
// heads of the call (of one K/V head group) share one K/V head, so every row
// of a tile reads the same 128-key K and V tiles.  Per key tile j:
//   S_j = Q K_j^T         tcgen05.mma (Q, K from shared memory), fp32 in TMEM
//   P_j = exp2(z - m)     softmax warps, one thread per row (TMEM lane); P_j
//                         goes to its own TMEM region as 16-bit pairs
//   O  += P_j V_j         tcgen05.mma with P_j read from TMEM
//
// Warp roles (384 threads, 12 warps): warp 0 issues TMA loads (lane 0: Q once per tile
// and K through two slots; lane 1: V through two slots, so a K load never
// waits for a V slot), warp 1 issues the S products and warp 2 the P V
// products (two issuing threads: an MMA issue blocks while the tensor pipe is
// busy, so one thread could not wait for P_j while S_{j+1} is queued), warps 4-11 run the
// softmax and the epilogue -- two warps per TMEM lane quadrant, each taking
// 64 of the 128 keys of a tile (the row max is exchanged through shared
// memory), so every SM sub-partition has two warps to hide MUFU latency.  S
// is double-buffered in TMEM so the tensor core computes S_{j+1} while the
// softmax works on S_j.
//
// Q and K are only K-major operands here and keep features 128..159 in a
// 64-byte-swizzled chunk; V is the MN-major operand of P V and stays in three
// 128-byte-swizzled chunks.
//
// With the softcap (c <= 9.5) P is taken against a per-row reference fixed
// before the first key tile (see row_bound), so the softmax needs no running
// max.  Otherwise (no cap, or a larger one):
// key tiles are visited starting with the one that holds the ALiBi peak of
// the tile's rows (the key aligned with the query, where the distance is 0),
// so the running max is (nearly) final after the first tile.  O is rescaled
// only when a row's max grows by more than 8 (base-2 units); until then P is
// taken relative to the stale max and stays below 2^8.  With the softcap
// (|t| <= c) and ALiBi (<= 0) no later tile can exceed the first tile's max
// by more than 2*c*log2(e) = 8.66, so rescales are rare.
// Warp 3 draws the query tiles from a global counter for the whole CTA
// (see TileRing).  Warpgroup 0 hands most of its registers to
// the elementwise warpgroups (setmaxnreg), so those can keep every column's
// MUFU/FMA chain of a batch in flight.
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace fwd {
constexpr int kThreadsF = kThreads;  // 12 warps
constexpr uint32_t kTile = 16384;        // one 64-feature chunk of a 128-row tile
constexpr uint32_t kTail = 8192;         // features 128..159 of 128 rows (64-byte rows)
constexpr uint32_t kTailed = 2 * kTile + kTail;
constexpr uint32_t kTile3 = 3 * kTile;   // a whole 128 x 160 tile in 128-byte rows
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kTailed;      // two K slots
constexpr uint32_t kOffV = kOffK + 2 * kTailed;  // two V slots
constexpr uint32_t kOffMax = kOffV + 2 * kTile3;  // [2 steps][2 halves][128] fp32
constexpr uint32_t kOffSum = kOffMax + 2 * 2 * 128 * 4;     // [2 tiles][2 halves][128] fp32
constexpr uint32_t kOffBar = kOffSum + 2 * 2 * 128 * 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColP = 256;          // S0: [0,128), S1: [128,256), P: [256,320)
constexpr uint32_t kColO = 320;          // O: [320, 480)
constexpr float kRescale = 8.f;          // lazy-rescale threshold (base 2)

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], s_read[2], p_full[2], pv_done;
  uint64_t o_full, o_empty, drain;
  uint64_t mx_x[2], l_x[2];  // row-max and row-sum exchanges between the halves
  TileRing ring;             // query tiles drawn by warp 3 for the whole CTA
};
// barriers, then the TMEM base address, the abort flag and the status copy
constexpr uint32_t kSmem = kOffBar + sizeof(Bars) + 16;  // base checked to be 1024-aligned
static_assert(kSmem <= 232448, "shared memory");
}  // namespace fwd

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

// Largest softcap that takes the fixed-reference softmax: P = 2^(z - ref)
// with ref = the row's ALiBi term at its admissible key nearest to (slope
// >= 0) or farthest from (slope < 0) the aligned key.  Every logit of the
// row is then at most c*log2(e) above ref and the largest at least that far
// below it, so P stays within [2^-14, 2^14] for the row maximum and below
// 2^14 everywhere: inside the normal range of fp16 and bf16.
constexpr float kFixedCapMax = 9.5f;

// The fixed reference of a row whose aligned key is k0 (base 2).  A row with
// no admissible key gets 0 (every P is then exp2(-inf) = 0).
template <bool MASK>
__device__ __forceinline__ float row_bound(const Params& p, int Lk, int k0, float slope2) {
  int64_t lo = 0, hi = static_cast<int64_t>(Lk) - 1;
  if (MASK) {
    const int wr = right_window(p);
    if (p.wl >= 0) lo = max(lo, static_cast<int64_t>(k0) - p.wl);
    if (wr >= 0) hi = min(hi, static_cast<int64_t>(k0) + wr);
  }
  if (lo > hi) return 0.f;
  int64_t d;
  if (slope2 >= 0.f)
    d = k0 < lo ? lo - k0 : (k0 > hi ? k0 - hi : 0);
  else
    d = max(k0 - lo, hi - k0);
  return -slope2 * static_cast<float>(d);
}

// The key tiles a query tile visits: the n tiles from t.kt0 on (those that
// hold a key some query of the tile may attend to), starting at t0, the tile
// of the key aligned with the tile's first query, and wrapping.
__device__ __forceinline__ void key_order(const QTile& t, int& n, int& t0) {
  n = t.nkt;
  int k0 = t.tok + t.Lk - t.Lq;  // key aligned with the tile's first query
  k0 = k0 < 0 ? 0 : (k0 >= t.Lk ? t.Lk - 1 : k0);
  t0 = n > 0 ? min(max(k0 / kKeys, t.kt0), t.kt0 + n - 1) : 0;
}

// The key tile after kt in the walk of a query tile.
__device__ __forceinline__ int next_key_tile(const QTile& t, int kt) {
  return kt + 1 == t.kt0 + t.nkt ? t.kt0 : kt + 1;
}

// HD: the head dimension (160, 128 or 64) -- the MMA shapes and the stores
// follow it; the shared-memory and TMEM layouts are those of 160 features.
// FIXED: the call takes the fixed-reference softmax (a softcap of at most
// kFixedCapMax) -- instances per path, so each holds only its own code.
template <bool BF16, bool MASK, int HD, bool DROP, bool FIXED>
__global__ void __launch_bounds__(fwd::kThreadsF, 1)
    fwd_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq2,
               const __grid_constant__ CUtensorMap tqt, const __grid_constant__ CUtensorMap tk2,
               const __grid_constant__ CUtensorMap tkt, const __grid_constant__ CUtensorMap tv2,
               const __grid_constant__ CUtensorMap tv) {
  using namespace fwd;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sQ = sm + kOffQ;
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
  float* sMax = reinterpret_cast<float*>(sm + kOffMax);
  float* sSum = reinterpret_cast<float*>(sm + kOffSum);
  Bars* bars = reinterpret_cast<Bars*>(sm + kOffBar);
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
  if (*s_status != 0 || static_cast<int>(blockIdx.x) >= ntiles) return;  // uniform

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->k_full[b], 1);
      mbar_init(&bars->k_empty[b], 1);
      mbar_init(&bars->v_full[b], 1);
      mbar_init(&bars->v_empty[b], 1);
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_read[b], 8);
      mbar_init(&bars->p_full[b], 8);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 8);
    mbar_init(&bars->drain, 2);  // one commit per issuing thread
    // readers: the K and the V load groups, the two MMA threads, 8 softmax warps
    tile_ring_init(&bars->ring, 12);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->mx_x[b], 8);
      mbar_init(&bars->l_x[b], 8);
    }
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

  // Each role runs inside the branch that set its register budget, so the
  // compiler allocates each branch against its own budget.
  if (warp < 4) {
  warpgroup_reg_dealloc<kRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lanes 0 and 2 load Q and K, lanes 1 and 3 load V.  Features 0..127 of a
    // tile arrive in one box (lanes 0, 1), the rest in a second (lanes 2, 3):
    // a TMA operation costs about the same time whatever its size, and
    // separate issuing threads overlap theirs.
    if (lane < 4) {
      const bool kq = (lane & 1) == 0;
      const bool lead = lane < 2;  // arrives on the full barriers
      const unsigned gmask = kq ? 0x5u : 0xAu;
      if (kq) {
        prefetch_tensormap(lead ? &tq2 : &tqt);
        prefetch_tensormap(lead ? &tk2 : &tkt);
      } else {
        prefetch_tensormap(lead ? &tv2 : &tv);
      }
      uint32_t g = 0;  // key steps loaded
      int tcount = 0;
      bool ok = true;
      // each load group reads the tile stream through its lead lane
      uint32_t ktake = 0;
      auto take = [&](int& it) -> bool {
        int v = -1, good = 1;
        if (lead) good = tile_take(&bars->ring, ktake, &v, s_abort) ? 1 : 0;
        v = __shfl_sync(gmask, v, kq ? 0 : 1);
        good = __shfl_sync(gmask, good, kq ? 0 : 1);
        it = v;
        return good != 0;
      };
      int item = -1;
      for (; (ok = take(item)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        int n, t0;
        key_order(t, n, t0);
        if (kq) {
          if (tcount > 0 &&
              !(ok = __all_sync(gmask, mbar_wait(&bars->q_empty, (tcount - 1) & 1, s_abort))))
            break;
          if (lead) mbar_arrive_expect_tx(&bars->q_full, kTailed);
          __syncwarp(gmask);
          if (lead)
            tma_load_4d(sQ, &tq2, &bars->q_full, 0, t.hg * G, t.q0 + t.tok, 0);
          else
            tma_load_3d(sQ + 2 * kTile, &tqt, &bars->q_full, 2 * kChunk, t.hg * G, t.q0 + t.tok);
        }
        // kt: key tile of step jj
        for (int jj = 0, kt = t0; jj < n; ++jj, ++g, kt = next_key_tile(t, kt)) {
          const int key = t.k0 + kt * kKeys;
          const int s = g & 1;
          if (g >= 2 && !(ok = __all_sync(gmask, mbar_wait(kq ? &bars->k_empty[s] : &bars->v_empty[s],
                                                            ((g - 2) >> 1) & 1, s_abort))))
            break;
          if (kq) {
            uint8_t* dst = sK + s * kTailed;
            if (lead) mbar_arrive_expect_tx(&bars->k_full[s], kTailed);
            __syncwarp(gmask);
            if (lead)
              tma_load_3d(dst, &tk2, &bars->k_full[s], 0, key, 0);
            else
              tma_load_2d(dst + 2 * kTile, &tkt, &bars->k_full[s], 2 * kChunk, key);
          } else {
            uint8_t* dst = sV + s * kTile3;
            if (lead) mbar_arrive_expect_tx(&bars->v_full[s], kTile3);
            __syncwarp(gmask);
            if (lead)
              tma_load_3d(dst, &tv2, &bars->v_full[s], 0, key, 0);
            else
              tma_load_2d(dst + 2 * kTile, &tv, &bars->v_full[s], 2 * kChunk, key);
          }
        }
      }
      if (*s_abort && lead) {
        // let every load this group started land before the CTA exits
        if (kq && tcount > 0) drain_wait(&bars->q_full, (tcount - 1) & 1);
        for (uint32_t f = g > 2 ? g - 2 : 0; f < g; ++f)
          drain_wait(kq ? &bars->k_full[f & 1] : &bars->v_full[f & 1], (f >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S = Q K^T issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
      constexpr int nk = HD / 16;
      uint32_t g = 0;  // global key-step counter of this CTA
      int tcount = 0;
      bool ok = true;
      // K-major operand stored as two 128-byte-swizzled chunks + a 64-byte tail
      auto tailed = [&](uint32_t base, int k) -> uint64_t {
        return k < 8 ? sdesc_sw128(base + (k >> 2) * kTile + (k & 3) * 32, 16, 1024)
                     : sdesc_sw64(base + 2 * kTile + (k - 8) * 32);
      };
      uint32_t ktake = 0;
      int item = -1;
      for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        int n, t0;
        key_order(t, n, t0);
        if (!(ok = mbar_wait(&bars->q_full, tcount & 1, s_abort))) break;
        if (n == 0) {  // no keys: nothing to multiply; keep every phase count
          mbar_arrive(&bars->q_empty);
          continue;
        }
        for (int jj = 0; jj < n; ++jj) {
          const uint32_t gs = g + jj;
          if (!(ok = mbar_wait(&bars->k_full[gs & 1], (gs >> 1) & 1, s_abort))) break;
          // the buffer's previous S (step gs - 2) has been read by the softmax
          if (gs >= 2 && !(ok = mbar_wait(&bars->s_read[gs & 1], ((gs - 2) >> 1) & 1, s_abort)))
            break;
          tc_fence_after();
          const uint32_t kb = smem_addr(sK + (gs & 1) * kTailed);
          const uint32_t qb = smem_addr(sQ);
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k)  // K steps below the head dimension
            if (k < nk) umma_ss(tmem + (gs & 1) * 128, tailed(qb, k), tailed(kb, k), kIdS, k > 0);
          umma_commit(&bars->s_full[gs & 1]);
          umma_commit(&bars->k_empty[gs & 1]);
          if (jj == n - 1) umma_commit(&bars->q_empty);
        }
        g += n;
      }
      // every MMA this thread issued completes before the CTA moves on
      umma_commit(&bars->drain);
      drain_wait(&bars->drain, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ O += P V issuer
    // A second issuing thread, so that the wait for P_j and the bookkeeping
    // between groups overlap the S products queued by warp 1.
    if (lane == 0) {
      constexpr uint32_t kIdO = idesc_f16(128, HD, BF16, false, true);  // N = d
      uint32_t g = 0;
      int tcount = 0;
      bool ok = true;
      uint32_t ktake = 0;
      int item = -1;
      for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        int n, t0;
        key_order(t, n, t0);
        if (n == 0) {
          if (tcount > 0 && !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort))) break;
          mbar_arrive(&bars->o_full);
          continue;
        }
        for (int jj = 0; jj < n; ++jj) {
          const uint32_t gg = g + jj;
          if (!(ok = mbar_wait(&bars->p_full[gg & 1], (gg >> 1) & 1, s_abort))) break;
          if (jj == 0 && tcount > 0 &&
              !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort)))
            break;
          if (!(ok = mbar_wait(&bars->v_full[gg & 1], (gg >> 1) & 1, s_abort))) break;
          tc_fence_after();
          const uint32_t vb = smem_addr(sV + (gg & 1) * kTile3);
          // keys 16k..16k+15: pair columns 8k..8k+7 of the P region
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k)
            umma_ts(tmem + kColO, tmem + kColP + k * 8, sdesc_sw128(vb + k * 2048, kTile, 1024),
                    kIdO, (jj > 0 || k > 0));
          umma_commit(&bars->pv_done);
          umma_commit(&bars->v_empty[gg & 1]);
          if (jj == n - 1) umma_commit(&bars->o_full);
        }
        g += n;
      }
      umma_commit(&bars->drain);
      drain_wait(&bars->drain, 0);
    }
  } else if (warp == 3) {
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
    const int half = (warp - 4) >> 2;  // keys [64*half, 64*half + 64) of each tile
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const LogitMap lm = make_logit_map(p);
    const bool capped = FIXED || lm.capped;  // the fixed reference needs a cap
    constexpr bool masked = MASK;
    // With the softcap every logit of a row lies within 2c of a bound known
    // before any key is seen, so P is taken against that bound: no row max,
    // no exchange between the halves, no rescale of O.
    constexpr bool fixed = FIXED;
    uint32_t g = 0;
    int tcount = 0;
    bool ok = true;
    uint32_t ktake = 0;
    int item = -1;
    for (; (ok = tile_take_warp(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
      QTile t;
      qtile_decode<MASK>(p, item, t);
      int n, t0;
      key_order(t, n, t0);
      const int i_loc = t.tok + r / G;
      const int h = t.hg * G + r % G;
      const bool row_valid = i_loc < t.Lq;
      const float slope2 = p.slopes ? __ldg(p.slopes + t.b * p.slopes_bs + h) * kLog2e : 0.f;
      const int pos_off = i_loc + t.Lk - t.Lq;  // dist(j) = |pos_off - j|
      float m_run = -INFINITY, l = 0.f;          // l: this half's share of the row sum
      uint64_t l2 = f2_make(0.f, 0.f), lu2 = l2;  // fixed reference: row sums as pairs
      if (fixed) m_run = row_bound<MASK>(p, t.Lk, pos_off, slope2);
      const float bref = fixed ? m_run : 0.f;  // subtracted inside the logit
      // dropout of this row: P V uses P * keep * scale, the sums plain P
      uint64_t dkb = 0, dhi = 0;
      uint32_t dT = 0;
      float dsc = 1.f;
      // with a stored keep mask: this row's words of the tile's blocks
      const uint64_t* mrow = nullptr;
      if (DROP) {
        dkb = splitmix64(p.drop_seed ^ static_cast<uint64_t>(t.b));
        dhi = drop_hi(p.head0 + h, i_loc);
        if (row_valid) drop_row(p, static_cast<int64_t>(t.q0) + i_loc, dT, dsc);
        if (p.drop_mask)
          mrow = drop_mask_block(p, t.b, t.Lk, t.tok / (kRowsQ / G), t.hg, 0) + half * kRowsQ + r;
      }

      for (int jj = 0, kt = t0; jj < n; ++jj, kt = next_key_tile(t, kt)) {
        const uint32_t gg = g + jj;
        const int key0 = kt * kKeys + half * 64;
        const uint32_t sb = tmem + (gg & 1) * 128 + half * 64 + lane_addr;
        // dropout keep bits of this half's 64 keys, hashed while S is computed
        uint64_t kbits = 0;
        if (DROP) {
          if (mrow) {  // written by the mask kernel
            kbits = __ldg(mrow + kt * kMaskBlockWords);
          } else {
#pragma unroll 4
            for (int c = 0; c < 64; c += 4)  // key0 is a multiple of 64
              kbits |= static_cast<uint64_t>(drop_keep4(drop_hash(dkb, dhi, (key0 + c) >> 2), dT))
                       << c;
          }
        }
        auto dropped = [&](float pv, int c) -> float { return ((kbits >> c) & 1) ? pv * dsc : 0.f; };
        if (!(ok = mbar_wait_warp(&bars->s_full[gg & 1], (gg >> 1) & 1, s_abort))) break;
        tc_fence_after();
        float x[64];
        tmem_ld32(sb, *reinterpret_cast<float(*)[32]>(x));
        tmem_ld32(sb + 32, *reinterpret_cast<float(*)[32]>(x + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_read[gg & 1]);  // S_gg may be overwritten
        const float pos0 = static_cast<float>(pos_off - key0);
        // the mask is applied per key only on the half tiles it cuts for some row
        const bool edge =
            key0 + 64 > t.Lk ||
            (masked && !__all_sync(0xffffffffu, !row_valid ||
                                                    all_admissible(p, t.Lq, t.Lk, i_loc, key0,
                                                                   key0 + 63)));
        // batched: all tanh of a 32-column group, then the logits
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float* xb = x + b * 32;
          if (capped) {
            float th[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) th[c] = tanh_approx(xb[c] * lm.in_scale);
#pragma unroll
            for (int c = 0; c < 32; ++c)
              xb[c] = fmaf(th[c], lm.out_scale,
                           fmaf(-slope2, fabsf(pos0 - static_cast<float>(b * 32 + c)), -bref));
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              xb[c] = fmaf(xb[c], lm.in_scale,
                           fmaf(-slope2, fabsf(pos0 - static_cast<float>(b * 32 + c)), -bref));
          }
        }
        if (edge) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int jg = key0 + c;
            bool adm = jg < t.Lk;
            if (masked) adm = adm && admissible(p, t.Lq, t.Lk, i_loc, jg);
            x[c] = adm ? x[c] : -INFINITY;
          }
        }
        if (fixed) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            x[c] = ex2_approx(x[c]);  // the reference is inside the logit
            x[c + 1] = ex2_approx(x[c + 1]);
            if (DROP) {
              pk[c >> 1] = Pack<BF16>::two(dropped(x[c], c), dropped(x[c + 1], c + 1));
              lu2 = f2_add(lu2, f2_make(x[c], x[c + 1]));
              continue;
            }
            pk[c >> 1] = Pack<BF16>::two(x[c], x[c + 1]);
            // two row sums: of P (for lse) and of the rounded P that
            // multiplies V (for out, which is then exactly a weighted mean of
            // V rows: one key gives out = v; with dropout out is normalised by
            // the plain sum)
            lu2 = f2_add(lu2, f2_make(x[c], x[c + 1]));
            l2 = f2_add(l2, Pack<BF16>::unpack(pk[c >> 1]));
          }
          // the previous P V has finished reading the P region
          if (gg >= 1 && !(ok = mbar_wait_warp(&bars->pv_done, (gg - 1) & 1, s_abort))) break;
          tc_fence_after();
          const uint32_t pb = tmem + kColP + half * 32 + lane_addr;
          tmem_st16(pb, *reinterpret_cast<uint32_t(*)[16]>(pk));
          tmem_st16(pb + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->p_full[gg & 1]);
          continue;
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) mx = fmaxf(mx, x[c]);
        // the row max over both halves of the tile
        float* mxs = sMax + (gg & 1) * 256;
        mxs[half * 128 + r] = mx;
        if (!(ok = warp_exchange(&bars->mx_x[gg & 1], (gg >> 1) & 1, s_abort))) break;
        mx = fmaxf(mx, mxs[(half ^ 1) * 128 + r]);
        const float m_new = fmaxf(m_run, mx);
        const bool need = m_new > m_run + kRescale;
        const float alpha = need ? ex2_approx(m_run - m_new) : 1.f;
        // the previous P V has finished reading the P region (and adding to O)
        if (gg >= 1 && !(ok = mbar_wait_warp(&bars->pv_done, (gg - 1) & 1, s_abort))) break;
        tc_fence_after();
        if (jj > 0 && __any_sync(0xffffffffu, need)) {
          // O must absorb the new max: scale this half's 80 columns
          const uint32_t ob = tmem + kColO + half * 80 + lane_addr;
#pragma unroll 1
          for (int c = 0; c < 3; ++c) {  // columns 0..31, 32..63, 48..79 (the overlapping
            float o[32];                 // 16 are scaled once, on the second pass)
            tmem_ld32(ob + (c < 2 ? c * 32 : 48), o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c < 2 || i >= 16) o[i] *= alpha;
            tmem_st32(ob + (c < 2 ? c * 32 : 48), o);
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
        for (int c = 0; c < 64; ++c) x[c] = ex2_approx(x[c] - m_use);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          l += x[c] + x[c + 1];
          pk[c >> 1] = DROP ? Pack<BF16>::two(dropped(x[c], c), dropped(x[c + 1], c + 1))
                            : Pack<BF16>::two(x[c], x[c + 1]);
        }
        // this half's 64 keys -> 32 pair columns of the P region
        const uint32_t pb = tmem + kColP + half * 32 + lane_addr;
        tmem_st16(pb, *reinterpret_cast<uint32_t(*)[16]>(pk));
        tmem_st16(pb + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[gg & 1]);
      }
      if (!ok) break;
      g += n;
      float lr = 0.f;  // rounded-P sum (fixed reference)
      if (fixed) {
        l = f2_lo(lu2) + f2_hi(lu2);
        lr = f2_lo(l2) + f2_hi(l2);
      }
      // ---- epilogue: out = O / l, lse = (m + log2 l) ln 2; each half 80 features
      float* ls = sSum + (tcount & 1) * 256;
      float* lrs = sMax + (tcount & 1) * 256;  // the max exchange is idle here
      ls[half * 128 + r] = l;
      if (fixed) lrs[half * 128 + r] = lr;
      if (!(ok = warp_exchange(&bars->l_x[tcount & 1], (tcount >> 1) & 1, s_abort))) break;
      const float lt = l + ls[(half ^ 1) * 128 + r];
      const float lrt = fixed ? lr + lrs[(half ^ 1) * 128 + r] : 0.f;
      if (!(ok = mbar_wait_warp(&bars->o_full, tcount & 1, s_abort))) break;
      tc_fence_after();
      const float lnorm = (fixed && !DROP) ? lrt : lt;
      const float inv = (lnorm > 0.f) ? 1.f / lnorm : 0.f;
      if (row_valid && half == 0)
        p.lse[static_cast<int64_t>(t.q0 + i_loc) * p.lse_rs + h] =
            (lt > 0.f) ? (m_run + log2f(lt)) * kLn2 : -INFINITY;
      const uint32_t ob = tmem + kColO + half * 80 + lane_addr;
      float o[80];
      tmem_ld32(ob, *reinterpret_cast<float(*)[32]>(o));
      tmem_ld32(ob + 32, *reinterpret_cast<float(*)[32]>(o + 32));
      {
        float tail[32];
        tmem_ld32(ob + 48, tail);  // columns 48..79 (x32 load; 48..63 already held)
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) o[64 + i] = tail[16 + i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty);
      if (row_valid) {
        uint16_t* orow = static_cast<uint16_t*>(p.out) +
                         static_cast<int64_t>(t.q0 + i_loc) * p.out_ts +
                         static_cast<int64_t>(h) * p.out_hs + half * 80;
        const int nu = feature_units(HD, half);
#pragma unroll
        for (int u = 0; u < 10; ++u) {
          float w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = n > 0 ? o[8 * u + i] * inv : 0.f;
          if (u < nu) *reinterpret_cast<uint4*>(orow + u * 8) = pack8<BF16>(w);
        }
      }
    }
  }

  }
  __syncthreads();
  if (tid == 0 && *s_abort) atomicOr(p.status, ATTN_DEV_TIMEOUT_FWD);
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <bool B, bool M, bool DR, bool FX>
auto fwd_for_d(int d) {
  return d == 128 ? fwd_kernel<B, M, 128, DR, FX>
                  : (d == 64 ? fwd_kernel<B, M, 64, DR, FX> : fwd_kernel<B, M, 160, DR, FX>);
}

template <bool DR, bool FX>
auto fwd_pick(const Params& p) {
  const bool m = masked_call(p);
  return p.dtype == 1 ? (m ? fwd_for_d<true, true, DR, FX>(p.d) : fwd_for_d<true, false, DR, FX>(p.d))
                      : (m ? fwd_for_d<false, true, DR, FX>(p.d) : fwd_for_d<false, false, DR, FX>(p.d));
}

cudaError_t launch_fwd(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tqt,
                       const CUtensorMap& tk2, const CUtensorMap& tkt, const CUtensorMap& tv2,
                       const CUtensorMap& tv, int grid, cudaStream_t s) {
  // the fixed-reference softmax needs a softcap (make_logit_map: capped when > 0)
  const bool fixed = p.softcap > 0.f && p.softcap <= kFixedCapMax;
  auto k = p.dropout ? (fixed ? fwd_pick<true, true>(p) : fwd_pick<true, false>(p))
                     : (fixed ? fwd_pick<false, true>(p) : fwd_pick<false, false>(p));
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::kSmem);
  k<<<grid, fwd::kThreadsF, fwd::kSmem, s>>>(p, tq2, tqt, tk2, tkt, tv2, tv);
  return cudaGetLastError();
}

}  // namespace attn
