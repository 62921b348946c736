// bwd_dq.cu -- backward pass, dq.
//
// dq_i = sigma * sum_j dS_ij k_j with dS_ij = P_ij (dP_ij - D_i)(1 - tanh^2),
// P_ij = exp(z_ij - lse_i) recomputed from the stored lse ("ragged flash
// attention gradient recompute", "Root causes addressed": no P is stored; the
// backward recomputes each tile from L).  dq has its own pass over the key
// tiles so that every dq row is written once, by one CTA, with no atomics:
// repeated calls are bitwise identical.
//
// Tile: the forward's 128 query rows.  Per key tile j:
//   S_j  = Q K_j^T    M=128 N=128 K=d, Q from TMEM, K from shared memory
//   dP_j = dO V_j^T   M=128 N=128 K=d, both from shared memory
//   dS_j              elementwise warps; written as 16-bit pairs over the
//                     columns of dP_j they have read
//   dQ  += dS_j K_j   M=128 N=d K=128, A operand from TMEM
// (d = 160 in the pages' workload; the layouts below are those of 160.)
//
// Warp roles (384 threads, 12 warps): warp 0 loads with TMA (dO once per
// tile; K through three slots, V through one; each tile as two boxes from two
// lanes), warp 1 issues the S and dP products, warp 2 the dQ products,
// warps 4-11 do the elementwise work (two warps per TMEM lane quadrant, each
// taking 64 of the 128 keys) and, at the start of each tile, copy the tile's
// Q rows from global memory into TMEM.  Q lives in TMEM so that shared memory
// holds three K slots: K of a key tile is read twice, by S early in the step
// and by dQ at its end, and with two slots the load of K_{j+2} (which waits
// for dQ of tile j) arrived after S_{j+2} was due.  S as a TMEM-A product also
// reads half the shared-memory bytes of the SS form.  dO and V are only
// K-major operands and keep their last 32 features in a 64-byte-swizzled
// chunk; K is also the MN-major operand of dQ and stays in three
// 128-byte-swizzled chunks.
// Warp 3 only completes warpgroup 0, which hands most of its registers to
// the elementwise warpgroups (setmaxnreg), so those can keep every column's
// MUFU/FMA chain of a batch in flight.
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace dqk {
constexpr int kThreadsDQ = kThreads;  // 12 warps
constexpr uint32_t kTile = 16384;            // 64-feature chunk of 128 rows
constexpr uint32_t kTail = 8192;             // features 128..159 of 128 rows
constexpr uint32_t kTailed = 2 * kTile + kTail;
constexpr int kKSlots = 3;
constexpr uint32_t kOffDO = 0;
constexpr uint32_t kOffK = kTailed;          // three K slots, 3 full chunks each
constexpr uint32_t kOffV = kOffK + kKSlots * 3 * kTile;
constexpr uint32_t kOffBar = kOffV + kTailed;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColP = 128;   // dP, then dS as 16-bit pairs over its read columns
constexpr uint32_t kColQ = 256;   // dQ accumulator
constexpr uint32_t kColQt = 416;  // the tile's Q rows as 16-bit pairs (80 columns)

struct Bars {
  uint64_t q_full, q_empty, qt_full;
  uint64_t k_full[kKSlots], k_empty[kKSlots], v_full, v_empty;
  uint64_t s_full, s_free, dp_full, p_full, dq_done;
  uint64_t o_full, o_empty, drain;
  TileRing ring;  // query tiles drawn by warp 0 for the whole CTA
};
// barriers, then the TMEM base address, the abort flag and the status copy
constexpr uint32_t kSmem = kOffBar + sizeof(Bars) + 16;  // base checked to be 1024-aligned
static_assert(kSmem <= 232448, "shared memory");

// Position in a three-slot ring: slot = n mod 3 and use = n / 3, advanced
// without a division.
struct Ring3 {
  int slot = 0;
  uint32_t use = 0;
  __device__ __forceinline__ void next() {
    if (++slot == kKSlots) {
      slot = 0;
      ++use;
    }
  }
};
}  // namespace dqk

__device__ __forceinline__ void drain_wait_dq(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

// HD: the head dimension (160, 128 or 64) -- the MMA shapes and the stores
// follow it; the shared-memory and TMEM layouts are those of 160 features.
// CAP: the call has a softcap (instances for capped calls hold no uncapped
// branch in their element code); otherwise read at run time.
template <bool BF16, bool MASK, int HD, bool DROP, bool CAP = false>
__global__ void __launch_bounds__(dqk::kThreadsDQ, 1)
    dq_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq2,
              const __grid_constant__ CUtensorMap tqt, const __grid_constant__ CUtensorMap tdo2,
              const __grid_constant__ CUtensorMap tdot, const __grid_constant__ CUtensorMap tk2,
              const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv2,
              const __grid_constant__ CUtensorMap tvt) {
  using namespace dqk;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sDO = sm + kOffDO;
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
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
  // Launched as a programmatic dependent of dk/dv, this grid may start before
  // dk/dv ends; every CTA waits for dk/dv to complete before exiting, so the
  // work after dq in the stream (the next K/V head group, or the next call,
  // whose schedule kernel resets the tile counters dk/dv draws from) never
  // overlaps dk/dv.  Without a prerequisite grid the wait returns at once.
  auto wait_prerequisite = [&]() {
    if (tid == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
  };
  if (*s_status != 0 || static_cast<int>(blockIdx.x) >= ntiles) {
    wait_prerequisite();
    return;
  }

  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->qt_full, 8);
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    mbar_init(&bars->v_full, 1);
    mbar_init(&bars->v_empty, 1);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_free, 8);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->dq_done, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_empty, 8);
    mbar_init(&bars->drain, 2);  // one commit per issuing thread
    tile_ring_init(&bars->ring, 10);  // the two MMA threads, the 8 elementwise warps
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
    // The whole warp walks the fills; each tile's boxes are issued from
    // separate lanes (features 0..127 of a tile in one box, the rest in a
    // second), since a TMA operation costs about the same time whatever its
    // size and separate issuing threads overlap theirs.
    if (lane == 0) {
      prefetch_tensormap(&tdo2);
      prefetch_tensormap(&tk2);
    } else if (lane == 1) {
      prefetch_tensormap(&tdot);
      prefetch_tensormap(&tk);
    } else if (lane == 2) {
      prefetch_tensormap(&tv2);
    } else if (lane == 3) {
      prefetch_tensormap(&tvt);
    }
    uint32_t g = 0;  // key tiles loaded
    Ring3 kr;        // K slot of key tile g
    int tcount = 0;
    bool ok = true;
    uint32_t kpub = 0;
    int item = -1, item_next = -1;
    ok = tile_publish(&bars->ring, kpub, p.counters + 2, ntiles, &item, s_abort);
    if (ok && item >= 0) ok = tile_publish(&bars->ring, kpub, p.counters + 2, ntiles, &item_next, s_abort);
    for (; item >= 0 && ok; item = item_next, ++tcount,
         ok = ok && (item < 0 || tile_publish(&bars->ring, kpub, p.counters + 2, ntiles,
                                              &item_next, s_abort))) {
      QTile t;
      qtile_decode<MASK>(p, item, t);
      const int n = t.nkt;  // key tiles t.kt0 .. t.kt0 + n - 1
      const int h0 = t.hg * G, tok = t.q0 + t.tok;
      if (tcount > 0 && !(ok = mbar_wait_warp(&bars->q_empty, (tcount - 1) & 1, s_abort))) break;
      if (lane == 0) mbar_arrive_expect_tx(&bars->q_full, kTailed);
      __syncwarp();
      if (lane == 0) tma_load_4d(sDO, &tdo2, &bars->q_full, 0, h0, tok, 0);
      if (lane == 1) tma_load_3d(sDO + 2 * kTile, &tdot, &bars->q_full, 2 * kChunk, h0, tok);
      for (int j = 0; j < n && ok; ++j, ++g, kr.next()) {
        const int key = t.k0 + (t.kt0 + j) * kKeys;
        if (kr.use > 0 &&
            !(ok = mbar_wait_warp(&bars->k_empty[kr.slot], (kr.use - 1) & 1, s_abort)))
          break;
        if (lane == 0) mbar_arrive_expect_tx(&bars->k_full[kr.slot], 3 * kTile);
        __syncwarp();
        uint8_t* dk = sK + kr.slot * 3 * kTile;
        if (lane == 0) tma_load_3d(dk, &tk2, &bars->k_full[kr.slot], 0, key, 0);
        if (lane == 1) tma_load_2d(dk + 2 * kTile, &tk, &bars->k_full[kr.slot], 2 * kChunk, key);
        if (g >= 1 && !(ok = mbar_wait_warp(&bars->v_empty, (g - 1) & 1, s_abort))) {
          ++g;  // the K fill above is armed
          kr.next();
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(&bars->v_full, kTailed);
        __syncwarp();
        if (lane == 2) tma_load_3d(sV, &tv2, &bars->v_full, 0, key, 0);
        if (lane == 3) tma_load_2d(sV + 2 * kTile, &tvt, &bars->v_full, 2 * kChunk, key);
      }
    }
    if (*s_abort && lane == 0) {
      // let every load this warp started land before the CTA exits
      if (tcount > 0) drain_wait_dq(&bars->q_full, (tcount - 1) & 1);
      for (uint32_t f = g > kKSlots ? g - kKSlots : 0; f < g; ++f)
        drain_wait_dq(&bars->k_full[f % kKSlots], (f / kKSlots) & 1);
      if (g > 0) drain_wait_dq(&bars->v_full, (g - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S, dP issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
      constexpr int nk = HD / 16;  // K steps of S and dP below the head dimension
      const uint32_t db = smem_addr(sDO), vb = smem_addr(sV);
      // K-major operand stored as two 128-byte-swizzled chunks + a 64-byte tail
      auto tailed = [&](uint32_t base, int k) -> uint64_t {
        return k < 8 ? sdesc_sw128(base + (k >> 2) * kTile + (k & 3) * 32, 16, 1024)
                     : sdesc_sw64(base + 2 * kTile + (k - 8) * 32);
      };
      uint32_t g = 0;
      Ring3 kr;
      int tcount = 0;
      bool ok = true;
      uint32_t ktake = 0;
      int item = -1;
      for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        const int n = t.nkt;  // key tiles t.kt0 .. t.kt0 + n - 1
        if (!(ok = mbar_wait(&bars->q_full, tcount & 1, s_abort))) break;   // dO tile
        if (!(ok = mbar_wait(&bars->qt_full, tcount & 1, s_abort))) break;  // Q rows in TMEM
        if (n == 0) {
          mbar_arrive(&bars->q_empty);
          continue;
        }
        for (int j = 0; j < n; ++j, kr.next()) {
          const uint32_t gs = g + j;
          // S = Q K^T once the previous S has been read
          if (gs >= 1 && !(ok = mbar_wait(&bars->s_free, (gs - 1) & 1, s_abort))) break;
          if (!(ok = mbar_wait(&bars->k_full[kr.slot], kr.use & 1, s_abort))) break;
          tc_fence_after();
          const uint32_t kb = smem_addr(sK + kr.slot * 3 * kTile);
          // features 16k..16k+15 of Q: pair columns 8k..8k+7 of its region
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k)
            if (k < nk)
              umma_ts(tmem + kColS, tmem + kColQt + k * 8,
                      sdesc_sw128(kb + (k >> 2) * kTile + (k & 3) * 32, 16, 1024), kIdS, k > 0);
          umma_commit(&bars->s_full);
          // dP = dO V^T once dQ of the previous key tile has read dS (written
          // over the previous dP, after it was read)
          if (gs >= 1 && !(ok = mbar_wait(&bars->dq_done, (gs - 1) & 1, s_abort))) break;
          if (!(ok = mbar_wait(&bars->v_full, gs & 1, s_abort))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kHeadDim / 16; ++k)
            if (k < nk) umma_ss(tmem + kColP, tailed(db, k), tailed(vb, k), kIdS, k > 0);
          umma_commit(&bars->dp_full);
          umma_commit(&bars->v_empty);
          if (j + 1 == n) umma_commit(&bars->q_empty);  // last dP of this tile issued
        }
        g += n;
      }
      umma_commit(&bars->drain);
      drain_wait_dq(&bars->drain, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ dQ issuer
    // A second issuing thread: an MMA issue blocks while the tensor pipe is
    // busy, so the wait for dS_j must not sit behind the S and dP products
    // of the next key tile.
    if (lane == 0) {
      constexpr uint32_t kIdQ = idesc_f16(128, HD, BF16, false, true);  // N = d
      uint32_t g = 0;
      Ring3 kr;
      int tcount = 0;
      bool ok = true;
      uint32_t ktake = 0;
      int item = -1;
      for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
        QTile t;
        qtile_decode<MASK>(p, item, t);
        const int n = t.nkt;  // key tiles t.kt0 .. t.kt0 + n - 1
        if (n == 0) {
          if (tcount > 0 && !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort))) break;
          mbar_arrive(&bars->o_full);
          continue;
        }
        for (int j = 0; j < n; ++j, kr.next()) {
          const uint32_t gg = g + j;
          if (!(ok = mbar_wait(&bars->p_full, gg & 1, s_abort))) break;
          if (j == 0 && tcount > 0 &&
              !(ok = mbar_wait(&bars->o_empty, (tcount - 1) & 1, s_abort)))
            break;
          tc_fence_after();
          const uint32_t kb = smem_addr(sK + kr.slot * 3 * kTile);
          // keys 16k..16k+15: half k/4, pair column 8*(k%4) of that half's dP columns
#pragma unroll
          for (int k = 0; k < kKeys / 16; ++k)
            umma_ts(tmem + kColQ, tmem + kColP + (k >> 2) * 64 + (k & 3) * 8,
                    sdesc_sw128(kb + k * 2048, kTile, 1024), kIdQ, (j > 0 || k > 0));
          umma_commit(&bars->dq_done);
          umma_commit(&bars->k_empty[kr.slot]);
          if (j + 1 == n) umma_commit(&bars->o_full);
        }
        g += n;
      }
      umma_commit(&bars->drain);
      drain_wait_dq(&bars->drain, 0);
    }
  }
  } else {
  warpgroup_reg_alloc<kRegsHigh>();
  {
    // ------------------------------------------------------------ elementwise
    const int quad = warp & 3;
    const int half = (warp - 4) >> 2;  // keys [64*half, 64*half + 64) of each tile
    const int r = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const LogitMap lm = make_logit_map(p);
    const bool capped = CAP || lm.capped;
    constexpr bool masked = MASK;
    const int lgG = __ffs(G) - 1;  // G is a power of two
    // This lane's Q row of a tile into TMEM: features 80*half..80*half+79 as
    // 40 pair columns (raw 16-bit pairs, the A-operand layout).  Rows outside
    // the sequence get zeros.  Written once the previous tile's last S has
    // completed (the caller has waited for it), then signalled to the S issuer.
    auto load_q = [&](int qitem) -> bool {
      QTile tq;
      qtile_decode<MASK>(p, qitem, tq);
      const int il = tq.tok + (r >> lgG);
      const int hq = tq.hg * G + (r & (G - 1));
      uint32_t w[40];
      if (il < tq.Lq) {
        const uint4* src = reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(p.q) + static_cast<int64_t>(tq.q0 + il) * p.q_ts +
            static_cast<int64_t>(hq) * p.q_hs + half * 80);
        const int nu = feature_units(HD, half);  // features past d read as 0
#pragma unroll
        for (int u = 0; u < 10; ++u) {
          const uint4 v = u < nu ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
          w[4 * u] = v.x;
          w[4 * u + 1] = v.y;
          w[4 * u + 2] = v.z;
          w[4 * u + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int u = 0; u < 40; ++u) w[u] = 0u;
      }
      const uint32_t qa = tmem + kColQt + half * 40 + lane_addr;
      tmem_st16(qa, *reinterpret_cast<uint32_t(*)[16]>(w));
      tmem_st16(qa + 16, *reinterpret_cast<uint32_t(*)[16]>(w + 16));
      tmem_st8(qa + 32, *reinterpret_cast<uint32_t(*)[8]>(w + 32));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->qt_full);
      return true;
    };
    uint32_t g = 0;
    int tcount = 0;
    uint32_t ktake = 0;
    int item = -1;
    bool ok = tile_take_warp(&bars->ring, ktake, &item, s_abort);
    if (ok && item >= 0) load_q(item);
    for (int item_next = -1; ok && item >= 0; item = item_next, ++tcount) {
      QTile t;
      qtile_decode<MASK>(p, item, t);
      const int n = t.nkt;  // key tiles t.kt0 .. t.kt0 + n - 1
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
      // dropout of this row: dS = P (1 - tanh^2) (keep * scale * dP - D)
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
      for (int j = 0; j < n; ++j) {
        const uint32_t gg = g + j;
        const int key0 = (t.kt0 + j) * kKeys + half * 64;
        const float pos0 = static_cast<float>(pos_off - key0);
        // dropout keep bits of this half's 64 keys, hashed while S is computed
        uint64_t kbits = 0;
        if (DROP) {
          if (mrow) {  // written by the mask kernel
            kbits = __ldg(mrow + (t.kt0 + j) * kMaskBlockWords);
          } else {
#pragma unroll 4
            for (int c = 0; c < 64; c += 4)  // key0 is a multiple of 64
              kbits |= static_cast<uint64_t>(drop_keep4(drop_hash(dkb, dhi, (key0 + c) >> 2), dT))
                       << c;
          }
        }
        if (!(ok = mbar_wait_warp(&bars->s_full, gg & 1, s_abort))) break;
        tc_fence_after();
        float x[64];
        tmem_ld32(tmem + kColS + half * 64 + lane_addr, *reinterpret_cast<float(*)[32]>(x));
        tmem_ld32(tmem + kColS + half * 64 + 32 + lane_addr,
                  *reinterpret_cast<float(*)[32]>(x + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free);  // S may be overwritten now
        // Two batches of 32 columns; within a batch all tanh, then the exponent
        // arguments, then all exp2, so dependent MUFU results are far apart.
        // the mask is applied per key only on the half tiles it cuts for some row
        const bool edge =
            key0 + 64 > t.Lk ||
            (masked && !__all_sync(0xffffffffu, !row_valid ||
                                                    all_admissible(p, t.Lq, t.Lk, i_loc, key0,
                                                                   key0 + 63)));
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          float* xb = x + b * 32;
          float th[32];
          if (capped) {
#pragma unroll
            for (int c = 0; c < 32; ++c) th[c] = tanh_approx(xb[c] * lm.in_scale);
          }
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float bias =
                fmaf(-slope2, fabsf(pos0 - static_cast<float>(b * 32 + c)), -lse2);
            xb[c] = capped ? fmaf(th[c], lm.out_scale, bias) : fmaf(xb[c], lm.in_scale, bias);
          }
          if (edge) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int jg = key0 + b * 32 + c;
              bool adm = jg < t.Lk;
              if (masked) adm = adm && admissible(p, t.Lq, t.Lk, i_loc, jg);
              xb[c] = adm ? xb[c] : -INFINITY;
            }
          }
#pragma unroll
          for (int c = 0; c < 32; ++c) xb[c] = ex2_approx(xb[c]);  // P
          if (capped) {
#pragma unroll
            for (int c = 0; c < 32; ++c) xb[c] *= fmaf(-th[c], th[c], 1.f);  // P (1 - tanh^2)
          }
        }
        if (!(ok = mbar_wait_warp(&bars->dp_full, gg & 1, s_abort))) break;
        tc_fence_after();
        const uint32_t pbuf = tmem + kColP + half * 64 + lane_addr;
        uint32_t pk[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float d[32];
          tmem_ld32(pbuf + cc * 32, d);
          tmem_wait_ld();
          if (DROP) {
#pragma unroll
            for (int c = 0; c < 32; ++c) d[c] = ((kbits >> (cc * 32 + c)) & 1) ? d[c] * dsc : 0.f;
          }
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            pk[cc * 16 + (c >> 1)] = Pack<BF16>::two(x[cc * 32 + c] * (d[c] - Drow),
                                                     x[cc * 32 + c + 1] * (d[c + 1] - Drow));
        }
        // dS pairs over this half's first 32 (already read) dP columns
        tmem_st16(pbuf, *reinterpret_cast<uint32_t(*)[16]>(pk));
        tmem_st16(pbuf + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
      }
      if (!ok) break;
      g += n;
      // Q of the next tile (every S of this tile has completed: its last
      // s_full was waited for above)
      if (!(ok = tile_take_warp(&bars->ring, ktake, &item_next, s_abort))) break;
      if (item_next >= 0) load_q(item_next);
      // ---- epilogue: dq = sigma * dQ, this half's 80 features
      if (!(ok = mbar_wait_warp(&bars->o_full, tcount & 1, s_abort))) break;
      tc_fence_after();
      uint16_t* qrow = static_cast<uint16_t*>(p.dq) + static_cast<int64_t>(t.q0 + i_loc) * p.dq_ts +
                       static_cast<int64_t>(h) * p.dq_hs + half * 80;
      const uint32_t acc = tmem + kColQ + half * 80 + lane_addr;
      float o[80];
      tmem_ld32(acc, *reinterpret_cast<float(*)[32]>(o));
      tmem_ld32(acc + 32, *reinterpret_cast<float(*)[32]>(o + 32));
      {
        float tail16[32];
        tmem_ld32(acc + 64 - 16, tail16);  // columns 48..79 (overlap keeps the load x32)
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) o[64 + i] = tail16[16 + i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_empty);
      if (row_valid) {
        const int nu = feature_units(HD, half);
#pragma unroll
        for (int u = 0; u < 10; ++u) {
          float w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = n > 0 ? o[8 * u + i] * p.sigma : 0.f;
          if (u < nu) *reinterpret_cast<uint4*>(qrow + u * 8) = pack8<BF16>(w);
        }
      }
    }
  }

  }
  __syncthreads();
  if (tid == 0 && *s_abort) atomicOr(p.status, ATTN_DEV_TIMEOUT_DQ);
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  wait_prerequisite();
}

template <bool B, bool M, bool DR, bool C>
auto dq_for_d(int d) {
  return d == 128 ? dq_kernel<B, M, 128, DR, C>
                  : (d == 64 ? dq_kernel<B, M, 64, DR, C> : dq_kernel<B, M, 160, DR, C>);
}

template <bool DR, bool C>
auto dq_pick(const Params& p) {
  const bool m = masked_call(p);
  return p.dtype == 1 ? (m ? dq_for_d<true, true, DR, C>(p.d) : dq_for_d<true, false, DR, C>(p.d))
                      : (m ? dq_for_d<false, true, DR, C>(p.d) : dq_for_d<false, false, DR, C>(p.d));
}

cudaError_t launch_dq(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tqt,
                      const CUtensorMap& tdo2, const CUtensorMap& tdot, const CUtensorMap& tk2,
                      const CUtensorMap& tk, const CUtensorMap& tv2, const CUtensorMap& tvt,
                      int grid, bool overlap, cudaStream_t s) {
  // capped calls take the instances with a known cap (the logit map's cap
  // test: softcap > 0)
  const bool cap = p.softcap > 0.f;
  auto k = p.dropout ? (cap ? dq_pick<true, true>(p) : dq_pick<true, false>(p))
                     : (cap ? dq_pick<false, true>(p) : dq_pick<false, false>(p));
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, dqk::kSmem);
  // With `overlap` the launch is a programmatic dependent of the kernel before
  // it (dk/dv, which signals at its start): dq reads nothing dk/dv writes, so
  // its CTAs may start on the SMs that dk/dv's last CTAs leave idle.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(dqk::kThreadsDQ);
  cfg.dynamicSmemBytes = dqk::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, p, tq2, tqt, tdo2, tdot, tk2, tk, tv2, tvt);
}

}  // namespace attn
