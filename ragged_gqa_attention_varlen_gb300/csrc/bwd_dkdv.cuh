// bwd_dkdv.cuh -- backward pass, dk and dv: the kernel template (instantiated
// by bwd_dkdv.cu without dropout and by bwd_dkdv_drop.cu with it).
//
// dv_j = sum_h sum_i P_ij dO_i and dk_j = sigma * sum_h sum_i dS_ij q_i, the
// sums running over every query head that shares the K/V head (all of them
// in the pages' case of one K/V head: "Noncausal Global Extreme-GQA Ragged
// Attention Full VJP", "Hard Constraints"; the query heads of one group when
// the host runs K/V head groups one after the other) and every query of the
// sequence.  P is recomputed from the
// stored lse ("ragged flash attention gradient recompute", "Root causes
// addressed").
//
// One CTA owns 128 keys of one sequence and keeps their dV and dK
// accumulators in TMEM (2 x 160 fp32 columns) while it walks every 128-row
// query step (128/G tokens x G heads, the forward's query tile) of the
// sequence in a fixed order, so the reduction order over heads and queries
// never changes: no atomics, bitwise repeatable.  Keys are the MMA M
// dimension.  The remaining 192 TMEM columns hold two regions that each
// matrix of a step passes through in turn:
//   SP [320,448): S^T = K Q^T, then (once S^T has been read) dP^T = V dO^T,
//                 then (once dP^T has been read) S^T of the next step
//   X  [448,512): P^T as 16-bit pairs, read by dV += P^T dO; then dS^T, read
//                 by dK += dS^T Q; then P^T of the next step
// so the tensor core computes S^T of the next step while the elementwise
// warps finish dS of this one.
//
// Warp roles (384 threads, 12 warps): warp 0 loads tiles with TMA, warp 1
// issues S^T and dP^T, warp 3 issues dV and dK, warp 2 stages each query
// step's per-column scalars (bias coefficients and D), warps 4-11 compute P^T
// and dS^T and write dk/dv -- two warps per TMEM lane quadrant, each taking 64
// of the step's 128 query columns.
//
// Shared memory: K and V are K-major operands only and keep features 128..159
// in a 64-byte-swizzled chunk (40 KB each).  Q and dO are also MN-major
// operands (of dK and dV) and use three 128-byte-swizzled 64-feature chunks
// (48 KB); Q has two slots, dO one.
#pragma once
#include <type_traits>
#include "../../include/attn_varlen.h"
#include "common.cuh"
#include "sched.cuh"

namespace attn {

namespace kv {
constexpr uint32_t kTile = 16384;  // 64-feature chunk of 128 rows
constexpr uint32_t kTail = 8192;   // features 128..159 of 128 rows (64-byte rows)
constexpr uint32_t kKV = 2 * kTile + kTail;
constexpr uint32_t kTile3 = 3 * kTile;

struct Cols {          // per-column scalars (column = token * G + head)
  float a[2][128];     // bias at key r = a + m * r (base 2) when the step is one-sided
  float m[2][128];
  float D[128];
  int general[2][2];   // [buffer][0]: some column needs |i - j| or a mask ([b][1] stays 0)
};

struct Bars {
  uint64_t kv_full, kv_empty, q_full[2], q_empty[2], do_full, do_empty;
  uint64_t s_full, s_read, dp_full, dp_read, p_full, dv_done, ds_full, dk_done;
  uint64_t acc_full, acc_empty, am_full[2], am_empty[2], d_full, d_empty, drain;
  TileRing ring;  // key tiles drawn by warp 0 for the whole CTA
};

constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kKV;
constexpr uint32_t kOffQ = 2 * kKV;              // two Q slots
constexpr uint32_t kOffDO = kOffQ + 2 * kTile3;  // one dO slot
constexpr uint32_t kOffCol = kOffDO + kTile3;
constexpr uint32_t kOffBar = kOffCol + sizeof(Cols);
constexpr uint32_t kSmem = kOffBar + sizeof(Bars) + 16;  // the base is checked to be 1024-aligned
static_assert(kSmem <= 232448, "shared memory");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDV = 0;
constexpr uint32_t kColDK = 160;
constexpr uint32_t kColSP = 320;  // S^T, then dP^T
constexpr uint32_t kColX = 448;   // P^T, then dS^T (16-bit pairs)
}  // namespace kv

__device__ __forceinline__ void drain_wait_kv(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
}

// Fill/use counters of a two-slot ring, kept in registers (no indexed arrays).
struct Pair {
  uint32_t c0 = 0, c1 = 0;
  __device__ __forceinline__ uint32_t get(int s) const { return s ? c1 : c0; }
  __device__ __forceinline__ uint32_t bump(int s) {
    const uint32_t v = s ? c1 : c0;
    if (s) ++c1; else ++c0;
    return v;
  }
};

// The order in which a key tile walks its query steps.  Step st is token
// block tb(st / ngroups), head group st % ngroups.  The steps whose columns'
// aligned keys may lie inside the tile (the "band" of token blocks [tbA, tbB),
// whose bias need not be one line per column over the tile's keys) go last.
// Without a mask the step loop then runs in two parts: the other steps with
// the one-sided element code only, then the band.  With a mask every step may
// be cut, so one loop checks each step; the order is the same, so a window
// wider than every sequence gives bitwise the unmasked results.
struct StepMap {
  int tb0, nA, nC, tbA, tbB;
  // token block of the j-th block in the walk: [tb0, tbA), [tbB, ..), [tbA, tbB)
  __device__ __forceinline__ int tb(int j) const {
    return j < nA ? tb0 + j : (j < nA + nC ? tbB + (j - nA) : tbA + (j - nA - nC));
  }
};

// band_last false: the natural order (the dropout instances walk it: their
// keep-mask reads and hashing keep the tiles of a sequence closer together so)
__device__ __forceinline__ StepMap step_map(const KTile& t, int step_tok, bool band_last) {
  StepMap m;
  m.tb0 = t.tb0;
  m.nA = t.ntb;
  m.nC = 0;
  m.tbA = m.tbB = t.tb0 + t.ntb;
  if (!band_last) return m;
  // tokens i with 0 < i + Lk - Lq - key < 127 (and i < Lq) straddle the tile
  const int off = t.Lk - t.Lq;
  const int lo = max(0, t.key - off + 1), hi = min(t.Lq - 1, t.key - off + kKeys - 2);
  if (lo > hi) return m;
  m.tbA = max(t.tb0, lo / step_tok);
  m.tbB = min(t.tb0 + t.ntb, hi / step_tok + 1);
  if (m.tbA >= m.tbB) {
    m.tbA = m.tbB = t.tb0 + t.ntb;
    return m;
  }
  m.nA = m.tbA - t.tb0;
  m.nC = t.tb0 + t.ntb - m.tbB;
  return m;
}

// HD: the head dimension (160, 128 or 64) -- the MMA shapes and the stores
// follow it; the shared-memory and TMEM layouts are those of 160 features.
// DM: dropout off (0), with the call's one rate (1), or with a rate per query
// token from the table the schedule kernel builds (2) -- separate instances,
// so the per-element work of the one-rate case holds no table lookup; 3 and 4
// are 1 and 2 with the keep bits read from the stored mask instead of hashed
// (separate instances too, so neither path's registers burden the other).
// CAP: the call has a softcap (set only on instances launched for capped
// calls, so their element code holds no uncapped branch); otherwise the cap
// is read from the parameters at run time.
template <bool BF16, bool MASK, int HD, int DM, bool CAP = false>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tq2,
                const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo2,
                const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk2,
                const __grid_constant__ CUtensorMap tkt, const __grid_constant__ CUtensorMap tv2,
                const __grid_constant__ CUtensorMap tvt) {
  using namespace kv;
  constexpr bool DROP = DM != 0;
  constexpr bool DTAB = DM == 2 || DM == 4;
  constexpr bool DMASK = DM >= 3;
  // without dropout the walk puts the band last (masked or not, so that a
  // window wider than every sequence stays bitwise the unmasked call), and
  // without a mask the step loop splits there
  constexpr bool kBandLast = !DROP;
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
  // the next kernel (dq, launched as a programmatic dependent) reads nothing
  // this one writes, so it may be scheduled as soon as SMs free up
  if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    *s_status = *reinterpret_cast<volatile int32_t*>(p.status);
    // every tile here needs a 1024-byte-aligned base (swizzle atoms)
    if (smem_addr(sm) & 1023u) {
      atomicOr(p.status, ATTN_DEV_SMEM_ALIGN);
      *s_status = 1;
    }
  }
  __syncthreads();
  // (the rows of keys outside every scheduled tile were zeroed by the
  // preprocess kernel)
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
    mbar_init(&bars->do_empty, 2);  // dO is read by dP^T (warp 1) and dV (warp 3)
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->s_read, 8);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->dp_read, 8);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->dv_done, 1);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->dk_done, 1);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->d_full, 1);
    mbar_init(&bars->d_empty, 8);
    mbar_init(&bars->drain, 2);  // one commit per issuing thread
    // readers: the two MMA threads, the staging warp, the 8 elementwise warps
    tile_ring_init(&bars->ring, 11);
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
  // steps of a key tile: query blocks t.tb0 .. t.tb0 + t.ntb - 1, each over every head group
  auto step_count = [&](const KTile& t) { return t.ntb * ngroups; };

  // Each role runs inside the branch that set its register budget, so the
  // compiler allocates each branch against its own budget.
  if (warp < 4) {
  warpgroup_reg_dealloc<kRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the fills in the order their slots are released
    // (Q of step g after dK of step g - 2, dO of step g after dV of step
    // g - 1); each tile's boxes are issued from separate lanes, since the
    // load rate grows with the number of issuing threads.
    if (lane < 4) {
      prefetch_tensormap(&tq2);
      prefetch_tensormap(&tq);
      prefetch_tensormap(&tdo2);
      prefetch_tensormap(&tdo);
    } else if (lane < 8) {
      prefetch_tensormap(&tk2);
      prefetch_tensormap(&tkt);
      prefetch_tensormap(&tv2);
      prefetch_tensormap(&tvt);
    }
    uint32_t nkv = 0, ndo = 0;
    Pair nq;
    bool ok = true;
    uint32_t kpub = 0;
    int item = -1, item_next = -1;
    ok = tile_publish(&bars->ring, kpub, p.counters + 1, ntiles, &item, s_abort);
    if (ok && item >= 0) ok = tile_publish(&bars->ring, kpub, p.counters + 1, ntiles, &item_next, s_abort);
    for (; item >= 0 && ok; item = item_next,
         ok = ok && (item < 0 || tile_publish(&bars->ring, kpub, p.counters + 1, ntiles,
                                              &item_next, s_abort))) {
      KTile t;
      ktile_decode<MASK>(p, item, t);
      const int nsteps = step_count(t);
      const int key = t.k0 + t.key;
      if (nkv > 0 && !(ok = mbar_wait_warp(&bars->kv_empty, (nkv - 1) & 1, s_abort))) break;
      if (lane == 0) mbar_arrive_expect_tx(&bars->kv_full, 2 * kKV);
      __syncwarp();
      if (lane == 0) tma_load_3d(sK, &tk2, &bars->kv_full, 0, key, 0);
      if (lane == 1) tma_load_2d(sK + 2 * kTile, &tkt, &bars->kv_full, 2 * kChunk, key);
      if (lane == 2) tma_load_3d(sV, &tv2, &bars->kv_full, 0, key, 0);
      if (lane == 3) tma_load_2d(sV + 2 * kTile, &tvt, &bars->kv_full, 2 * kChunk, key);
      const StepMap sm = step_map(t, step_tok, kBandLast);
      ++nkv;
      // Q and dO stream from memory (a sequence's Q alone can exceed L2).
      // No L2 prefetch ahead of the loads: with every SM prefetching a few
      // steps ahead the prefetches crowded the memory system and made the
      // kernel about 5 % slower (and the SMs' step rates 15 % apart).
      for (int st = 0; st < nsteps; ++st, ++ndo) {
        const int tok = t.q0 + sm.tb(st / ngroups) * step_tok;
        const int h0 = (st % ngroups) * G;
        // Q of the step into slot g & 1
        const int s = (nq.c0 + nq.c1) & 1;
        const uint32_t n = nq.bump(s);
        if (n > 0 && !(ok = mbar_wait_warp(&bars->q_empty[s], (n - 1) & 1, s_abort))) break;
        if (lane == 0) mbar_arrive_expect_tx(&bars->q_full[s], kTile3);
        __syncwarp();
        uint8_t* dq = sQ + s * kTile3;
        if (lane == 0) tma_load_4d(dq, &tq2, &bars->q_full[s], 0, h0, tok, 0);
        if (lane == 1) tma_load_3d(dq + 2 * kTile, &tq, &bars->q_full[s], 2 * kChunk, h0, tok);
        // dO of the step
        if (ndo > 0 && !(ok = mbar_wait_warp(&bars->do_empty, (ndo - 1) & 1, s_abort))) break;
        if (lane == 0) mbar_arrive_expect_tx(&bars->do_full, kTile3);
        __syncwarp();
        if (lane == 2) tma_load_4d(sDO, &tdo2, &bars->do_full, 0, h0, tok, 0);
        if (lane == 3) tma_load_3d(sDO + 2 * kTile, &tdo, &bars->do_full, 2 * kChunk, h0, tok);
      }
    }
    if (*s_abort && lane == 0) {
      if (nkv > 0) drain_wait_kv(&bars->kv_full, (nkv - 1) & 1);
      for (int s = 0; s < 2; ++s)
        if (nq.get(s) > 0) drain_wait_kv(&bars->q_full[s], (nq.get(s) - 1) & 1);
      if (ndo > 0) drain_wait_kv(&bars->do_full, (ndo - 1) & 1);
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues S^T and dP^T (they pass through SP in turn), warp 3 the
    // dV and dK accumulations.  An MMA issue blocks while the tensor pipe is
    // busy, so with one issuing thread the wait for P^T or dS^T of a step
    // would hold back the next step's S^T and dP^T (and the reverse).
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(128, 128, BF16, false, false);
      // N = d: features past the head dimension are neither multiplied nor stored
      constexpr uint32_t kIdG = idesc_f16(128, HD, BF16, false, true);
      constexpr int nk = HD / 16;  // K steps of S^T and dP^T over the features
      const uint32_t kb = smem_addr(sK), vb = smem_addr(sV), db = smem_addr(sDO);
      // A = K or V: features 0..127 in 128-byte-swizzled chunks, 128..159 in a
      // 64-byte-swizzled chunk.  B = Q or dO, three 128-byte-swizzled chunks,
      // K-major (S^T, dP^T) or MN-major (dK, dV: N = features, K = query rows).
      // Descriptors are built once; each K step adds a byte offset.
      const SDesc kA = sdesc_split(sdesc_sw128(kb, 16, 1024));
      const SDesc kT = sdesc_split(sdesc_sw64(kb + 2 * kTile));
      const SDesc vA = sdesc_split(sdesc_sw128(vb, 16, 1024));
      const SDesc vT = sdesc_split(sdesc_sw64(vb + 2 * kTile));
      const SDesc dK = sdesc_split(sdesc_sw128(db, 16, 1024));
      const SDesc dMN = sdesc_split(sdesc_sw128(db, kTile, 1024));
      // Q slot s: its descriptors differ from slot 0's by s * kTile3 in the address
      const SDesc qK0 = sdesc_split(sdesc_sw128(smem_addr(sQ), 16, 1024));
      const SDesc qMN0 = sdesc_split(sdesc_sw128(smem_addr(sQ), kTile, 1024));
      auto qslot = [](SDesc d, uint32_t gg) { return SDesc{d.lo + (gg & 1) * (kTile3 >> 4), d.hi}; };
      // D = A B^T over the 160 features (K-major A and B)
      auto mma_kmajor = [&](uint32_t d, SDesc a, SDesc at, SDesc b) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k >> 2) * kTile + (k & 3) * 32;
          if (k < nk) umma_ss_off(d, a, off, b, off, kIdS, k > 0);
        }
        if (nk > 8) {
          umma_ss_off(d, at, 0, b, 2 * kTile, kIdS, 1);
          umma_ss_off(d, at, 32, b, 2 * kTile + 32, kIdS, 1);
        }
      };
      // D (+)= X^T B over the step's 128 query rows; rows 16k..16k+15 are the
      // pair columns 448 + 32*(k/4) + 8*(k%4)
      auto mma_x = [&](uint32_t d, SDesc bmn, bool acc) {
#pragma unroll
        for (int k = 0; k < kRowsQ / 16; ++k)
          umma_ts_off(d, tmem + kColX + (k >> 2) * 32 + (k & 3) * 8, bmn, k * 2048, kIdG,
                      (acc || k > 0) ? 1u : 0u);
      };
      uint32_t g = 0;  // query steps of all earlier tiles
      int tcount = 0;
      bool ok = true;
      if (warp == 1) {
        // S^T of step gg into SP once the previous content of SP (dP^T of
        // step gg - 1) has been read
        auto issue_s = [&](uint32_t gg) -> bool {
          if (gg >= 1 && !mbar_wait(&bars->dp_read, (gg - 1) & 1, s_abort)) return false;
          if (!mbar_wait(&bars->q_full[gg & 1], (gg >> 1) & 1, s_abort)) return false;
          tc_fence_after();
          mma_kmajor(tmem + kColSP, kA, kT, qslot(qK0, gg));
          umma_commit(&bars->s_full);
          return true;
        };
        uint32_t ktake = 0;
        int item = -1;
        for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
          KTile t;
          ktile_decode<MASK>(p, item, t);
          const int nsteps = step_count(t);
          if (!(ok = mbar_wait(&bars->kv_full, tcount & 1, s_abort))) break;
          if (nsteps == 0) {  // no queries: keep every phase count
            mbar_arrive(&bars->kv_empty);
            continue;
          }
          if (!(ok = issue_s(g))) break;
          for (int st = 0; st < nsteps && ok; ++st) {
            const uint32_t gg = g + st;
            // dP^T = V dO^T over SP once S^T has been read
            if (!(ok = mbar_wait(&bars->s_read, gg & 1, s_abort))) break;
            if (!(ok = mbar_wait(&bars->do_full, gg & 1, s_abort))) break;
            tc_fence_after();
            mma_kmajor(tmem + kColSP, vA, vT, dK);
            umma_commit(&bars->dp_full);
            umma_commit(&bars->do_empty);
            // S^T of the next step over SP once dP^T has been read (this
            // product overlaps the elementwise warps' dS work)
            if (st + 1 < nsteps && !(ok = issue_s(gg + 1))) break;
          }
          if (!ok) break;
          umma_commit(&bars->kv_empty);  // K and V are read by S^T and dP^T only
          g += nsteps;
        }
      } else {
        uint32_t ktake = 0;
        int item = -1;
        for (; (ok = tile_take(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
          KTile t;
          ktile_decode<MASK>(p, item, t);
          const int nsteps = step_count(t);
          if (nsteps == 0) {  // no queries: dk = dv = 0
            if (tcount > 0 && !(ok = mbar_wait(&bars->acc_empty, (tcount - 1) & 1, s_abort)))
              break;
            mbar_arrive(&bars->acc_full);
            continue;
          }
          for (int st = 0; st < nsteps && ok; ++st) {
            const uint32_t gg = g + st;
            // dV += P^T dO (P^T is written before dP^T is read, so the dO
            // tile's arrival is not implied by p_full: wait for it here too)
            if (!(ok = mbar_wait(&bars->p_full, gg & 1, s_abort))) break;
            if (!(ok = mbar_wait(&bars->do_full, gg & 1, s_abort))) break;
            if (st == 0 && tcount > 0 &&
                !(ok = mbar_wait(&bars->acc_empty, (tcount - 1) & 1, s_abort)))
              break;
            tc_fence_after();
            mma_x(tmem + kColDV, dMN, st > 0);
            umma_commit(&bars->dv_done);
            umma_commit(&bars->do_empty);
            // dK += dS^T Q (S^T, the other reader of the Q slot, has completed)
            if (!(ok = mbar_wait(&bars->ds_full, gg & 1, s_abort))) break;
            tc_fence_after();
            mma_x(tmem + kColDK, qslot(qMN0, gg), st > 0);
            umma_commit(&bars->dk_done);
            umma_commit(&bars->q_empty[gg & 1]);
          }
          if (!ok) break;
          umma_commit(&bars->acc_full);
          g += nsteps;
        }
      }
      umma_commit(&bars->drain);
      drain_wait_kv(&bars->drain, 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ column scalars
    // Lane u of warp 2 stages columns u, u + 32, u + 64 and u + 96 of every
    // query step: the bias coefficients into a two-deep ring, D into one
    // buffer.  The global loads of a step are issued two steps before it is
    // staged.
    const int u = lane;
    constexpr bool masked = MASK;
    const int lgGs = __ffs(G) - 1;  // G is a power of two
    struct Pos {  // a (key tile, query step) of this CTA: step st is (tb, hg)
      int item, st, tb, hg, nsteps;
      KTile t;
      StepMap sm;
    };
    struct Vals {
      float lse[4], sl2[4], D[4];
    };
    // the warp reads the tile stream as far ahead as its lookahead needs;
    // a position past the end has item = ntiles
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
        q.sm = step_map(q.t, step_tok, kBandLast);
        q.tb = q.sm.tb(0);
        if (q.nsteps > 0) return;
        q.item = take();
      }
    };
    auto next = [&](const Pos& q) {
      Pos n = q;
      if (q.item >= ntiles) return n;
      if (++n.st < n.nsteps) {
        n.hg = n.st % ngroups;
        n.tb = n.sm.tb(n.st / ngroups);
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
        // bias(r) = -sl2 * |prel - r| + nl2 = a + m * r for every key r of the
        // tile when prel >= 127 (m = sl2) or prel <= 0 (m = -sl2).  In every
        // case nl2 = a + m * prel, and the general form recovers sl2 from m
        // and the sign of prel (a slope may be negative).
        const bool right = prel <= 0.f;  // every key at or right of i
        const float m = right ? -sl2 : sl2;
        cols->a[b][lc] = fmaf(-m, prel, nl2);
        cols->m[b][lc] = m;
        straddle |= !right && prel < static_cast<float>(kKeys - 1) && i < q0.t.Lq;
        // the mask is applied per key only on the steps it cuts for some column
        if (masked && i < q0.t.Lq)
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
      // D of the step, once every elementwise warp is done with the previous one
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
    const LogitMap lm = make_logit_map(p);
    const bool capped = CAP || lm.capped;
    constexpr bool masked = MASK;
    const int wl = p.wl;
    const int wr = right_window(p);
    const int lgG = __ffs(G) - 1;  // G is a power of two
    uint32_t g = 0;
    int tcount = 0;
    bool ok = true;
    uint32_t ktake = 0;
    int item = -1;
    for (; (ok = tile_take_warp(&bars->ring, ktake, &item, s_abort)) && item >= 0; ++tcount) {
      KTile t;
      ktile_decode<MASK>(p, item, t);
      const int nsteps = step_count(t);
      const uint64_t dkb =
          (DROP && !DMASK) ? splitmix64(p.drop_seed ^ static_cast<uint64_t>(t.b)) : 0;
      // stored keep mask (written by the mask kernel): step st's block is the
      // tile's first one plus st rows of key-tile blocks.  Of each 64-bit word
      // (64 keys of one column) this warp needs the 32-bit half of its 32
      // keys; the halves of step st + 1 are loaded during step st, once P^T
      // of step st has gone out (their memory latency then hides behind the
      // dP^T and dS work)
      const StepMap sm = step_map(t, step_tok, kBandLast);
      const uint32_t* mbase = nullptr;
      int mstep = 0;  // 32-bit words from one block (token block, head group) to the next
      uint32_t mw0 = 0, mw1 = 0;
      // the mask words of step st: its block relative to the tile's first
      auto mwords = [&](int s_) {
        return mbase + static_cast<int64_t>((sm.tb(s_ / ngroups) - t.tb0) * ngroups +
                                            s_ % ngroups) * mstep;
      };
      if (DMASK && nsteps > 0) {
        mbase = reinterpret_cast<const uint32_t*>(
                    drop_mask_block(p, t.b, t.Lk, t.tb0, 0, t.key / kKeys) +
                    (quad >> 1) * kRowsQ + half * 64 + lane) +
                (quad & 1);
        mstep = (t.Lk + kKeys - 1) / kKeys * (2 * kMaskBlockWords);
        mw0 = __ldg(mwords(0));
        mw1 = __ldg(mwords(0) + 64);
      }
      // one step of the walk; K = 0: a step outside the band (one-sided element
      // code only), 1: a band step (general code only), 2: with a mask, either,
      // by the staging warp's flag
      auto step = [&](int st, auto kind) -> bool {
        constexpr int K = decltype(kind)::value;
        const uint32_t gg = g + st;
        const int b = gg & 1;
        const int tb = sm.tb(st / ngroups);
        // dropout keep bits of this step's 64 columns (query token, head) for
        // this thread's key, hashed while S^T is computed
        const int dtok0 = DROP ? tb * step_tok : 0;
        uint64_t kbits = 0;
        if (DMASK) {
          // stored keep mask: the words of this half's 64 columns hold 64
          // keys each; this warp's 32 keys are one 32-bit half of them, turned
          // from one column per lane into one key per lane
          kbits = (static_cast<uint64_t>(bit_transpose32(mw1)) << 32) | bit_transpose32(mw0);
        } else if (DROP) {
          // one hash serves the four keys 4m .. 4m + 3, held by four
          // neighbouring lanes (key = t.key + r): each lane hashes 16 of the
          // 64 columns (c = 4k + f, f = its key mod 4) for the group, and
          // column c's hash is then read from lane f = c mod 4 of the group
          const int dh0 = p.head0 + (st % ngroups) * G;
          const int f = lane & 3;
          const int m = (t.key + r) >> 2;
          const int src0 = lane & ~3;
          int t_tok = -1;            // token of the threshold in T (per-token rates)
          uint32_t T = p.drop_T;
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {  // columns 32 bb .. 32 bb + 31
            uint32_t hlo[8], hhi[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int lc = half * 64 + 32 * bb + 4 * k + f;
              const int it = dtok0 + (lc >> lgG);
              const uint64_t x = drop_hash(dkb, drop_hi(dh0 + (lc & (G - 1)), it), m);
              hlo[k] = static_cast<uint32_t>(x);
              hhi[k] = static_cast<uint32_t>(x >> 32);
            }
#pragma unroll
            for (int cc = 0; cc < 32; ++cc) {
              const int c = 32 * bb + cc;
              const uint32_t lo = __shfl_sync(0xffffffffu, hlo[cc >> 2], src0 | (c & 3));
              const uint32_t hw = __shfl_sync(0xffffffffu, hhi[cc >> 2], src0 | (c & 3));
              const uint32_t u = ((f < 2 ? lo : hw) >> (16 * (f & 1))) & 0xFFFFu;
              const int it = dtok0 + ((half * 64 + c) >> lgG);
              if (DTAB && it != t_tok && it < t.Lq) {  // a new token every G columns
                T = __ldg(p.drop_tab + t.q0 + it).x;
                t_tok = it;
              }
              kbits |= static_cast<uint64_t>(it < t.Lq && u >= T) << c;
            }
          }
        }
        // S^T: read it and release SP for dP^T
        if (!(ok = mbar_wait_warp(&bars->s_full, gg & 1, s_abort))) return false;
        tc_fence_after();
        const uint32_t spbuf = tmem + kColSP + half * 64 + lane_addr;
        uint64_t t2[32];  // column pairs: S, then tanh, then -P (1 - tanh^2)
        {
          float x[64];
          tmem_ld32(spbuf, *reinterpret_cast<float(*)[32]>(x));
          tmem_ld32(spbuf + 32, *reinterpret_cast<float(*)[32]>(x + 32));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) t2[i] = f2_make(x[2 * i], x[2 * i + 1]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_read);
        const uint64_t is2 = f2_make(lm.in_scale, lm.in_scale);
        const uint64_t os2 = f2_make(lm.out_scale, lm.out_scale);
        const uint64_t m12 = f2_make(-1.f, -1.f);
        if (capped) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint64_t v = f2_mul(t2[i], is2);
            t2[i] = f2_make(tanh_approx(f2_lo(v)), tanh_approx(f2_hi(v)));
          }
        }
        // P = exp2(c*log2e*tanh(sigma*x/c) + bias) per group of 4 columns, with
        // the base-2 bias -slope2 * |i + Lk - Lq - j| - lse2 formed from the
        // staged column scalars (a + m * j when the tile lies on one side of
        // every column's aligned key)
        if (!(ok = mbar_wait_warp(&bars->am_full[b], (gg >> 1) & 1, s_abort))) return false;
        const float4* pa = reinterpret_cast<const float4*>(cols->a[b] + half * 64);
        const float4* pm = reinterpret_cast<const float4*>(cols->m[b] + half * 64);
        uint32_t pk[32];
        // dropout: P^T for dV is P * keep * scale and dS uses keep * scale * dP
        // (keep bits hashed at the start of the step)
        auto dscale = [&](int c) -> float {  // the scale of column c (its query token)
          if (!DTAB) return p.drop_scale;
          // per-token rates: loaded where used (a volatile load is not hoisted
          // ahead of the unrolled element loop, which would hold 64 of them)
          const int it = dtok0 + ((half * 64 + c) >> lgG);
          const volatile uint32_t* e =
              reinterpret_cast<const volatile uint32_t*>(p.drop_tab + t.q0 + it);
          return it < t.Lq ? __uint_as_float(e[1]) : 0.f;
        };
        auto pack_p = [&](int c, float a, float bb) -> uint32_t {  // columns c, c + 1
          if (DROP) {
            a = ((kbits >> c) & 1) ? a * dscale(c) : 0.f;
            bb = ((kbits >> (c + 1)) & 1) ? bb * dscale(c + 1) : 0.f;
          }
          return Pack<BF16>::two(a, bb);
        };
        // columns col .. col + 3, held in pairs 2 s and 2 s + 1 of t2 and pk
        auto p_group = [&](int s, int col, float b0, float b1, float b2, float b3) {
          const uint64_t z0 = f2_fma(t2[2 * s], capped ? os2 : is2, f2_make(b0, b1));
          const uint64_t z1 = f2_fma(t2[2 * s + 1], capped ? os2 : is2, f2_make(b2, b3));
          const uint64_t p0 = f2_make(ex2_approx(f2_lo(z0)), ex2_approx(f2_hi(z0)));
          const uint64_t p1 = f2_make(ex2_approx(f2_lo(z1)), ex2_approx(f2_hi(z1)));
          pk[2 * s] = pack_p(col, f2_lo(p0), f2_hi(p0));
          pk[2 * s + 1] = pack_p(col + 2, f2_lo(p1), f2_hi(p1));
          // -P (1 - tanh^2) = P (tanh^2 - 1); dS = this * (D - dP)
          t2[2 * s] = capped ? f2_mul(p0, f2_fma(t2[2 * s], t2[2 * s], m12)) : f2_mul(p0, m12);
          t2[2 * s + 1] =
              capped ? f2_mul(p1, f2_fma(t2[2 * s + 1], t2[2 * s + 1], m12)) : f2_mul(p1, m12);
        };
        // K = 0 steps are one-sided by the walk's order; in the band (and
        // with a mask) the staging warp's flag tells
        const bool gen = K != 0 && (cols->general[b][0] | cols->general[b][1]) != 0;
        if (!gen) {
          // one-sided tile: in three passes (all exponents, all exp2, then
          // the packing and chain factors), so the 64 MUFU operations issue
          // back to back
          const uint64_t r2 = f2_make(rf, rf);
          uint64_t z[32];
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const float4 a4 = pa[q4], m4 = pm[q4];
            const uint64_t b0 = f2_fma(f2_make(m4.x, m4.y), r2, f2_make(a4.x, a4.y));
            const uint64_t b1 = f2_fma(f2_make(m4.z, m4.w), r2, f2_make(a4.z, a4.w));
            z[2 * q4] = f2_fma(t2[2 * q4], capped ? os2 : is2, b0);
            z[2 * q4 + 1] = f2_fma(t2[2 * q4 + 1], capped ? os2 : is2, b1);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            z[i] = f2_make(ex2_approx(f2_lo(z[i])), ex2_approx(f2_hi(z[i])));
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            pk[i] = pack_p(2 * i, f2_lo(z[i]), f2_hi(z[i]));
            // -P (1 - tanh^2) = P (tanh^2 - 1); dS = this * (D - dP)
            t2[i] = capped ? f2_mul(z[i], f2_fma(t2[i], t2[i], m12)) : f2_mul(z[i], m12);
          }
        } else if (K == 1) {
          // a general band step (no mask): the general bias per element, then
          // the same exp2 and packing passes as a one-sided step
          const int tok0 = tb * step_tok;
          const int off = t.Lk - t.Lq - t.key;
          uint64_t z[32];
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const float4 a4 = pa[q4], m4 = pm[q4];
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
            float bv[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int c = half * 64 + q4 * 4 + v;
              const float prel = static_cast<float>(tok0 + (c >> lgG) + off);
              const float sl = prel <= 0.f ? -mv[v] : mv[v];
              bv[v] = fmaf(-sl, fabsf(prel - rf), fmaf(mv[v], prel, av[v]));
            }
            z[2 * q4] = f2_fma(t2[2 * q4], capped ? os2 : is2, f2_make(bv[0], bv[1]));
            z[2 * q4 + 1] = f2_fma(t2[2 * q4 + 1], capped ? os2 : is2, f2_make(bv[2], bv[3]));
          }
#pragma unroll
          for (int i = 0; i < 32; ++i)
            z[i] = f2_make(ex2_approx(f2_lo(z[i])), ex2_approx(f2_hi(z[i])));
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            pk[i] = pack_p(2 * i, f2_lo(z[i]), f2_hi(z[i]));
            t2[i] = capped ? f2_mul(z[i], f2_fma(t2[i], t2[i], m12)) : f2_mul(z[i], m12);
          }
        } else {
          // some column's aligned key lies inside the tile, or a mask applies:
          // prel = i + Lk - Lq - key0 of column c is tok0 + c / G + off,
          // a + m * prel = -lse2, and the column's slope2 is m where its
          // scalars were staged for keys left of prel (prel > 0), else -m
          const int tok0 = tb * step_tok;
          const int off = t.Lk - t.Lq - t.key;
#pragma unroll 1
          for (int q4 = 0; q4 < 16; ++q4) {
            const float4 a4 = pa[q4], m4 = pm[q4];
            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
            const float mv[4] = {m4.x, m4.y, m4.z, m4.w};
            float bv[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int c = half * 64 + q4 * 4 + v;
              const float prel = static_cast<float>(tok0 + (c >> lgG) + off);
              const float sl = prel <= 0.f ? -mv[v] : mv[v];
              bv[v] = fmaf(-sl, fabsf(prel - rf), fmaf(mv[v], prel, av[v]));
              if (masked) {
                const bool adm = (wl < 0 || rf >= prel - static_cast<float>(wl)) &&
                                 (wr < 0 || rf <= prel + static_cast<float>(wr));
                bv[v] = adm ? bv[v] : -INFINITY;
              }
            }
            // The group being processed is always pairs 0 and 1: the pair
            // arrays turn by one group per iteration (16 turns bring them back
            // into place), so the loop body indexes them with constants only
            // and they stay in registers.  This keeps the code of the rare
            // general steps small: the hot loop's instructions then fit the
            // instruction caches better.
            p_group(0, 4 * q4, bv[0], bv[1], bv[2], bv[3]);
            const uint64_t s0 = t2[0], s1 = t2[1];
            const uint32_t k0 = pk[0], k1 = pk[1];
#pragma unroll
            for (int i = 0; i < 30; ++i) {
              t2[i] = t2[i + 2];
              pk[i] = pk[i + 2];
            }
            t2[30] = s0;
            t2[31] = s1;
            pk[30] = k0;
            pk[31] = k1;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->am_empty[b]);
        // P^T pairs: this half's 64 columns -> 32 pair columns at 448 + 32*half,
        // once dK of the previous step has read X
        if (gg >= 1 && !(ok = mbar_wait_warp(&bars->dk_done, (gg - 1) & 1, s_abort))) return false;
        tc_fence_after();
        const uint32_t xbuf = tmem + kColX + half * 32 + lane_addr;
        tmem_st16(xbuf, *reinterpret_cast<uint32_t(*)[16]>(pk));
        tmem_st16(xbuf + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
        if (DMASK && st + 1 < nsteps) {  // the next step's keep-mask halves
          const uint32_t* nx = mwords(st + 1);
          mw0 = __ldg(nx);
          mw1 = __ldg(nx + 64);
        }
        // dP^T: read it and release SP for S^T of the next step (P^T went out
        // first, so dV, and with it the release of the dO slot, starts early)
        if (!(ok = mbar_wait_warp(&bars->dp_full, gg & 1, s_abort))) return false;
        tc_fence_after();
        float d[64];
        tmem_ld32(spbuf, *reinterpret_cast<float(*)[32]>(d));
        tmem_ld32(spbuf + 32, *reinterpret_cast<float(*)[32]>(d + 32));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dp_read);
        if (DROP) {
#pragma unroll
          for (int c = 0; c < 64; ++c) d[c] = ((kbits >> c) & 1) ? d[c] * dscale(c) : 0.f;
        }
        // dS^T = P (1 - tanh^2) (dP - D) = t2 (D - dP), D per group of 4 columns
        if (!(ok = mbar_wait_warp(&bars->d_full, gg & 1, s_abort))) return false;
        {
          const float4* pd = reinterpret_cast<const float4*>(cols->D + half * 64);
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            const float4 d4 = pd[q4];
            const uint64_t e0 = f2_fma(f2_make(d[4 * q4], d[4 * q4 + 1]), m12, f2_make(d4.x, d4.y));
            const uint64_t e1 = f2_fma(f2_make(d[4 * q4 + 2], d[4 * q4 + 3]), m12, f2_make(d4.z, d4.w));
            const uint64_t v0 = f2_mul(t2[2 * q4], e0);
            const uint64_t v1 = f2_mul(t2[2 * q4 + 1], e1);
            pk[2 * q4] = Pack<BF16>::two(f2_lo(v0), f2_hi(v0));
            pk[2 * q4 + 1] = Pack<BF16>::two(f2_lo(v1), f2_hi(v1));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->d_empty);
        // dS^T pairs over P^T once dV has read it
        if (!(ok = mbar_wait_warp(&bars->dv_done, gg & 1, s_abort))) return false;
        tc_fence_after();
        tmem_st16(xbuf, *reinterpret_cast<uint32_t(*)[16]>(pk));
        tmem_st16(xbuf + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->ds_full);
        return true;
      };
      if (kBandLast && !MASK) {
        const int n_one = (sm.nA + sm.nC) * ngroups;
        int st = 0;
        for (; st < n_one && ok; ++st) ok = step(st, std::integral_constant<int, 0>{});
        for (; st < nsteps && ok; ++st) ok = step(st, std::integral_constant<int, 1>{});
      } else {
        for (int st = 0; st < nsteps && ok; ++st) ok = step(st, std::integral_constant<int, 2>{});
      }
      if (!ok) break;
      g += nsteps;
      // ---- epilogue: half 0 writes dv = dV, half 1 writes dk = sigma * dK
      if (!(ok = mbar_wait_warp(&bars->acc_full, tcount & 1, s_abort))) break;
      tc_fence_after();
      const int j = t.key + r;
      const bool key_valid = j < t.Lk;
      const float scale = half ? p.sigma : 1.f;
      uint16_t* row = half ? static_cast<uint16_t*>(p.dk) + static_cast<int64_t>(t.k0 + j) * p.dk_ts
                           : static_cast<uint16_t*>(p.dv) + static_cast<int64_t>(t.k0 + j) * p.dv_ts;
      const uint32_t acc = tmem + (half ? kColDK : kColDV) + lane_addr;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        float a[32];
        tmem_ld32(acc + c * 32, a);
        tmem_wait_ld();
        if (key_valid) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float w8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w8[i] = nsteps > 0 ? a[8 * v + i] * scale : 0.f;
            *reinterpret_cast<uint4*>(row + c * 32 + v * 8) = pack8<BF16>(w8);
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

}  // namespace attn
