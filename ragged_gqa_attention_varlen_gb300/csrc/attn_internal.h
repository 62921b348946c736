// attn_internal.h -- parameters and launch entry points shared by the CUDA
// translation units of the library (not part of the public ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

constexpr int kHeadDim = 160;
constexpr int kChunk = 64;        // elements per 128-byte swizzled row
constexpr int kChunks = 3;        // 64-wide chunks covering 160 features
constexpr int kRowsQ = 128;       // query rows per forward / dq tile
constexpr int kKeys = 128;        // keys per tile
constexpr int kThreads = 384;     // warpgroup 0: loads + MMA issue; warpgroups 1-2: elementwise
// Register split (setmaxnreg): launched at 168 per thread (384 x 168 = 64512);
// warpgroup 0 gives registers up to the two elementwise warpgroups.
constexpr int kRegsLow = 104;
constexpr int kRegsHigh = 200;
static_assert(4 * kRegsLow + 8 * kRegsHigh <= 12 * 168, "register split exceeds the launch");

// Query rows of a tile are (token, head) pairs: G consecutive heads of one
// head group times 128/G consecutive tokens, row r = token*G + head.
//
// With Hkv > 1 K/V heads, query heads g*R .. g*R+R-1 (R = Hq/Hkv) read K/V
// head g, and each such group runs as its own one-K/V-head problem: Params
// then describe the group (Hq = R, every pointer offset to the group's first
// head), with lse/D rows still strided by the whole call's head count.
struct Params {
  int dtype;  // 0 fp16, 1 bf16
  int B, Hq, G;
  int d;      // head dimension: 160, 128 or 64 (the kernels' tiles hold 160
              // features; the TMA maps fill features >= d with zeros and
              // every other load or store stops at d)
  int64_t total_q, total_k;
  // outputs (element strides)
  void* out;
  int64_t out_ts, out_hs;
  void* dq;
  int64_t dq_ts, dq_hs;
  void* dk;
  int64_t dk_ts, dk_hs;
  void* dv;
  int64_t dv_ts, dv_hs;
  int Hkv;  // K/V heads of the call (the preprocess zeroes dk/dv rows of all of them)
  // inputs read outside TMA
  const void* outp;  // = out, read back by the preprocess kernel
  const void* dout;
  int64_t do_ts, do_hs;
  const void* q;  // read row by row by the dq kernel (into TMEM)
  int64_t q_ts, q_hs;
  const int32_t* cu_q;
  const int32_t* cu_k;
  const float* slopes;  // may be null
  int64_t slopes_bs;
  int causal, wl, wr;
  float softcap;  // <= 0: no cap
  float sigma;    // scale_multiplier / sqrt(d)
  float* lse;     // [total_q, lse_rs]
  float* Dbuf;    // [total_q, lse_rs]
  int64_t lse_rs; // row stride of lse and D: every query head of the call
  // counter-based dropout ("ragged flash attention gradient recompute", "Root
  // causes addressed"): element (b, h, i, j) is kept when the 16-bit field
  // j mod 4 of splitmix64(splitmix64(seed ^ b) ^ (h << 48 | i << 24 | j / 4))
  // reaches the rate's threshold T = rate * 2^16, and then scaled by
  // 1 / (1 - rate)
  int dropout;
  uint64_t drop_seed;
  uint32_t drop_T;           // threshold of the call's rate (when drop_tab is null)
  float drop_scale;
  const float* drop_rates;   // per query token [total_q], or null
  uint2* drop_tab;           // per query token (T, scale bits), made by the schedule kernel
  int head0;                 // first query head of this K/V head group (hash input h)
  // stored keep bits (null: the backward regenerates them from the hash):
  // written by the forward, read by the backward kernels; layout below
  uint8_t* drop_mask;
  uint64_t drop_mask_bytes;
  int32_t* status;
  int32_t* counters;  // [3]: fwd, dkdv, dq tile counters (of this K/V head group)
  int ncounters;      // counters the schedule kernel resets (every group's)
  int32_t* sched;     // schedule arrays, see sched.cu
  // sigmoid gate ("Pairwise-Gated Attention Engine", "Why it is hard"):
  // G_ij = sigmoid(qg_i . kg_j / sqrt(R)) scales the normalised weight
  const void* qg;     // [total_q, Hq, R] (null: no gate)
  int64_t qg_ts, qg_hs;
  void* dqg;
  int64_t dqg_ts, dqg_hs;
  void* dkg;          // [total_k, Hkv, R]
  int64_t dkg_ts, dkg_hs;
  int R;              // gate width (32 or 64)
  float gscale;       // 1 / sqrt(R)
};

// 16-byte units (8 features) of a row's features [80*half, 80*half + 80)
// that lie below the head dimension.
__host__ __device__ constexpr int feature_units(int d, int half) {
  return (d - 80 * half) / 8 < 0 ? 0 : ((d - 80 * half) / 8 > 10 ? 10 : (d - 80 * half) / 8);
}

// The call has a causal or window mask (selects the masked kernel instances).
inline bool masked_call(const Params& p) { return p.causal || p.wl >= 0 || p.wr >= 0; }

// Layout of the schedule arrays inside Params::sched (all int32):
//   [0, B)          fwd/dq sequence order (longest key range first)
//   [B, 2B+1)       fwd/dq item prefix over that order
//   [2B+1, 3B+1)    dk/dv sequence order (longest query range first)
//   [3B+1, 4B+2)    dk/dv item prefix over that order (key tiles that some
//                   query may attend to: a contiguous run per sequence)
//   [4B+2, 5B+2)    first such key tile of each order position
inline int sched_words(int B) { return 5 * B + 2; }

// Keep-mask layout: a header of B + 1 int32 (the prefix over the sequences,
// in batch order, of their (query tile, key tile) blocks), padded to 256
// bytes, then K/V head group g's blocks at g * total, and within a group
// sequence b's block (tb, hg, kt) -- query token block tb, head group hg, key
// tile kt -- at prefix[b] + (tb * (Hq/G) + hg) * ceil(Lk/128) + kt.  A block
// is 256 words: word kh * 128 + r holds the keep bits of query row r of the
// tile (token r / G, head r % G) for keys 64 kh .. 64 kh + 63 of the key tile
// (bit c for key 64 kh + c), zero for rows past the sequence.
constexpr int kMaskBlockWords = 2 * kRowsQ;  // 64-bit words per block (2 KB)
__host__ __device__ constexpr uint64_t drop_mask_header(int B) {
  return (4ull * (static_cast<uint64_t>(B) + 1) + 255) / 256 * 256;
}

// Workspace bytes a call uses (host.cu): the status word, tile counters,
// schedule and D, plus the per-token dropout rate table when `rate_table`.
// attn_varlen_fvjp_workspace_size reports the size with the table.
size_t workspace_bytes_needed(int B, int Hq, int64_t total_q, bool rate_table);

cudaError_t launch_sched(const Params& p, cudaStream_t s);
// The stored keep mask of a dropout call with a mask buffer (every group).
cudaError_t launch_mask(const Params& p, cudaStream_t s);
cudaError_t launch_fwd(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tqt,
                       const CUtensorMap& tk2, const CUtensorMap& tkt, const CUtensorMap& tv2,
                       const CUtensorMap& tv, int grid, cudaStream_t s);
cudaError_t launch_preprocess(const Params& p, cudaStream_t s);
// Tensor maps: *2 load feature chunks 0-1 of a tile in one box; tq/tdo load
// chunk 2 (features 128..191, the part past 159 filled with zeros); tkt/tvt
// load features 128..159 with the 64-byte swizzle.
cudaError_t launch_dkdv(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tq,
                        const CUtensorMap& tdo2, const CUtensorMap& tdo, const CUtensorMap& tk2,
                        const CUtensorMap& tkt, const CUtensorMap& tv2, const CUtensorMap& tvt,
                        int grid, cudaStream_t s);
cudaError_t launch_dkdv_drop(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tq,
                             const CUtensorMap& tdo2, const CUtensorMap& tdo,
                             const CUtensorMap& tk2, const CUtensorMap& tkt,
                             const CUtensorMap& tv2, const CUtensorMap& tvt,
                             int grid, cudaStream_t s);
cudaError_t launch_dkdv_dmask(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tq,
                              const CUtensorMap& tdo2, const CUtensorMap& tdo,
                              const CUtensorMap& tk2, const CUtensorMap& tkt,
                              const CUtensorMap& tv2, const CUtensorMap& tvt,
                              int grid, cudaStream_t s);
cudaError_t launch_dq(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tqt,
                      const CUtensorMap& tdo2, const CUtensorMap& tdot, const CUtensorMap& tk2,
                      const CUtensorMap& tk, const CUtensorMap& tv2, const CUtensorMap& tvt,
                      int grid, bool overlap, cudaStream_t s);
// Gated kernels (gate.cu): head dimension 64 or 128, gate width padded to
// 64 by the tensor maps.  Maps: *2 cover a whole 128-row tile (both 64-wide
// chunks when d = 128), *g the gate projections.
cudaError_t launch_gate_fwd(const Params& p, const CUtensorMap& tq, const CUtensorMap& tqg,
                            const CUtensorMap& tk, const CUtensorMap& tkg, const CUtensorMap& tv,
                            int grid, cudaStream_t s);
cudaError_t launch_gate_dq(const Params& p, const CUtensorMap& tq, const CUtensorMap& tqg,
                           const CUtensorMap& tdo, const CUtensorMap& tk, const CUtensorMap& tkg,
                           const CUtensorMap& tv, int grid, cudaStream_t s);
cudaError_t launch_gate_dkdv(const Params& p, const CUtensorMap& tq, const CUtensorMap& tqg,
                             const CUtensorMap& tdo, const CUtensorMap& tk, const CUtensorMap& tkg,
                             const CUtensorMap& tv, int grid, cudaStream_t s);

cudaError_t launch_zero_fill(void* base, int64_t T, int H, int64_t ts, int64_t hs, int d,
                             cudaStream_t s);
cudaError_t launch_fill_f32(float* base, int64_t n, float value, cudaStream_t s);

}  // namespace attn
