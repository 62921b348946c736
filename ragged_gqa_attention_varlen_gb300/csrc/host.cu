// host.cu -- the C ABI: argument validation, TMA tensor-map encoding and the
// launch sequence of one fused forward + VJP call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>

#include "../../include/attn_varlen.h"
#include "attn_internal.h"
#include "common.cuh"

namespace attn {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load();
  if (f) return f;
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  f = reinterpret_cast<EncodeTiledFn>(ptr);
  fn.store(f);
  return f;
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Workspace layout: [status + counters | schedule | D].
struct WsLayout {
  size_t status, counters, sched, dbuf, droptab, total;
};

// Counters: three per K/V head group, and Hkv <= Hq.
WsLayout ws_layout(int B, int Hq, int64_t total_q) {
  WsLayout w;
  w.status = 0;
  w.counters = 16;
  w.sched = align_up(w.counters + sizeof(int32_t) * 3 * static_cast<size_t>(Hq < 2 ? 2 : Hq));
  w.dbuf = w.sched + align_up(sizeof(int32_t) * static_cast<size_t>(sched_words(B)));
  w.droptab = w.dbuf + align_up(sizeof(float) * static_cast<size_t>(total_q) * Hq);
  w.total = w.droptab + align_up(sizeof(uint2) * static_cast<size_t>(total_q));
  return w;
}

}  // namespace

// Bytes of workspace a call uses: everything up to the per-token dropout
// rate table, plus the table when the call has per-token rates.
size_t workspace_bytes_needed(int B, int Hq, int64_t total_q, bool rate_table) {
  const WsLayout w = ws_layout(B, Hq, total_q);
  return rate_table ? w.total : w.droptab;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_ok(int64_t s) { return s > 0 && (s % 8) == 0; }

// Every map's feature extent is the head dimension d (160, 128 or 64); the
// kernels' tiles always span 160 features, and a box part past d is filled
// with zeros by the TMA unit (it contributes nothing to any product).
//
// [T, H, d] view -> 3-D map (feature, head, token) with a box of
// 64 features x G heads x (rows/G) tokens and the 128-byte swizzle, or (tail)
// 32 features (128..159) with the 64-byte swizzle.
bool encode_q(CUtensorMap* m, int dtype, int d, const void* base, int64_t T, int H, int64_t ts,
              int64_t hs, int G, int rows, bool tail = false) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(hs) * 2, static_cast<cuuint64_t>(ts) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(tail ? kHeadDim - 2 * kChunk : kChunk),
                       static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(rows / G)};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     tail ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T, d] view of one K/V head -> 2-D map (feature, token), box 64 x 128 keys
// with the 128-byte swizzle, or (tail) 32 x 128 with the 64-byte swizzle for
// features 128..159.
bool encode_kv(CUtensorMap* m, int dtype, int d, const void* base, int64_t T, int64_t ts,
               bool tail = false) {
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(T)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ts) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(tail ? kHeadDim - 2 * kChunk : kChunk),
                       static_cast<cuuint32_t>(kKeys)};
  cuuint32_t estr[2] = {1, 1};
  return encode_fn()(m, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     tail ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same views with features 0..127 as two 64-feature chunks along an
// outer axis (stride 128 bytes): one box then loads both 128-byte-swizzled
// chunks of a tile, in the layout of two separate chunk boxes (chunk c at
// c * 16 KB).  A TMA operation costs about the same time whatever its size,
// so fewer, larger boxes raise the load rate.  With d = 64 the chunk axis has
// extent 1, so the second chunk of the box reads as zeros.
cuuint64_t chunk_count(int d) { return d >= 2 * kChunk ? 2 : 1; }

bool encode_q_pair(CUtensorMap* m, int dtype, int d, const void* base, int64_t T, int H,
                   int64_t ts, int64_t hs, int G, int rows) {
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(kChunk), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(T), chunk_count(d)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(hs) * 2, static_cast<cuuint64_t>(ts) * 2,
                           static_cast<cuuint64_t>(kChunk) * 2};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(kChunk), static_cast<cuuint32_t>(G),
                       static_cast<cuuint32_t>(rows / G), 2};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode_fn()(m, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_kv_pair(CUtensorMap* m, int dtype, int d, const void* base, int64_t T,
                    int64_t ts) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kChunk), static_cast<cuuint64_t>(T),
                        chunk_count(d)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ts) * 2, static_cast<cuuint64_t>(kChunk) * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kChunk), static_cast<cuuint32_t>(kKeys), 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode_fn()(m, dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     3, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Events of the timing hook (one-shot, per host thread).
thread_local cudaEvent_t g_events[6];
thread_local int g_nevents = 0;

int head_group(int Hq) {
  int g = 16;
  while (Hq % g) g >>= 1;
  return g;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" size_t attn_varlen_fvjp_workspace_size(int B, int Hq, int64_t total_q,
                                                  int64_t total_k) {
  (void)total_k;
  if (B < 0 || Hq <= 0 || total_q < 0) return 0;
  return ws_layout(B, Hq, total_q).total;
}

extern "C" int attn_varlen_launch_count(int mode, int B, int Hq, int Hkv, int64_t total_q,
                                        int64_t total_k) {
  (void)B;
  (void)Hq;
  const bool fwd = (mode & 1) != 0, bwd = (mode & 2) != 0;
  if (Hkv < 1 || (!fwd && !bwd)) return 0;
  if (total_q == 0 && total_k == 0) return 0;
  if (total_q == 0) return bwd ? 2 : 0;               // dk, dv zero fills
  if (total_k == 0) return (fwd ? 2 : 0) + (bwd ? 1 : 0);  // out + lse fills; dq fill
  // schedule; a forward per K/V head group; preprocess, dk/dv and dq per group
  return 1 + (fwd ? Hkv : 0) + (bwd ? 1 + 2 * Hkv : 0);
}

extern "C" int attn_varlen_fvjp_launch_count(int B, int Hq, int64_t total_q, int64_t total_k) {
  return attn_varlen_launch_count(3, B, Hq, 1, total_q, total_k);
}

extern "C" attn_status attn_varlen_fvjp_record_events(void* const* events, int n) {
  if (n == 0) {
    g_nevents = 0;
    return ATTN_OK;
  }
  if (n != 6 || !events) return ATTN_ERR_INVALID;
  for (int i = 0; i < 6; ++i) g_events[i] = static_cast<cudaEvent_t>(events[i]);
  g_nevents = 6;
  return ATTN_OK;
}

extern "C" const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_ALIGNMENT: return "pointer or stride not aligned for TMA (16 B / 8 elements)";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_DEVICE_STATUS: return "device reported an error in the status word";
    case ATTN_ERR_TIMEOUT: return "a bounded device wait ran out";
    case ATTN_ERR_SCRATCH_LIMIT:
      return "problem needs more than the no-allocation entry point's fixed scratch";
  }
  return "unknown status";
}

namespace {
constexpr int kModeFwd = 1;  // out, lse
constexpr int kModeBwd = 2;  // dq, dk, dv from out and lse

// Dropout arguments of a call (off by default).
struct Dropout {
  bool on = false;
  uint64_t seed = 0;
  float rate = 0.f;
  const float* rates = nullptr;  // per query token, device
  void* mask = nullptr;          // stored keep bits (the _mask entry points), device
  size_t mask_bytes = 0;
  bool mask_call = false;        // a _mask entry point: the mask must be given
};

// The three entry points share one body: host-side validation, the tensor
// maps, and the launches of the requested passes.
attn_status run_call(
    int mode, attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts, int64_t do_hs,
    const int32_t* cu_q, const int32_t* cu_k, const float* alibi_slopes,
    int64_t slopes_batch_stride, int causal, int window_left, int window_right, float softcap,
    float scale_multiplier, void* out, int64_t out_ts, int64_t out_hs, void* dq, int64_t dq_ts,
    int64_t dq_hs, void* dk, int64_t dk_ts, int64_t dk_hs, void* dv, int64_t dv_ts,
    int64_t dv_hs, float* lse, void* workspace, size_t workspace_bytes, int32_t* device_status,
    void* stream_ptr, const Dropout& drop = Dropout()) {
  const bool fwd = (mode & kModeFwd) != 0, bwd = (mode & kModeBwd) != 0;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  // ---- host-side validation (nothing is enqueued on failure)
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
  if (B < 0 || Hq <= 0 || total_q < 0 || total_k < 0) return ATTN_ERR_INVALID;
  if (head_dim != 160 && head_dim != 128 && head_dim != 64) return ATTN_ERR_UNSUPPORTED;
  if (drop.on && !(drop.rate == drop.rate)) return ATTN_ERR_INVALID;
  if (drop.mask_call) {
    if (!drop.mask || drop.mask_bytes < drop_mask_header(B)) return ATTN_ERR_INVALID;
    if (reinterpret_cast<uintptr_t>(drop.mask) & 255u) return ATTN_ERR_ALIGNMENT;
  }
  if (Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID;
  if (B > ATTN_MAX_BATCH) return ATTN_ERR_UNSUPPORTED;
  if (total_q > INT32_MAX || total_k > INT32_MAX) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 && (total_q != 0 || total_k != 0)) return ATTN_ERR_INVALID;
  if (!(softcap == softcap) || !(scale_multiplier == scale_multiplier)) return ATTN_ERR_INVALID;
  if (B > 0 && (!cu_q || !cu_k)) return ATTN_ERR_INVALID;
  if (alibi_slopes && slopes_batch_stride < Hq && B > 1) return ATTN_ERR_INVALID;
  const bool has_q = total_q > 0, has_k = total_k > 0;
  if (has_q && (!q || !out || !lse)) return ATTN_ERR_INVALID;
  if (has_q && bwd && (!dout || !dq)) return ATTN_ERR_INVALID;
  if (has_k && (!k || !v)) return ATTN_ERR_INVALID;
  if (has_k && bwd && (!dk || !dv)) return ATTN_ERR_INVALID;
  if (has_q) {
    for (const void* ptr : {q, static_cast<const void*>(out)})
      if (!aligned16(ptr)) return ATTN_ERR_ALIGNMENT;
    for (int64_t s : {q_ts, q_hs, out_ts, out_hs})
      if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    if (bwd) {
      for (const void* ptr : {dout, static_cast<const void*>(dq)})
        if (!aligned16(ptr)) return ATTN_ERR_ALIGNMENT;
      for (int64_t s : {do_ts, do_hs, dq_ts, dq_hs})
        if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    }
  }
  if (has_k) {
    for (const void* ptr : {k, v})
      if (!aligned16(ptr)) return ATTN_ERR_ALIGNMENT;
    for (int64_t s : {k_ts, v_ts})
      if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    if (Hkv > 1)  // head strides matter only with several K/V heads
      for (int64_t s : {k_hs, v_hs})
        if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    if (bwd) {
      for (const void* ptr : {static_cast<const void*>(dk), static_cast<const void*>(dv)})
        if (!aligned16(ptr)) return ATTN_ERR_ALIGNMENT;
      for (int64_t s : {dk_ts, dv_ts})
        if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
      if (Hkv > 1)
        for (int64_t s : {dk_hs, dv_hs})
          if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    }
  }
  const WsLayout ws = ws_layout(B, Hq, total_q);
  // the per-token dropout rate table (the layout's last part) is used only
  // by calls with per-token rates
  const size_t ws_need = (drop.on && drop.rates) ? ws.total : ws.droptab;
  if (!workspace || workspace_bytes < ws_need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_WORKSPACE;

  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  Params p;
  std::memset(&p, 0, sizeof p);
  p.dtype = dtype;
  p.B = B;
  p.Hq = Hq;
  p.G = head_group(Hq / (Hkv > 0 ? Hkv : 1));
  p.d = head_dim;
  p.total_q = total_q;
  p.total_k = total_k;
  p.out = out;
  p.out_ts = out_ts;
  p.out_hs = out_hs;
  p.dq = dq;
  p.dq_ts = dq_ts;
  p.dq_hs = dq_hs;
  p.dk = dk;
  p.dk_ts = dk_ts;
  p.dk_hs = Hkv > 1 ? dk_hs : 0;
  p.dv = dv;
  p.dv_ts = dv_ts;
  p.dv_hs = Hkv > 1 ? dv_hs : 0;
  p.Hkv = Hkv;
  p.outp = out;
  p.dout = dout;
  p.q = q;
  p.q_ts = q_ts;
  p.q_hs = q_hs;
  p.do_ts = do_ts;
  p.do_hs = do_hs;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.slopes = alibi_slopes;
  p.slopes_bs = slopes_batch_stride;
  p.causal = causal ? 1 : 0;
  p.wl = window_left;
  p.wr = window_right;
  p.softcap = softcap;
  p.sigma = static_cast<float>(static_cast<double>(scale_multiplier) /
                               std::sqrt(static_cast<double>(head_dim)));
  p.lse = lse;
  p.lse_rs = Hq;
  p.Dbuf = reinterpret_cast<float*>(wsb + ws.dbuf);
  p.status = device_status ? device_status : reinterpret_cast<int32_t*>(wsb + ws.status);
  p.counters = reinterpret_cast<int32_t*>(wsb + ws.counters);
  p.ncounters = 3 * Hkv;
  if (drop.on) {
    p.dropout = 1;
    p.drop_seed = drop.seed;
    drop_params(drop.rate, p.drop_T, p.drop_scale);
    p.drop_rates = drop.rates;
    p.drop_tab = drop.rates ? reinterpret_cast<uint2*>(wsb + ws.droptab) : nullptr;
    if (drop.mask_call) {
      p.drop_mask = static_cast<uint8_t*>(drop.mask);
      p.drop_mask_bytes = drop.mask_bytes;
    }
  }
  p.sched = reinterpret_cast<int32_t*>(wsb + ws.sched);

  // ---- degenerate sizes: no query or no key at all
  if (!has_q || !has_k) {
    if (cudaMemsetAsync(p.status, 0, sizeof(int32_t), stream) != cudaSuccess) return ATTN_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (has_k && bwd) {  // no queries: dk = dv = 0
      e = launch_zero_fill(dk, total_k, Hkv, dk_ts, Hkv > 1 ? dk_hs : 8, head_dim, stream);
      if (e == cudaSuccess)
        e = launch_zero_fill(dv, total_k, Hkv, dv_ts, Hkv > 1 ? dv_hs : 8, head_dim, stream);
    }
    if (has_q) {  // no keys: every row is empty
      if (fwd) {
        if (e == cudaSuccess)
          e = launch_zero_fill(out, total_q, Hq, out_ts, out_hs, head_dim, stream);
        if (e == cudaSuccess) e = launch_fill_f32(lse, total_q * Hq, -INFINITY, stream);
      }
      if (bwd && e == cudaSuccess)
        e = launch_zero_fill(dq, total_q, Hq, dq_ts, dq_hs, head_dim, stream);
    }
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }

  // ---- TMA tensor maps of one K/V head group (all of them when Hkv = 1)
  if (!encode_fn()) return ATTN_ERR_CUDA;
  struct Maps {
    CUtensorMap tq, tdo, tqt, tdot, tk, tv, tkt, tvt, tq2, tdo2, tk2, tv2;
  };
  const int R = Hq / Hkv;  // query heads per K/V head
  auto group_params = [&](int g) {
    Params pg = p;
    pg.Hq = R;
    auto off = [](const void* base, int64_t elems) -> const uint16_t* {
      return base ? static_cast<const uint16_t*>(base) + elems : nullptr;
    };
    const int64_t h0 = static_cast<int64_t>(g) * R;
    pg.q = off(q, h0 * q_hs);
    pg.out = const_cast<uint16_t*>(off(out, h0 * out_hs));
    pg.outp = pg.out;
    pg.dq = const_cast<uint16_t*>(off(dq, h0 * dq_hs));
    pg.dout = off(dout, h0 * do_hs);
    pg.dk = const_cast<uint16_t*>(off(dk, static_cast<int64_t>(g) * dk_hs));
    pg.dv = const_cast<uint16_t*>(off(dv, static_cast<int64_t>(g) * dv_hs));
    pg.lse = lse + h0;
    pg.Dbuf = p.Dbuf + h0;
    pg.slopes = alibi_slopes ? alibi_slopes + h0 : nullptr;
    pg.counters = p.counters + 3 * g;
    pg.head0 = static_cast<int>(h0);
    return pg;
  };
  auto encode_group = [&](const Params& pg, int g, Maps& m) -> bool {
    const void* kg = static_cast<const uint16_t*>(k) + static_cast<int64_t>(g) * k_hs;
    const void* vg = static_cast<const uint16_t*>(v) + static_cast<int64_t>(g) * v_hs;
    if (!encode_q_pair(&m.tq2, dtype, head_dim, pg.q, total_q, R, q_ts, q_hs, p.G, kRowsQ) ||
        !encode_kv_pair(&m.tk2, dtype, head_dim, kg, total_k, k_ts) ||
        !encode_kv_pair(&m.tv2, dtype, head_dim, vg, total_k, v_ts) ||
        !encode_q(&m.tq, dtype, head_dim, pg.q, total_q, R, q_ts, q_hs, p.G, kRowsQ) ||
        !encode_q(&m.tqt, dtype, head_dim, pg.q, total_q, R, q_ts, q_hs, p.G, kRowsQ, true) ||
        !encode_kv(&m.tk, dtype, head_dim, kg, total_k, k_ts) || !encode_kv(&m.tv, dtype, head_dim, vg, total_k, v_ts) ||
        !encode_kv(&m.tkt, dtype, head_dim, kg, total_k, k_ts, true) ||
        !encode_kv(&m.tvt, dtype, head_dim, vg, total_k, v_ts, true))
      return false;
    if (bwd && (!encode_q_pair(&m.tdo2, dtype, head_dim, pg.dout, total_q, R, do_ts, do_hs, p.G, kRowsQ) ||
                !encode_q(&m.tdo, dtype, head_dim, pg.dout, total_q, R, do_ts, do_hs, p.G, kRowsQ) ||
                !encode_q(&m.tdot, dtype, head_dim, pg.dout, total_q, R, do_ts, do_hs, p.G, kRowsQ, true)))
      return false;
    return true;
  };

  const int sms = sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  // Upper bounds of the tile counts of one group (the device schedule has
  // the exact ones).
  const int64_t rows_tok = kRowsQ / p.G;
  const int64_t qtiles_max = (total_q / rows_tok + B) * (R / p.G);
  const int64_t ktiles_max = total_k / kKeys + B;
  const int grid_q = static_cast<int>(qtiles_max < sms ? qtiles_max : sms);
  const int grid_k = static_cast<int>(ktiles_max < sms ? ktiles_max : sms);

  // the timing hook applies to the fused call with one K/V head only
  const int nev = (fwd && bwd && Hkv == 1) ? g_nevents : 0;
  if (fwd && bwd) g_nevents = 0;
  auto mark = [&](int i) {
    if (nev) cudaEventRecord(g_events[i], stream);
  };
  Params p0 = group_params(0);
  p0.counters = p.counters;  // the schedule resets every group's counters
  mark(0);
  if (launch_sched(p0, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  // the forward of a stored-mask dropout call first writes the keep bits
  if (fwd && p.drop_mask && launch_mask(p0, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  mark(1);
  Maps m;
  if (fwd) {
    for (int g = 0; g < Hkv; ++g) {
      const Params pg = group_params(g);
      if (!encode_group(pg, g, m)) return ATTN_ERR_ALIGNMENT;
      if (launch_fwd(pg, m.tq2, m.tqt, m.tk2, m.tkt, m.tv2, m.tv, grid_q, stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    }
  }
  if (!bwd) return ATTN_OK;
  mark(2);
  if (launch_preprocess(p, stream) != cudaSuccess) return ATTN_ERR_CUDA;  // every head
  mark(3);
  for (int g = 0; g < Hkv; ++g) {
    const Params pg = group_params(g);
    if (!encode_group(pg, g, m)) return ATTN_ERR_ALIGNMENT;
    if (launch_dkdv(pg, m.tq2, m.tq, m.tdo2, m.tdo, m.tk2, m.tkt, m.tv2, m.tvt, grid_k,
                    stream) != cudaSuccess)
      return ATTN_ERR_CUDA;
    mark(4);
    // dq may overlap the tail of dk/dv (no per-kernel events in between)
    if (launch_dq(pg, m.tq2, m.tqt, m.tdo2, m.tdot, m.tk2, m.tk, m.tv2, m.tvt, grid_q, nev == 0,
                  stream) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  mark(5);
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_varlen_fvjp_fwd_bwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts, int64_t do_hs,
    const int32_t* cu_q, const int32_t* cu_k, const float* alibi_slopes,
    int64_t slopes_batch_stride, int causal, int window_left, int window_right, float softcap,
    float scale_multiplier, void* out, int64_t out_ts, int64_t out_hs, void* dq, int64_t dq_ts,
    int64_t dq_hs, void* dk, int64_t dk_ts, int64_t dk_hs, void* dv, int64_t dv_ts,
    int64_t dv_hs, float* lse, void* workspace, size_t workspace_bytes, int32_t* device_status,
    void* stream) {
  return run_call(kModeFwd | kModeBwd, dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts,
                  q_hs, k, k_ts, k_hs, v, v_ts, v_hs, dout, do_ts, do_hs, cu_q, cu_k,
                  alibi_slopes, slopes_batch_stride, causal, window_left, window_right, softcap,
                  scale_multiplier, out, out_ts, out_hs, dq, dq_ts, dq_hs, dk, dk_ts, dk_hs, dv,
                  dv_ts, dv_hs, lse, workspace, workspace_bytes, device_status, stream);
}

extern "C" attn_status attn_varlen_fwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const int32_t* cu_q, const int32_t* cu_k,
    const float* alibi_slopes, int64_t slopes_batch_stride, int causal, int window_left,
    int window_right, float softcap, float scale_multiplier, void* out, int64_t out_ts,
    int64_t out_hs, float* lse, void* workspace, size_t workspace_bytes, int32_t* device_status,
    void* stream) {
  return run_call(kModeFwd, dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts, q_hs, k,
                  k_ts, k_hs, v, v_ts, v_hs, nullptr, 0, 0, cu_q, cu_k, alibi_slopes,
                  slopes_batch_stride, causal, window_left, window_right, softcap,
                  scale_multiplier, out, out_ts, out_hs, nullptr, 0, 0, nullptr, 0, 0, nullptr,
                  0, 0, lse, workspace, workspace_bytes, device_status, stream);
}

extern "C" attn_status attn_varlen_bwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts, int64_t do_hs,
    const int32_t* cu_q, const int32_t* cu_k, const float* alibi_slopes,
    int64_t slopes_batch_stride, int causal, int window_left, int window_right, float softcap,
    float scale_multiplier, const void* out, int64_t out_ts, int64_t out_hs, const float* lse,
    void* dq, int64_t dq_ts, int64_t dq_hs, void* dk, int64_t dk_ts, int64_t dk_hs, void* dv,
    int64_t dv_ts, int64_t dv_hs, void* workspace, size_t workspace_bytes,
    int32_t* device_status, void* stream) {
  // out and lse are only read on this path
  return run_call(kModeBwd, dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts, q_hs, k,
                  k_ts, k_hs, v, v_ts, v_hs, dout, do_ts, do_hs, cu_q, cu_k, alibi_slopes,
                  slopes_batch_stride, causal, window_left, window_right, softcap,
                  scale_multiplier, const_cast<void*>(out), out_ts, out_hs, dq, dq_ts, dq_hs, dk,
                  dk_ts, dk_hs, dv, dv_ts, dv_hs, const_cast<float*>(lse), workspace,
                  workspace_bytes, device_status, stream);
}

extern "C" attn_status attn_varlen_fvjp_fwd_bwd_dropout(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts, int64_t do_hs,
    const int32_t* cu_q, const int32_t* cu_k, const float* alibi_slopes,
    int64_t slopes_batch_stride, int causal, int window_left, int window_right, float softcap,
    float scale_multiplier, uint64_t dropout_seed, float dropout_rate,
    const float* dropout_rates, void* out, int64_t out_ts, int64_t out_hs, void* dq,
    int64_t dq_ts, int64_t dq_hs, void* dk, int64_t dk_ts, int64_t dk_hs, void* dv,
    int64_t dv_ts, int64_t dv_hs, float* lse, void* workspace, size_t workspace_bytes,
    int32_t* device_status, void* stream) {
  Dropout dr;
  dr.on = true;
  dr.seed = dropout_seed;
  dr.rate = dropout_rate;
  dr.rates = dropout_rates;
  return run_call(kModeFwd | kModeBwd, dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts,
                  q_hs, k, k_ts, k_hs, v, v_ts, v_hs, dout, do_ts, do_hs, cu_q, cu_k,
                  alibi_slopes, slopes_batch_stride, causal, window_left, window_right, softcap,
                  scale_multiplier, out, out_ts, out_hs, dq, dq_ts, dq_hs, dk, dk_ts, dk_hs, dv,
                  dv_ts, dv_hs, lse, workspace, workspace_bytes, device_status, stream, dr);
}

extern "C" attn_status attn_varlen_fwd_dropout(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const int32_t* cu_q, const int32_t* cu_k,
    const float* alibi_slopes, int64_t slopes_batch_stride, int causal, int window_left,
    int window_right, float softcap, float scale_multiplier, uint64_t dropout_seed,
    float dropout_rate, const float* dropout_rates, void* out, int64_t out_ts, int64_t out_hs,
    float* lse, void* workspace, size_t workspace_bytes, int32_t* device_status, void* stream) {
  Dropout dr;
  dr.on = true;
  dr.seed = dropout_seed;
  dr.rate = dropout_rate;
  dr.rates = dropout_rates;
  return run_call(kModeFwd, dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts, q_hs, k,
                  k_ts, k_hs, v, v_ts, v_hs, nullptr, 0, 0, cu_q, cu_k, alibi_slopes,
                  slopes_batch_stride, causal, window_left, window_right, softcap,
                  scale_multiplier, out, out_ts, out_hs, nullptr, 0, 0, nullptr, 0, 0, nullptr,
                  0, 0, lse, workspace, workspace_bytes, device_status, stream, dr);
}

extern "C" attn_status attn_varlen_bwd_dropout(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts, int64_t do_hs,
    const int32_t* cu_q, const int32_t* cu_k, const float* alibi_slopes,
    int64_t slopes_batch_stride, int causal, int window_left, int window_right, float softcap,
    float scale_multiplier, uint64_t dropout_seed, float dropout_rate,
    const float* dropout_rates, const void* out, int64_t out_ts, int64_t out_hs,
    const float* lse, void* dq, int64_t dq_ts, int64_t dq_hs, void* dk, int64_t dk_ts,
    int64_t dk_hs, void* dv, int64_t dv_ts, int64_t dv_hs, void* workspace,
    size_t workspace_bytes, int32_t* device_status, void* stream) {
  Dropout dr;
  dr.on = true;
  dr.seed = dropout_seed;
  dr.rate = dropout_rate;
  dr.rates = dropout_rates;
  return run_call(kModeBwd, dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts, q_hs, k,
                  k_ts, k_hs, v, v_ts, v_hs, dout, do_ts, do_hs, cu_q, cu_k, alibi_slopes,
                  slopes_batch_stride, causal, window_left, window_right, softcap,
                  scale_multiplier, const_cast<void*>(out), out_ts, out_hs, dq, dq_ts, dq_hs, dk,
                  dk_ts, dk_hs, dv, dv_ts, dv_hs, const_cast<float*>(lse), workspace,
                  workspace_bytes, device_status, stream, dr);
}

extern "C" attn_status attn_varlen_fvjp_fwd_bwd_dropout_mask(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts, int64_t do_hs,
    const int32_t* cu_q, const int32_t* cu_k, const float* alibi_slopes,
    int64_t slopes_batch_stride, int causal, int window_left, int window_right, float softcap,
    float scale_multiplier, uint64_t dropout_seed, float dropout_rate,
    const float* dropout_rates, void* keep_mask, size_t keep_mask_bytes, void* out,
    int64_t out_ts, int64_t out_hs, void* dq, int64_t dq_ts, int64_t dq_hs, void* dk,
    int64_t dk_ts, int64_t dk_hs, void* dv, int64_t dv_ts, int64_t dv_hs, float* lse,
    void* workspace, size_t workspace_bytes, int32_t* device_status, void* stream) {
  Dropout dr;
  dr.on = true;
  dr.seed = dropout_seed;
  dr.rate = dropout_rate;
  dr.rates = dropout_rates;
  dr.mask = keep_mask;
  dr.mask_bytes = keep_mask_bytes;
  dr.mask_call = true;
  return run_call(kModeFwd | kModeBwd, dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts,
                  q_hs, k, k_ts, k_hs, v, v_ts, v_hs, dout, do_ts, do_hs, cu_q, cu_k,
                  alibi_slopes, slopes_batch_stride, causal, window_left, window_right, softcap,
                  scale_multiplier, out, out_ts, out_hs, dq, dq_ts, dq_hs, dk, dk_ts, dk_hs, dv,
                  dv_ts, dv_hs, lse, workspace, workspace_bytes, device_status, stream, dr);
}

extern "C" attn_status attn_varlen_fwd_dropout_mask(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const int32_t* cu_q, const int32_t* cu_k,
    const float* alibi_slopes, int64_t slopes_batch_stride, int causal, int window_left,
    int window_right, float softcap, float scale_multiplier, uint64_t dropout_seed,
    float dropout_rate, const float* dropout_rates, void* keep_mask, size_t keep_mask_bytes,
    void* out, int64_t out_ts, int64_t out_hs, float* lse, void* workspace,
    size_t workspace_bytes, int32_t* device_status, void* stream) {
  Dropout dr;
  dr.on = true;
  dr.seed = dropout_seed;
  dr.rate = dropout_rate;
  dr.rates = dropout_rates;
  dr.mask = keep_mask;
  dr.mask_bytes = keep_mask_bytes;
  dr.mask_call = true;
  return run_call(kModeFwd, dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts, q_hs, k,
                  k_ts, k_hs, v, v_ts, v_hs, nullptr, 0, 0, cu_q, cu_k, alibi_slopes,
                  slopes_batch_stride, causal, window_left, window_right, softcap,
                  scale_multiplier, out, out_ts, out_hs, nullptr, 0, 0, nullptr, 0, 0, nullptr,
                  0, 0, lse, workspace, workspace_bytes, device_status, stream, dr);
}

extern "C" attn_status attn_varlen_bwd_dropout_mask(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts, int64_t do_hs,
    const int32_t* cu_q, const int32_t* cu_k, const float* alibi_slopes,
    int64_t slopes_batch_stride, int causal, int window_left, int window_right, float softcap,
    float scale_multiplier, uint64_t dropout_seed, float dropout_rate,
    const float* dropout_rates, const void* keep_mask, size_t keep_mask_bytes, const void* out,
    int64_t out_ts, int64_t out_hs, const float* lse, void* dq, int64_t dq_ts, int64_t dq_hs,
    void* dk, int64_t dk_ts, int64_t dk_hs, void* dv, int64_t dv_ts, int64_t dv_hs,
    void* workspace, size_t workspace_bytes, int32_t* device_status, void* stream) {
  Dropout dr;
  dr.on = true;
  dr.seed = dropout_seed;
  dr.rate = dropout_rate;
  dr.rates = dropout_rates;
  // the backward only reads the blocks (the schedule kernel rewrites the
  // header with the same values)
  dr.mask = const_cast<void*>(keep_mask);
  dr.mask_bytes = keep_mask_bytes;
  dr.mask_call = true;
  return run_call(kModeBwd, dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts, q_hs, k,
                  k_ts, k_hs, v, v_ts, v_hs, dout, do_ts, do_hs, cu_q, cu_k, alibi_slopes,
                  slopes_batch_stride, causal, window_left, window_right, softcap,
                  scale_multiplier, const_cast<void*>(out), out_ts, out_hs, dq, dq_ts, dq_hs, dk,
                  dk_ts, dk_hs, dv, dv_ts, dv_hs, const_cast<float*>(lse), workspace,
                  workspace_bytes, device_status, stream, dr);
}

extern "C" size_t attn_varlen_dropout_mask_bytes(int B, const int32_t* cu_q, const int32_t* cu_k,
                                                 int Hq, int Hkv) {
  if (B < 0 || B > ATTN_MAX_BATCH || Hq <= 0 || Hkv < 1 || Hq % Hkv ||
      (B > 0 && (!cu_q || !cu_k)))
    return 0;
  const int G = head_group(Hq / Hkv);
  const int64_t rows_tok = kRowsQ / G, ngroups = Hq / Hkv / G;
  uint64_t blocks = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t lq = static_cast<int64_t>(cu_q[b + 1]) - cu_q[b];
    const int64_t lk = static_cast<int64_t>(cu_k[b + 1]) - cu_k[b];
    if (lq < 0 || lk < 0) return 0;
    blocks += static_cast<uint64_t>((lq + rows_tok - 1) / rows_tok * ngroups *
                                    ((lk + kKeys - 1) / kKeys));
  }
  return drop_mask_header(B) + blocks * Hkv * 8ull * kMaskBlockWords;
}

// ------------------------------------------------------------------ gated

namespace {

// The sigmoid-gated call ("Pairwise-Gated Attention Engine", "Why it is
// hard"): validation, tensor maps per K/V head group and the launches of the
// requested passes (forward: schedule, forward per group; backward:
// schedule, preprocess, dk/dv and dq per group).
attn_status run_gated(
    int mode, attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int gate_dim,
    int64_t total_q, int64_t total_k, const void* q, int64_t q_ts, int64_t q_hs, const void* k,
    int64_t k_ts, int64_t k_hs, const void* v, int64_t v_ts, int64_t v_hs, const void* dout,
    int64_t do_ts, int64_t do_hs, const void* qg, int64_t qg_ts, int64_t qg_hs, const void* kg,
    int64_t kg_ts, int64_t kg_hs, const int32_t* cu_q, const int32_t* cu_k,
    const float* alibi_slopes, int64_t slopes_batch_stride, int causal, int window_left,
    int window_right, float scale_multiplier, void* out, int64_t out_ts, int64_t out_hs,
    void* dq, int64_t dq_ts, int64_t dq_hs, void* dk, int64_t dk_ts, int64_t dk_hs, void* dv,
    int64_t dv_ts, int64_t dv_hs, void* dqg, int64_t dqg_ts, int64_t dqg_hs, void* dkg,
    int64_t dkg_ts, int64_t dkg_hs, float* lse, void* workspace, size_t workspace_bytes,
    int32_t* device_status, void* stream_ptr) {
  const bool fwd = (mode & kModeFwd) != 0, bwd = (mode & kModeBwd) != 0;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
  if (B < 0 || Hq <= 0 || total_q < 0 || total_k < 0) return ATTN_ERR_INVALID;
  if (head_dim != 128 && head_dim != 64) return ATTN_ERR_UNSUPPORTED;
  if (gate_dim < 8 || gate_dim > 64 || gate_dim % 8) return ATTN_ERR_UNSUPPORTED;
  if (Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID;
  if (B > ATTN_MAX_BATCH) return ATTN_ERR_UNSUPPORTED;
  if (total_q > INT32_MAX || total_k > INT32_MAX) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 && (total_q != 0 || total_k != 0)) return ATTN_ERR_INVALID;
  if (!(scale_multiplier == scale_multiplier)) return ATTN_ERR_INVALID;
  if (B > 0 && (!cu_q || !cu_k)) return ATTN_ERR_INVALID;
  if (alibi_slopes && slopes_batch_stride < Hq && B > 1) return ATTN_ERR_INVALID;
  const bool has_q = total_q > 0, has_k = total_k > 0;
  if (has_q && (!q || !qg || !out || !lse)) return ATTN_ERR_INVALID;
  if (has_q && bwd && (!dout || !dq || !dqg)) return ATTN_ERR_INVALID;
  if (has_k && (!k || !v || !kg)) return ATTN_ERR_INVALID;
  if (has_k && bwd && (!dk || !dv || !dkg)) return ATTN_ERR_INVALID;
  if (has_q) {
    for (const void* ptr : {q, qg, static_cast<const void*>(out)})
      if (!aligned16(ptr)) return ATTN_ERR_ALIGNMENT;
    for (int64_t s : {q_ts, q_hs, qg_ts, qg_hs, out_ts, out_hs})
      if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    if (bwd) {
      for (const void* ptr : {dout, static_cast<const void*>(dq), static_cast<const void*>(dqg)})
        if (!aligned16(ptr)) return ATTN_ERR_ALIGNMENT;
      for (int64_t s : {do_ts, do_hs, dq_ts, dq_hs, dqg_ts, dqg_hs})
        if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    }
  }
  if (has_k) {
    for (const void* ptr : {k, v, kg})
      if (!aligned16(ptr)) return ATTN_ERR_ALIGNMENT;
    for (int64_t s : {k_ts, v_ts, kg_ts})
      if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    if (Hkv > 1)
      for (int64_t s : {k_hs, v_hs, kg_hs})
        if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    if (bwd) {
      for (const void* ptr : {static_cast<const void*>(dk), static_cast<const void*>(dv),
                              static_cast<const void*>(dkg)})
        if (!aligned16(ptr)) return ATTN_ERR_ALIGNMENT;
      for (int64_t s : {dk_ts, dv_ts, dkg_ts})
        if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
      if (Hkv > 1)
        for (int64_t s : {dk_hs, dv_hs, dkg_hs})
          if (!stride_ok(s)) return ATTN_ERR_ALIGNMENT;
    }
  }
  const WsLayout ws = ws_layout(B, Hq, total_q);
  if (!workspace || workspace_bytes < ws.droptab ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_WORKSPACE;

  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  Params p;
  std::memset(&p, 0, sizeof p);
  p.dtype = dtype;
  p.B = B;
  p.Hq = Hq;
  p.G = head_group(Hq / Hkv);
  p.d = head_dim;
  p.total_q = total_q;
  p.total_k = total_k;
  p.out = out;
  p.out_ts = out_ts;
  p.out_hs = out_hs;
  p.dq = dq;
  p.dq_ts = dq_ts;
  p.dq_hs = dq_hs;
  p.dk = dk;
  p.dk_ts = dk_ts;
  p.dk_hs = Hkv > 1 ? dk_hs : 0;
  p.dv = dv;
  p.dv_ts = dv_ts;
  p.dv_hs = Hkv > 1 ? dv_hs : 0;
  p.Hkv = Hkv;
  p.outp = out;
  p.dout = dout;
  p.q = q;
  p.q_ts = q_ts;
  p.q_hs = q_hs;
  p.do_ts = do_ts;
  p.do_hs = do_hs;
  p.cu_q = cu_q;
  p.cu_k = cu_k;
  p.slopes = alibi_slopes;
  p.slopes_bs = slopes_batch_stride;
  p.causal = causal ? 1 : 0;
  p.wl = window_left;
  p.wr = window_right;
  p.softcap = 0.f;
  p.sigma = static_cast<float>(static_cast<double>(scale_multiplier) /
                               std::sqrt(static_cast<double>(head_dim)));
  p.lse = lse;
  p.lse_rs = Hq;
  p.Dbuf = reinterpret_cast<float*>(wsb + ws.dbuf);
  p.status = device_status ? device_status : reinterpret_cast<int32_t*>(wsb + ws.status);
  p.counters = reinterpret_cast<int32_t*>(wsb + ws.counters);
  p.ncounters = 3 * Hkv;
  p.sched = reinterpret_cast<int32_t*>(wsb + ws.sched);
  p.qg = qg;
  p.qg_ts = qg_ts;
  p.qg_hs = qg_hs;
  p.dqg = dqg;
  p.dqg_ts = dqg_ts;
  p.dqg_hs = dqg_hs;
  p.dkg = bwd ? dkg : nullptr;
  p.dkg_ts = dkg_ts;
  p.dkg_hs = Hkv > 1 ? dkg_hs : 0;
  p.R = gate_dim;
  p.gscale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(gate_dim)));

  if (!has_q || !has_k) {
    if (cudaMemsetAsync(p.status, 0, sizeof(int32_t), stream) != cudaSuccess) return ATTN_ERR_CUDA;
    cudaError_t e = cudaSuccess;
    if (has_k && bwd) {  // no queries: dk = dv = dk_g = 0
      e = launch_zero_fill(dk, total_k, Hkv, dk_ts, Hkv > 1 ? dk_hs : 8, head_dim, stream);
      if (e == cudaSuccess)
        e = launch_zero_fill(dv, total_k, Hkv, dv_ts, Hkv > 1 ? dv_hs : 8, head_dim, stream);
      if (e == cudaSuccess)
        e = launch_zero_fill(dkg, total_k, Hkv, dkg_ts, Hkv > 1 ? dkg_hs : 8, gate_dim, stream);
    }
    if (has_q) {  // no keys: every row is empty
      if (fwd) {
        if (e == cudaSuccess)
          e = launch_zero_fill(out, total_q, Hq, out_ts, out_hs, head_dim, stream);
        if (e == cudaSuccess) e = launch_fill_f32(lse, total_q * Hq, -INFINITY, stream);
      }
      if (bwd && e == cudaSuccess)
        e = launch_zero_fill(dq, total_q, Hq, dq_ts, dq_hs, head_dim, stream);
      if (bwd && e == cudaSuccess)
        e = launch_zero_fill(dqg, total_q, Hq, dqg_ts, dqg_hs, gate_dim, stream);
    }
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }

  if (!encode_fn()) return ATTN_ERR_CUDA;
  const int R = Hq / Hkv;
  auto off = [](const void* base, int64_t elems) -> uint16_t* {
    return base ? const_cast<uint16_t*>(static_cast<const uint16_t*>(base)) + elems : nullptr;
  };
  auto group_params = [&](int g) {
    Params pg = p;
    pg.Hq = R;
    const int64_t h0 = static_cast<int64_t>(g) * R;
    pg.q = off(q, h0 * q_hs);
    pg.out = off(out, h0 * out_hs);
    pg.outp = pg.out;
    pg.dq = off(dq, h0 * dq_hs);
    pg.dout = off(dout, h0 * do_hs);
    pg.dk = off(dk, static_cast<int64_t>(g) * dk_hs);
    pg.dv = off(dv, static_cast<int64_t>(g) * dv_hs);
    pg.qg = off(qg, h0 * qg_hs);
    pg.dqg = off(dqg, h0 * dqg_hs);
    pg.dkg = off(dkg, static_cast<int64_t>(g) * dkg_hs);
    pg.lse = lse + h0;
    pg.Dbuf = p.Dbuf + h0;
    pg.slopes = alibi_slopes ? alibi_slopes + h0 : nullptr;
    pg.counters = p.counters + 3 * g;
    pg.head0 = static_cast<int>(h0);
    return pg;
  };
  struct Maps {
    CUtensorMap tq, tqg, tdo, tk, tkg, tv;
  };
  // a 128-row tile of head_dim features: both 64-wide chunks in one box
  // when head_dim = 128; the gate projections as one 64-wide box (zeros
  // past gate_dim)
  auto encode_group = [&](const Params& pg, int g, Maps& m) -> bool {
    const void* kgrp = static_cast<const uint16_t*>(k) + static_cast<int64_t>(g) * k_hs;
    const void* vgrp = static_cast<const uint16_t*>(v) + static_cast<int64_t>(g) * v_hs;
    const void* kggrp = static_cast<const uint16_t*>(kg) + static_cast<int64_t>(g) * kg_hs;
    const bool two = head_dim == 128;
    bool ok = two ? encode_q_pair(&m.tq, dtype, head_dim, pg.q, total_q, R, q_ts, q_hs, p.G, kRowsQ)
                  : encode_q(&m.tq, dtype, head_dim, pg.q, total_q, R, q_ts, q_hs, p.G, kRowsQ);
    ok = ok && encode_q(&m.tqg, dtype, gate_dim, pg.qg, total_q, R, qg_ts, qg_hs, p.G, kRowsQ);
    ok = ok && (two ? encode_kv_pair(&m.tk, dtype, head_dim, kgrp, total_k, k_ts)
                    : encode_kv(&m.tk, dtype, head_dim, kgrp, total_k, k_ts));
    ok = ok && (two ? encode_kv_pair(&m.tv, dtype, head_dim, vgrp, total_k, v_ts)
                    : encode_kv(&m.tv, dtype, head_dim, vgrp, total_k, v_ts));
    ok = ok && encode_kv(&m.tkg, dtype, gate_dim, kggrp, total_k, kg_ts);
    if (bwd)
      ok = ok && (two ? encode_q_pair(&m.tdo, dtype, head_dim, pg.dout, total_q, R, do_ts, do_hs,
                                      p.G, kRowsQ)
                      : encode_q(&m.tdo, dtype, head_dim, pg.dout, total_q, R, do_ts, do_hs,
                                 p.G, kRowsQ));
    return ok;
  };
  const int sms = sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const int64_t rows_tok = kRowsQ / p.G;
  const int64_t qtiles_max = (total_q / rows_tok + B) * (R / p.G);
  const int64_t ktiles_max = total_k / kKeys + B;
  const int grid_q = static_cast<int>(qtiles_max < sms ? qtiles_max : sms);
  const int grid_k = static_cast<int>(ktiles_max < sms ? ktiles_max : sms);
  Params p0 = group_params(0);
  p0.counters = p.counters;
  if (launch_sched(p0, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  Maps m;
  if (fwd) {
    for (int g = 0; g < Hkv; ++g) {
      const Params pg = group_params(g);
      if (!encode_group(pg, g, m)) return ATTN_ERR_ALIGNMENT;
      if (launch_gate_fwd(pg, m.tq, m.tqg, m.tk, m.tkg, m.tv, grid_q, stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    }
  }
  if (!bwd) return ATTN_OK;
  if (launch_preprocess(p, stream) != cudaSuccess) return ATTN_ERR_CUDA;
  for (int g = 0; g < Hkv; ++g) {
    const Params pg = group_params(g);
    if (!encode_group(pg, g, m)) return ATTN_ERR_ALIGNMENT;
    if (launch_gate_dkdv(pg, m.tq, m.tqg, m.tdo, m.tk, m.tkg, m.tv, grid_k, stream) !=
        cudaSuccess)
      return ATTN_ERR_CUDA;
    if (launch_gate_dq(pg, m.tq, m.tqg, m.tdo, m.tk, m.tkg, m.tv, grid_q, stream) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_varlen_gated_fvjp_fwd_bwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int gate_dim, int64_t total_q,
    int64_t total_k, const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts,
    int64_t k_hs, const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts,
    int64_t do_hs, const void* q_gate, int64_t qg_ts, int64_t qg_hs, const void* k_gate,
    int64_t kg_ts, int64_t kg_hs, const int32_t* cu_q, const int32_t* cu_k,
    const float* alibi_slopes, int64_t slopes_batch_stride, int causal, int window_left,
    int window_right, float scale_multiplier, void* out, int64_t out_ts, int64_t out_hs,
    void* dq, int64_t dq_ts, int64_t dq_hs, void* dk, int64_t dk_ts, int64_t dk_hs, void* dv,
    int64_t dv_ts, int64_t dv_hs, void* dq_gate, int64_t dqg_ts, int64_t dqg_hs, void* dk_gate,
    int64_t dkg_ts, int64_t dkg_hs, float* lse, void* workspace, size_t workspace_bytes,
    int32_t* device_status, void* stream) {
  return run_gated(kModeFwd | kModeBwd, dtype, B, Hq, Hkv, head_dim, gate_dim, total_q, total_k,
                   q, q_ts, q_hs, k, k_ts, k_hs, v, v_ts, v_hs, dout, do_ts, do_hs, q_gate, qg_ts,
                   qg_hs, k_gate, kg_ts, kg_hs, cu_q, cu_k, alibi_slopes, slopes_batch_stride,
                   causal, window_left, window_right, scale_multiplier, out, out_ts, out_hs, dq,
                   dq_ts, dq_hs, dk, dk_ts, dk_hs, dv, dv_ts, dv_hs, dq_gate, dqg_ts, dqg_hs,
                   dk_gate, dkg_ts, dkg_hs, lse, workspace, workspace_bytes, device_status,
                   stream);
}

extern "C" attn_status attn_varlen_gated_fwd(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int gate_dim, int64_t total_q,
    int64_t total_k, const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts,
    int64_t k_hs, const void* v, int64_t v_ts, int64_t v_hs, const void* q_gate, int64_t qg_ts,
    int64_t qg_hs, const void* k_gate, int64_t kg_ts, int64_t kg_hs, const int32_t* cu_q,
    const int32_t* cu_k, const float* alibi_slopes, int64_t slopes_batch_stride, int causal,
    int window_left, int window_right, float scale_multiplier, void* out, int64_t out_ts,
    int64_t out_hs, float* lse, void* workspace, size_t workspace_bytes, int32_t* device_status,
    void* stream) {
  return run_gated(kModeFwd, dtype, B, Hq, Hkv, head_dim, gate_dim, total_q, total_k, q, q_ts,
                   q_hs, k, k_ts, k_hs, v, v_ts, v_hs, nullptr, 0, 0, q_gate, qg_ts, qg_hs,
                   k_gate, kg_ts, kg_hs, cu_q, cu_k, alibi_slopes, slopes_batch_stride, causal,
                   window_left, window_right, scale_multiplier, out, out_ts, out_hs, nullptr, 0,
                   0, nullptr, 0, 0, nullptr, 0, 0, nullptr, 0, 0, nullptr, 0, 0, lse,
                   workspace, workspace_bytes, device_status, stream);
}
