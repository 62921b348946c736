// host_pipeline.cu -- the fused forward + VJP call on host-resident inputs and
// outputs: the batch is cut into chunks of whole sequences, and each chunk's
// copies over the host link run on their own streams, overlapped with the
// kernels of the neighbouring chunks.
//
// Sequences are independent, so a chunk is an ordinary call on device copies
// of its sequences (rebased cu arrays, pointers at its first token): each
// sequence's results are those of one call over the whole batch, bit for bit.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <utility>
#include <vector>

#include "../../include/attn_varlen.h"

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
constexpr int kMaxSlots = 4;   // chunks in flight: copies in, two computing, copies out
constexpr int kCompStreams = 2;

// Offsets in the caller's device buffer: the shared part (status words of
// every chunk, rebased cu arrays, slopes), then `slots` ring slots, each
// holding one chunk's workspace and dense device copies [T, H, d] (token
// stride H*d, head stride d) sized for the largest chunk.
struct Layout {
  size_t status, cu, slopes, slot0, slot_bytes, total;
  size_t ws, ws_bytes, q, dout, out, dq, k, v, dk, dv, lse;  // offsets within a slot
  int slots;
};

Layout layout(int B, int Hq, int Hkv, int d, int chunks, int nslots, int Bc, int64_t Tq,
              int64_t Tk) {
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  L.status = take(sizeof(int32_t) * static_cast<size_t>(chunks));
  L.cu = take(sizeof(int32_t) * 2 * static_cast<size_t>(B + chunks));  // cu_q, then cu_k
  L.slopes = take(sizeof(float) * static_cast<size_t>(B) * Hq);
  L.slot0 = off;
  off = 0;
  L.ws_bytes = attn_varlen_fvjp_workspace_size(Bc, Hq, Tq, Tk);
  L.ws = take(L.ws_bytes);
  const size_t qbytes = static_cast<size_t>(Tq) * Hq * d * 2;
  const size_t kbytes = static_cast<size_t>(Tk) * Hkv * d * 2;
  L.q = take(qbytes);
  L.dout = take(qbytes);
  L.out = take(qbytes);
  L.dq = take(qbytes);
  L.k = take(kbytes);
  L.v = take(kbytes);
  L.dk = take(kbytes);
  L.dv = take(kbytes);
  L.lse = take(sizeof(float) * static_cast<size_t>(Tq) * Hq);
  L.slot_bytes = off;
  L.slots = nslots;
  L.total = L.slot0 + static_cast<size_t>(nslots) * L.slot_bytes;
  return L;
}

// The chunking of these lengths and the layout its largest chunk needs.
struct Plan {
  std::vector<int32_t> cut;
  int nc;
  Layout L;
};

Plan plan_of(int B, const int32_t* cu_q, const int32_t* cu_k, int Hq, int Hkv, int d,
             int chunks);

// Rows [r0, r1) of a 16-bit [T, H, d] tensor between host (strides ts, hs in
// elements) and a dense device copy whose first row is r0.  One 2-D copy
// when the host heads are dense, else one per head; feature padding is never
// touched.
cudaError_t copy_rows(bool to_device, void* dev, const void* host_c, int64_t ts, int64_t hs,
                      int H, int d, int64_t r0, int64_t r1, cudaStream_t s) {
  if (r1 <= r0) return cudaSuccess;
  uint8_t* host = static_cast<uint8_t*>(const_cast<void*>(host_c));
  uint8_t* devb = static_cast<uint8_t*>(dev);
  const size_t drow = static_cast<size_t>(H) * d * 2;  // device token stride (bytes)
  const size_t hpitch = static_cast<size_t>(ts) * 2;
  const size_t rows = static_cast<size_t>(r1 - r0);
  uint8_t* h = host + static_cast<size_t>(r0) * hpitch;
  if (H == 1 || hs == d) {
    return to_device ? cudaMemcpy2DAsync(devb, drow, h, hpitch, drow, rows, cudaMemcpyHostToDevice, s)
                     : cudaMemcpy2DAsync(h, hpitch, devb, drow, drow, rows, cudaMemcpyDeviceToHost, s);
  }
  for (int hh = 0; hh < H; ++hh) {
    uint8_t* hp = h + static_cast<size_t>(hh) * hs * 2;
    uint8_t* gp = devb + static_cast<size_t>(hh) * d * 2;
    const cudaError_t e =
        to_device
            ? cudaMemcpy2DAsync(gp, drow, hp, hpitch, static_cast<size_t>(d) * 2, rows,
                                cudaMemcpyHostToDevice, s)
            : cudaMemcpy2DAsync(hp, hpitch, gp, drow, static_cast<size_t>(d) * 2, rows,
                                cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// A host tensor's strides fit the copies: every (token, head) row of d
// features lies inside its token's pitch.
bool host_strides_ok(int64_t ts, int64_t hs, int H, int d) {
  if (ts <= 0 || ts % 8 || (H > 1 && (hs <= 0 || hs % 8))) return false;
  const int64_t span = H > 1 ? (H - 1) * hs + d : d;
  return ts >= span && (H == 1 || hs >= d);
}

// The streams and events of one call, released (deferred until the device is
// done with them) when it goes out of scope.
struct Resources {
  cudaStream_t in = nullptr, out = nullptr, comp[kCompStreams] = {nullptr, nullptr};
  std::vector<cudaEvent_t> events;
  // On an error part-way, the caller's stream still waits for the work the
  // call has enqueued on its own streams, so the caller can free its buffers
  // once it has synchronised that stream.
  void join(cudaStream_t caller) {
    for (cudaStream_t s : {in, out, comp[0], comp[1]}) {
      cudaEvent_t e;
      if (s && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess) {
        if (cudaEventRecord(e, s) == cudaSuccess) cudaStreamWaitEvent(caller, e, 0);
        cudaEventDestroy(e);
      }
    }
  }
  ~Resources() {
    for (cudaEvent_t e : events) cudaEventDestroy(e);
    for (cudaStream_t s : {in, out, comp[0], comp[1]})
      if (s) cudaStreamDestroy(s);
  }
  cudaError_t event(cudaEvent_t* e) {
    const cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
    if (r == cudaSuccess) events.push_back(*e);
    return r;
  }
};

}  // namespace

extern "C" int attn_varlen_host_chunks(int B, const int32_t* cu_q, const int32_t* cu_k,
                                       int chunks, int32_t* cuts) {
  if (B < 0 || chunks < 1 || !cuts || (B > 0 && (!cu_q || !cu_k))) return 0;
  // each sequence weighs Lq*Lk + 1, so empty ones still spread over the chunks
  double total = 0;
  for (int b = 0; b < B; ++b)
    total += static_cast<double>(cu_q[b + 1] - cu_q[b]) * (cu_k[b + 1] - cu_k[b]) + 1.0;
  // chunk c's share: with three chunks or more the first and the last take a
  // quarter of the others', so the copies that nothing overlaps (the first
  // chunk's inputs, the last chunk's results) are short
  auto share = [&](int c) { return (chunks >= 3 && (c == 0 || c == chunks - 1)) ? 0.25 : 1.0; };
  double shares = 0;
  for (int c = 0; c < chunks; ++c) shares += share(c);
  int n = 0;
  cuts[0] = 0;
  double acc = 0, bound = total * share(0) / shares;  // where chunk n ends
  for (int b = 0; b < B; ++b) {
    acc += static_cast<double>(cu_q[b + 1] - cu_q[b]) * (cu_k[b + 1] - cu_k[b]) + 1.0;
    if (n + 1 < chunks && b + 1 < B && acc >= bound) {
      cuts[++n] = b + 1;
      bound += total * share(n) / shares;
    }
  }
  cuts[++n] = B;
  return n;
}

namespace {
Plan plan_of(int B, const int32_t* cu_q, const int32_t* cu_k, int Hq, int Hkv, int d,
             int chunks) {
  Plan P;
  P.cut.assign(static_cast<size_t>(chunks) + 1, 0);
  P.nc = attn_varlen_host_chunks(B, cu_q, cu_k, chunks, P.cut.data());
  int Bc = 0;
  int64_t Tq = 0, Tk = 0;
  for (int c = 0; c < P.nc; ++c) {
    const int s = P.cut[c], e = P.cut[c + 1];
    Bc = e - s > Bc ? e - s : Bc;
    Tq = cu_q[e] - cu_q[s] > Tq ? cu_q[e] - cu_q[s] : Tq;
    Tk = cu_k[e] - cu_k[s] > Tk ? cu_k[e] - cu_k[s] : Tk;
  }
  const int slots = P.nc < kMaxSlots ? (P.nc > 0 ? P.nc : 1) : kMaxSlots;
  P.L = layout(B, Hq, Hkv, d, chunks, slots, Bc, Tq, Tk);
  return P;
}
}  // namespace

extern "C" size_t attn_varlen_fvjp_host_buffer_size(int B, int Hq, int Hkv, int head_dim,
                                                     int64_t total_q, int64_t total_k,
                                                     int chunks) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0 || total_q < 0 || total_k < 0 ||
      chunks < 1)
    return 0;
  // any lengths: every slot sized for the whole batch
  const int slots = chunks < kMaxSlots ? chunks : kMaxSlots;
  return layout(B, Hq, Hkv, head_dim, chunks, slots, B, total_q, total_k).total;
}

extern "C" size_t attn_varlen_fvjp_host_buffer_size_for(int B, const int32_t* cu_q,
                                                         const int32_t* cu_k, int Hq, int Hkv,
                                                         int head_dim, int chunks) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0 || chunks < 1 ||
      (B > 0 && (!cu_q || !cu_k)))
    return 0;
  for (int b = 0; b < B; ++b)
    if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return 0;
  return plan_of(B, cu_q, cu_k, Hq, Hkv, head_dim, chunks).L.total;
}

extern "C" attn_status attn_varlen_fvjp_fwd_bwd_host(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts, int64_t do_hs,
    const int32_t* cu_q, const int32_t* cu_k, const float* alibi_slopes,
    int64_t slopes_batch_stride, int causal, int window_left, int window_right, float softcap,
    float scale_multiplier, void* out, int64_t out_ts, int64_t out_hs, void* dq, int64_t dq_ts,
    int64_t dq_hs, void* dk, int64_t dk_ts, int64_t dk_hs, void* dv, int64_t dv_ts,
    int64_t dv_hs, float* lse, void* device_buffer, size_t device_buffer_bytes, int chunks,
    int32_t* host_status, void* stream_ptr) {
  // ---- host-side validation (nothing is enqueued on failure)
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
  if (B < 0 || Hq <= 0 || Hkv < 1 || Hq % Hkv || total_q < 0 || total_k < 0 || chunks < 1)
    return ATTN_ERR_INVALID;
  if (head_dim != 160 && head_dim != 128 && head_dim != 64) return ATTN_ERR_UNSUPPORTED;
  if (B > ATTN_MAX_BATCH) return ATTN_ERR_UNSUPPORTED;
  if (!host_status || (B > 0 && (!cu_q || !cu_k))) return ATTN_ERR_INVALID;
  if (total_q > 0 && (!q || !dout || !out || !dq || !lse)) return ATTN_ERR_INVALID;
  if (total_k > 0 && (!k || !v || !dk || !dv)) return ATTN_ERR_INVALID;
  if (alibi_slopes && B > 1 && slopes_batch_stride < Hq) return ATTN_ERR_INVALID;
  const int d = head_dim;
  if (total_q > 0)
    for (auto st : {std::pair<int64_t, int64_t>{q_ts, q_hs}, {do_ts, do_hs}, {out_ts, out_hs},
                    {dq_ts, dq_hs}})
      if (!host_strides_ok(st.first, st.second, Hq, d)) return ATTN_ERR_ALIGNMENT;
  if (total_k > 0)
    for (auto st : {std::pair<int64_t, int64_t>{k_ts, k_hs}, {v_ts, v_hs}, {dk_ts, dk_hs},
                    {dv_ts, dv_hs}})
      if (!host_strides_ok(st.first, st.second, Hkv, d)) return ATTN_ERR_ALIGNMENT;
  // the cu arrays are read here to cut the chunks
  if (B > 0 && (cu_q[0] != 0 || cu_k[0] != 0 || cu_q[B] != total_q || cu_k[B] != total_k))
    return ATTN_ERR_INVALID;
  for (int b = 0; b < B; ++b)
    if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return ATTN_ERR_INVALID;
  const Plan P = plan_of(B, cu_q, cu_k, Hq, Hkv, d, chunks);
  const Layout& L = P.L;
  if (!device_buffer || device_buffer_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(device_buffer) & (kAlign - 1)))
    return ATTN_ERR_WORKSPACE;
  const int nc = P.nc;
  const std::vector<int32_t>& cut = P.cut;
  // rebased cu arrays of every chunk: chunk c's cu_q at [cut[c] + c], its cu_k
  // B + chunks entries later
  std::vector<int32_t> cus(2 * static_cast<size_t>(B + chunks), 0);
  for (int c = 0; c < nc; ++c) {
    const int s = cut[c], e = cut[c + 1];
    for (int b = s; b <= e; ++b) {
      cus[s + c + (b - s)] = cu_q[b] - cu_q[s];
      cus[B + chunks + s + c + (b - s)] = cu_k[b] - cu_k[s];
    }
  }

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* base = static_cast<uint8_t*>(device_buffer);
  int32_t* status_dev = reinterpret_cast<int32_t*>(base + L.status);
  int32_t* cu_dev = reinterpret_cast<int32_t*>(base + L.cu);
  float* slopes_dev = reinterpret_cast<float*>(base + L.slopes);
  Resources r;
  cudaEvent_t entry, done;
#define ATTN_TRY(x)                 \
  do {                              \
    if ((x) != cudaSuccess) {       \
      r.join(stream);               \
      return ATTN_ERR_CUDA;         \
    }                               \
  } while (0)
  ATTN_TRY(cudaStreamCreateWithFlags(&r.in, cudaStreamNonBlocking));
  ATTN_TRY(cudaStreamCreateWithFlags(&r.out, cudaStreamNonBlocking));
  for (int i = 0; i < kCompStreams; ++i)
    ATTN_TRY(cudaStreamCreateWithFlags(&r.comp[i], cudaStreamNonBlocking));
  ATTN_TRY(r.event(&entry));
  ATTN_TRY(r.event(&done));
  // the buffer may still be in use by earlier work on `stream`
  ATTN_TRY(cudaEventRecord(entry, stream));
  for (cudaStream_t s : {r.in, r.out, r.comp[0], r.comp[1]})
    ATTN_TRY(cudaStreamWaitEvent(s, entry, 0));
  ATTN_TRY(cudaMemsetAsync(status_dev, 0, sizeof(int32_t) * chunks, r.in));
  // small host arrays first (cus is pageable: the copy is staged before the
  // call returns)
  ATTN_TRY(cudaMemcpyAsync(cu_dev, cus.data(), sizeof(int32_t) * cus.size(),
                           cudaMemcpyHostToDevice, r.in));
  if (alibi_slopes && B > 0)
    ATTN_TRY(cudaMemcpy2DAsync(slopes_dev, sizeof(float) * Hq, alibi_slopes,
                               sizeof(float) * (B > 1 ? slopes_batch_stride : Hq),
                               sizeof(float) * Hq, B, cudaMemcpyHostToDevice, r.in));

  // Chunk c uses ring slot c % slots: its inputs go in on `in` once the slot's
  // previous chunk has come back, it computes on comp[c % 2] (so a chunk's
  // first kernels overlap the last kernels of the chunk before), and its
  // results come back on `out`.
  const int64_t qts = static_cast<int64_t>(Hq) * d, kts = static_cast<int64_t>(Hkv) * d;
  std::vector<cudaEvent_t> out_done(static_cast<size_t>(nc > 0 ? nc : 1));
  for (int c = 0; c < nc; ++c) {
    const int s = cut[c], e = cut[c + 1];
    const int64_t t0 = cu_q[s], t1 = cu_q[e], u0 = cu_k[s], u1 = cu_k[e];
    uint8_t* slot = base + L.slot0 + static_cast<size_t>(c % L.slots) * L.slot_bytes;
    cudaStream_t comp = r.comp[c % kCompStreams];
    cudaEvent_t in_done, comp_done;
    ATTN_TRY(r.event(&in_done));
    ATTN_TRY(r.event(&comp_done));
    ATTN_TRY(r.event(&out_done[c]));
    if (c >= L.slots) ATTN_TRY(cudaStreamWaitEvent(r.in, out_done[c - L.slots], 0));
    ATTN_TRY(copy_rows(true, slot + L.q, q, q_ts, q_hs, Hq, d, t0, t1, r.in));
    ATTN_TRY(copy_rows(true, slot + L.dout, dout, do_ts, do_hs, Hq, d, t0, t1, r.in));
    ATTN_TRY(copy_rows(true, slot + L.k, k, k_ts, k_hs, Hkv, d, u0, u1, r.in));
    ATTN_TRY(copy_rows(true, slot + L.v, v, v_ts, v_hs, Hkv, d, u0, u1, r.in));
    ATTN_TRY(cudaEventRecord(in_done, r.in));
    ATTN_TRY(cudaStreamWaitEvent(comp, in_done, 0));
    const attn_status st = attn_varlen_fvjp_fwd_bwd(
        dtype, e - s, Hq, Hkv, d, t1 - t0, u1 - u0, slot + L.q, qts, d, slot + L.k, kts, d,
        slot + L.v, kts, d, slot + L.dout, qts, d, cu_dev + s + c, cu_dev + B + chunks + s + c,
        alibi_slopes ? slopes_dev + static_cast<int64_t>(s) * Hq : nullptr, Hq, causal,
        window_left, window_right, softcap, scale_multiplier, slot + L.out, qts, d,
        slot + L.dq, qts, d, slot + L.dk, kts, d, slot + L.dv, kts, d,
        reinterpret_cast<float*>(slot + L.lse), slot + L.ws, L.ws_bytes, status_dev + c, comp);
    if (st != ATTN_OK) {
      r.join(stream);
      return st;
    }
    ATTN_TRY(cudaEventRecord(comp_done, comp));
    ATTN_TRY(cudaStreamWaitEvent(r.out, comp_done, 0));
    ATTN_TRY(copy_rows(false, slot + L.out, out, out_ts, out_hs, Hq, d, t0, t1, r.out));
    ATTN_TRY(copy_rows(false, slot + L.dq, dq, dq_ts, dq_hs, Hq, d, t0, t1, r.out));
    ATTN_TRY(copy_rows(false, slot + L.dk, dk, dk_ts, dk_hs, Hkv, d, u0, u1, r.out));
    ATTN_TRY(copy_rows(false, slot + L.dv, dv, dv_ts, dv_hs, Hkv, d, u0, u1, r.out));
    if (t1 > t0)
      ATTN_TRY(cudaMemcpyAsync(lse + t0 * Hq, slot + L.lse,
                               sizeof(float) * static_cast<size_t>(t1 - t0) * Hq,
                               cudaMemcpyDeviceToHost, r.out));
    ATTN_TRY(cudaEventRecord(out_done[c], r.out));
  }
  ATTN_TRY(cudaMemcpyAsync(host_status, status_dev, sizeof(int32_t) * chunks,
                           cudaMemcpyDeviceToHost, r.out));
  // the caller's stream passes the call once every result is on the host
  ATTN_TRY(cudaEventRecord(done, r.out));
  ATTN_TRY(cudaStreamWaitEvent(stream, done, 0));
#undef ATTN_TRY
  return ATTN_OK;
}
