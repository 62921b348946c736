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

// Offsets in the caller's device buffer.  Device copies are dense:
// [T, H, d] with token stride H*d and head stride d.
struct Layout {
  size_t ws, ws_bytes, status, cu, slopes, q, dout, out, dq, k, v, dk, dv, lse, total;
};

Layout layout(int B, int Hq, int Hkv, int d, int64_t Tq, int64_t Tk, int chunks) {
  Layout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  L.ws_bytes = attn_varlen_fvjp_workspace_size(B, Hq, Tq, Tk);
  L.ws = take(L.ws_bytes);
  L.status = take(sizeof(int32_t) * static_cast<size_t>(chunks));
  L.cu = take(sizeof(int32_t) * 2 * static_cast<size_t>(B + chunks));  // cu_q, then cu_k
  L.slopes = take(sizeof(float) * static_cast<size_t>(B) * Hq);
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
  L.total = off;
  return L;
}

// Rows [r0, r1) of a 16-bit [T, H, d] tensor between host (strides ts, hs in
// elements) and a dense device copy.  One 2-D copy when the host heads are
// dense, else one per head; feature padding is never touched.
cudaError_t copy_rows(bool to_device, void* dev, const void* host_c, int64_t ts, int64_t hs,
                      int H, int d, int64_t r0, int64_t r1, cudaStream_t s) {
  if (r1 <= r0) return cudaSuccess;
  uint8_t* host = static_cast<uint8_t*>(const_cast<void*>(host_c));
  uint8_t* devb = static_cast<uint8_t*>(dev);
  const size_t drow = static_cast<size_t>(H) * d * 2;  // device token stride (bytes)
  const size_t hpitch = static_cast<size_t>(ts) * 2;
  const size_t rows = static_cast<size_t>(r1 - r0);
  if (H == 1 || hs == d) {
    uint8_t* h = host + static_cast<size_t>(r0) * hpitch;
    uint8_t* g = devb + static_cast<size_t>(r0) * drow;
    return to_device ? cudaMemcpy2DAsync(g, drow, h, hpitch, drow, rows, cudaMemcpyHostToDevice, s)
                     : cudaMemcpy2DAsync(h, hpitch, g, drow, drow, rows, cudaMemcpyDeviceToHost, s);
  }
  for (int h = 0; h < H; ++h) {
    uint8_t* hp = host + static_cast<size_t>(r0) * hpitch + static_cast<size_t>(h) * hs * 2;
    uint8_t* gp = devb + static_cast<size_t>(r0) * drow + static_cast<size_t>(h) * d * 2;
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
  cudaStream_t in = nullptr, out = nullptr;
  std::vector<cudaEvent_t> events;
  // On an error part-way, the caller's stream still waits for the work the
  // call has enqueued on its own streams, so the caller can free its buffers
  // once it has synchronised that stream.
  void join(cudaStream_t caller) {
    for (cudaStream_t s : {in, out}) {
      cudaEvent_t e;
      if (s && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess) {
        if (cudaEventRecord(e, s) == cudaSuccess) cudaStreamWaitEvent(caller, e, 0);
        cudaEventDestroy(e);
      }
    }
  }
  ~Resources() {
    for (cudaEvent_t e : events) cudaEventDestroy(e);
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
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
  int n = 0;
  cuts[0] = 0;
  double acc = 0;
  for (int b = 0; b < B; ++b) {
    acc += static_cast<double>(cu_q[b + 1] - cu_q[b]) * (cu_k[b + 1] - cu_k[b]) + 1.0;
    if (n + 1 < chunks && b + 1 < B && acc >= total * (n + 1) / chunks) cuts[++n] = b + 1;
  }
  cuts[++n] = B;
  return n;
}

extern "C" size_t attn_varlen_fvjp_host_buffer_size(int B, int Hq, int Hkv, int head_dim,
                                                     int64_t total_q, int64_t total_k,
                                                     int chunks) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0 || total_q < 0 || total_k < 0 ||
      chunks < 1)
    return 0;
  return layout(B, Hq, Hkv, head_dim, total_q, total_k, chunks).total;
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
  const Layout L = layout(B, Hq, Hkv, d, total_q, total_k, chunks);
  if (!device_buffer || device_buffer_bytes < L.total ||
      (reinterpret_cast<uintptr_t>(device_buffer) & (kAlign - 1)))
    return ATTN_ERR_WORKSPACE;

  // ---- chunks: runs of whole sequences of about equal sum Lq*Lk
  std::vector<int> cut(static_cast<size_t>(chunks) + 1);
  const int nc = attn_varlen_host_chunks(B, cu_q, cu_k, chunks, cut.data());
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
  float* lse_dev = reinterpret_cast<float*>(base + L.lse);
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
  ATTN_TRY(r.event(&entry));
  ATTN_TRY(r.event(&done));
  // the buffer may still be in use by earlier work on `stream`
  ATTN_TRY(cudaEventRecord(entry, stream));
  ATTN_TRY(cudaStreamWaitEvent(r.in, entry, 0));
  ATTN_TRY(cudaStreamWaitEvent(r.out, entry, 0));
  ATTN_TRY(cudaMemsetAsync(status_dev, 0, sizeof(int32_t) * chunks, r.in));
  // small host arrays first (cus is pageable: the copy is staged before the
  // call returns)
  ATTN_TRY(cudaMemcpyAsync(cu_dev, cus.data(), sizeof(int32_t) * cus.size(),
                           cudaMemcpyHostToDevice, r.in));
  if (alibi_slopes && B > 0)
    ATTN_TRY(cudaMemcpy2DAsync(slopes_dev, sizeof(float) * Hq, alibi_slopes,
                               sizeof(float) * (B > 1 ? slopes_batch_stride : Hq),
                               sizeof(float) * Hq, B, cudaMemcpyHostToDevice, r.in));

  const int64_t qts = static_cast<int64_t>(Hq) * d, kts = static_cast<int64_t>(Hkv) * d;
  for (int c = 0; c < nc; ++c) {
    const int s = cut[c], e = cut[c + 1];
    const int64_t t0 = cu_q[s], t1 = cu_q[e], u0 = cu_k[s], u1 = cu_k[e];
    cudaEvent_t in_done, comp_done;
    ATTN_TRY(r.event(&in_done));
    ATTN_TRY(r.event(&comp_done));
    // inputs of chunk c
    ATTN_TRY(copy_rows(true, base + L.q, q, q_ts, q_hs, Hq, d, t0, t1, r.in));
    ATTN_TRY(copy_rows(true, base + L.dout, dout, do_ts, do_hs, Hq, d, t0, t1, r.in));
    ATTN_TRY(copy_rows(true, base + L.k, k, k_ts, k_hs, Hkv, d, u0, u1, r.in));
    ATTN_TRY(copy_rows(true, base + L.v, v, v_ts, v_hs, Hkv, d, u0, u1, r.in));
    ATTN_TRY(cudaEventRecord(in_done, r.in));
    // the call on the chunk
    ATTN_TRY(cudaStreamWaitEvent(stream, in_done, 0));
    auto at = [&](size_t off, int64_t row, int64_t rowlen) -> uint16_t* {
      return reinterpret_cast<uint16_t*>(base + off) + row * rowlen;
    };
    const attn_status st = attn_varlen_fvjp_fwd_bwd(
        dtype, e - s, Hq, Hkv, d, t1 - t0, u1 - u0, at(L.q, t0, qts), qts, d, at(L.k, u0, kts),
        kts, d, at(L.v, u0, kts), kts, d, at(L.dout, t0, qts), qts, d, cu_dev + s + c,
        cu_dev + B + chunks + s + c, alibi_slopes ? slopes_dev + static_cast<int64_t>(s) * Hq : nullptr,
        Hq, causal, window_left, window_right, softcap, scale_multiplier, at(L.out, t0, qts), qts,
        d, at(L.dq, t0, qts), qts, d, at(L.dk, u0, kts), kts, d, at(L.dv, u0, kts), kts, d,
        lse_dev + t0 * Hq, base + L.ws, L.ws_bytes, status_dev + c, stream);
    if (st != ATTN_OK) {
      r.join(stream);
      return st;
    }
    ATTN_TRY(cudaEventRecord(comp_done, stream));
    // results of chunk c
    ATTN_TRY(cudaStreamWaitEvent(r.out, comp_done, 0));
    ATTN_TRY(copy_rows(false, base + L.out, out, out_ts, out_hs, Hq, d, t0, t1, r.out));
    ATTN_TRY(copy_rows(false, base + L.dq, dq, dq_ts, dq_hs, Hq, d, t0, t1, r.out));
    ATTN_TRY(copy_rows(false, base + L.dk, dk, dk_ts, dk_hs, Hkv, d, u0, u1, r.out));
    ATTN_TRY(copy_rows(false, base + L.dv, dv, dv_ts, dv_hs, Hkv, d, u0, u1, r.out));
    if (t1 > t0)
      ATTN_TRY(cudaMemcpyAsync(lse + t0 * Hq, lse_dev + t0 * Hq,
                               sizeof(float) * static_cast<size_t>(t1 - t0) * Hq,
                               cudaMemcpyDeviceToHost, r.out));
  }
  ATTN_TRY(cudaMemcpyAsync(host_status, status_dev, sizeof(int32_t) * chunks,
                           cudaMemcpyDeviceToHost, r.out));
  // the caller's stream passes the call once every result is on the host
  ATTN_TRY(cudaEventRecord(done, r.out));
  ATTN_TRY(cudaStreamWaitEvent(stream, done, 0));
#undef ATTN_TRY
  return ATTN_OK;
}
