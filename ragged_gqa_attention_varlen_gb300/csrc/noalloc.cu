// noalloc.cu -- the fused forward + VJP call for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc at all: a plugin running inside a host
// framework that owns every device allocation through its own allocator, or
// a latency-critical service that forbids allocator calls (which can
// synchronise the device) once it is serving.  The ordinary entry point needs
// a caller-provided workspace; this one uses a fixed scratch array compiled
// into the library instead, so such a caller only passes inputs and outputs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/attn_varlen.h"
#include "attn_internal.h"

namespace {

// The scratch: status word, tile counters, tile schedule and the fp32 D term
// of the backward pass.  Every GPU that loads the library holds these
// ATTN_NOALLOC_SCRATCH_BYTES until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

// The array's device address belongs to the context the library's module is
// loaded in.  It is looked up once per device and context: a new context on
// the same device (after cudaDeviceReset, or once the primary context was
// released and created again) loads the module again, and the array may then
// live elsewhere.  Contexts are told apart by their process-unique id.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, std::atomic<Fn>& slot) {
  Fn f = slot.load();
  if (f) return f;
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  f = reinterpret_cast<Fn>(ptr);
  slot.store(f);
  return f;
}

// Id of the context current on this thread; false when there is none yet or
// the driver functions are unavailable.
bool current_context_id(unsigned long long* id) {
  static std::atomic<CtxGetCurrentFn> get_current{nullptr};
  static std::atomic<CtxGetIdFn> get_id{nullptr};
  CtxGetCurrentFn cur = driver_fn("cuCtxGetCurrent", get_current);
  CtxGetIdFn gid = driver_fn("cuCtxGetId", get_id);
  if (!cur || !gid) return false;
  CUcontext ctx = nullptr;
  if (cur(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return gid(ctx, id) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
struct Entry {
  unsigned long long ctx_id;
  void* addr;
};
Entry g_entry[kMaxDevices];
std::mutex g_entry_mu;

// In host code the array's name is only a host-side stand-in; its device
// address comes from the runtime, with the device current.
attn_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_entry_mu);
  if (have_id && g_entry[dev].addr && g_entry[dev].ctx_id == id) {
    *out = g_entry[dev].addr;
    return ATTN_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ATTN_ERR_CUDA;
  // the lookup makes the device's primary context current if none was; the
  // address is kept only when the context it belongs to is known
  if (have_id || current_context_id(&id))
    g_entry[dev] = Entry{id, p};
  else
    g_entry[dev] = Entry{0, nullptr};
  *out = p;
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_varlen_fvjp_fwd_bwd_noalloc(
    attn_dtype dtype, int B, int Hq, int Hkv, int head_dim, int64_t total_q, int64_t total_k,
    const void* q, int64_t q_ts, int64_t q_hs, const void* k, int64_t k_ts, int64_t k_hs,
    const void* v, int64_t v_ts, int64_t v_hs, const void* dout, int64_t do_ts, int64_t do_hs,
    const int32_t* cu_q, const int32_t* cu_k, const float* alibi_slopes,
    int64_t slopes_batch_stride, int causal, int window_left, int window_right, float softcap,
    float scale_multiplier, void* out, int64_t out_ts, int64_t out_hs, void* dq, int64_t dq_ts,
    int64_t dq_hs, void* dk, int64_t dk_ts, int64_t dk_hs, void* dv, int64_t dv_ts,
    int64_t dv_hs, float* lse, int32_t* device_status, void* stream) {
  if (B < 0 || Hq <= 0 || total_q < 0 || total_k < 0) return ATTN_ERR_INVALID;
  // no dropout here, so the workspace's per-token rate table is not needed
  if (attn::workspace_bytes_needed(B, Hq, total_q, false) > ATTN_NOALLOC_SCRATCH_BYTES)
    return ATTN_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  attn_status s = scratch_address(&scratch);
  if (s != ATTN_OK) return s;
  return attn_varlen_fvjp_fwd_bwd(
      dtype, B, Hq, Hkv, head_dim, total_q, total_k, q, q_ts, q_hs, k, k_ts, k_hs, v, v_ts, v_hs,
      dout, do_ts, do_hs, cu_q, cu_k, alibi_slopes, slopes_batch_stride, causal, window_left,
      window_right, softcap, scale_multiplier, out, out_ts, out_hs, dq, dq_ts, dq_hs, dk, dk_ts,
      dk_hs, dv, dv_ts, dv_hs, lse, scratch, ATTN_NOALLOC_SCRATCH_BYTES, device_status, stream);
}
