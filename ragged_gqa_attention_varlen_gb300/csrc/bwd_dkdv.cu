// bwd_dkdv.cu -- the dk/dv kernel's instances without dropout, and its
// launcher (the dropout instances are compiled in bwd_dkdv_drop.cu).
#include "bwd_dkdv.cuh"

namespace attn {

template <bool B, bool M, bool C>
auto dkdv_for_d(int d) {
  return d == 128 ? dkdv_kernel<B, M, 128, 0, C>
                  : (d == 64 ? dkdv_kernel<B, M, 64, 0, C> : dkdv_kernel<B, M, 160, 0, C>);
}

template <bool C>
auto dkdv_pick(const Params& p) {
  const bool m = masked_call(p);
  return p.dtype == 1 ? (m ? dkdv_for_d<true, true, C>(p.d) : dkdv_for_d<true, false, C>(p.d))
                      : (m ? dkdv_for_d<false, true, C>(p.d) : dkdv_for_d<false, false, C>(p.d));
}

cudaError_t launch_dkdv(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tq,
                        const CUtensorMap& tdo2, const CUtensorMap& tdo, const CUtensorMap& tk2,
                        const CUtensorMap& tkt, const CUtensorMap& tv2, const CUtensorMap& tvt,
                        int grid, cudaStream_t s) {
  if (p.dropout)
    return launch_dkdv_drop(p, tq2, tq, tdo2, tdo, tk2, tkt, tv2, tvt, grid, s);
  // instances for capped calls (the logit map's cap test: softcap > 0)
  auto k = p.softcap > 0.f ? dkdv_pick<true>(p) : dkdv_pick<false>(p);
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kSmem);
  k<<<grid, kThreads, kv::kSmem, s>>>(p, tq2, tq, tdo2, tdo, tk2, tkt, tv2, tvt);
  return cudaGetLastError();
}

}  // namespace attn
