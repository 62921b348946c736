// bwd_dkdv_dmask.cu -- the dk/dv kernel's dropout instances that read the
// stored keep mask (one rate or a rate per query token; head dimensions 160,
// 128 and 64), compiled apart from the hashing instances.
#include "bwd_dkdv.cuh"

namespace attn {

template <bool B, bool M, int DM, bool C>
auto dkdv_dmask_for_d(int d) {
  return d == 128 ? dkdv_kernel<B, M, 128, DM, C>
                  : (d == 64 ? dkdv_kernel<B, M, 64, DM, C> : dkdv_kernel<B, M, 160, DM, C>);
}

// the call's one rate takes instances with a known cap when the call is
// capped (softcap > 0); per-token rates read the cap at run time
template <bool B, bool M>
auto dkdv_dmask_kernel(int d, bool table, bool cap) {
  return table ? dkdv_dmask_for_d<B, M, 4, false>(d)
               : (cap ? dkdv_dmask_for_d<B, M, 3, true>(d) : dkdv_dmask_for_d<B, M, 3, false>(d));
}

cudaError_t launch_dkdv_dmask(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tq,
                              const CUtensorMap& tdo2, const CUtensorMap& tdo,
                              const CUtensorMap& tk2, const CUtensorMap& tkt,
                              const CUtensorMap& tv2, const CUtensorMap& tvt,
                              int grid, cudaStream_t s) {
  const bool m = masked_call(p);
  const bool tab = p.drop_tab != nullptr;
  const bool cap = p.softcap > 0.f;
  auto k = p.dtype == 1 ? (m ? dkdv_dmask_kernel<true, true>(p.d, tab, cap)
                             : dkdv_dmask_kernel<true, false>(p.d, tab, cap))
                        : (m ? dkdv_dmask_kernel<false, true>(p.d, tab, cap)
                             : dkdv_dmask_kernel<false, false>(p.d, tab, cap));
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kSmem);
  k<<<grid, kThreads, kv::kSmem, s>>>(p, tq2, tq, tdo2, tdo, tk2, tkt, tv2, tvt);
  return cudaGetLastError();
}

}  // namespace attn
