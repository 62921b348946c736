// bwd_dkdv.cu -- the dk/dv kernel's instances without dropout, and its
// launcher (the dropout instances are compiled in bwd_dkdv_drop.cu).
#include "bwd_dkdv.cuh"

namespace attn {

template <bool B, bool M>
auto dkdv_for_d(int d) {
  return d == 128 ? dkdv_kernel<B, M, 128, 0>
                  : (d == 64 ? dkdv_kernel<B, M, 64, 0> : dkdv_kernel<B, M, 160, 0>);
}

cudaError_t launch_dkdv(const Params& p, const CUtensorMap& tq2, const CUtensorMap& tq,
                        const CUtensorMap& tdo2, const CUtensorMap& tdo, const CUtensorMap& tk2,
                        const CUtensorMap& tkt, const CUtensorMap& tv2, const CUtensorMap& tvt,
                        const CUtensorMap& tqf, const CUtensorMap& tdof, int grid, cudaStream_t s) {
  if (p.dropout)
    return launch_dkdv_drop(p, tq2, tq, tdo2, tdo, tk2, tkt, tv2, tvt, tqf, tdof, grid, s);
  const bool m = masked_call(p);
  auto k = p.dtype == 1 ? (m ? dkdv_for_d<true, true>(p.d) : dkdv_for_d<true, false>(p.d))
                        : (m ? dkdv_for_d<false, true>(p.d) : dkdv_for_d<false, false>(p.d));
  cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kSmem);
  k<<<grid, kThreads, kv::kSmem, s>>>(p, tq2, tq, tdo2, tdo, tk2, tkt, tv2, tvt, tqf, tdof);
  return cudaGetLastError();
}

}  // namespace attn
