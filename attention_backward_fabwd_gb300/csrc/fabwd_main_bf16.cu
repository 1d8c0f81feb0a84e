// bf16 instantiations of the kv-stationary and q-stationary backward kernels.
#include "fabwd_dq.cuh"
#include "fabwd_main.cuh"

namespace fabwd {
cudaError_t launch_main_bf16(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, bool fused,
                             cudaStream_t st) {
  return fused ? launch_main_dispatch<false, true>(a, m, D, Dv, n_kv_blocks, st)
               : launch_main_dispatch<false, false>(a, m, D, Dv, n_kv_blocks, st);
}
cudaError_t launch_dq_bf16(const MainArgs& a, const MainMaps& m, int D, int Dv, cudaStream_t st) {
  return launch_dq_dispatch<false>(a, m, D, Dv, st);
}
}  // namespace fabwd
