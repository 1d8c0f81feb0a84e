// fp16 instantiations of the kv-stationary and q-stationary backward kernels.
#include "fabwd_dq.cuh"
#include "fabwd_kv.cuh"
#include "fabwd_sep.cuh"
#include "fabwd_fwd.cuh"
#include "fabwd_main.cuh"

namespace fabwd {
cudaError_t launch_main_fp16(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, bool fused,
                             cudaStream_t st) {
  return fused ? launch_main_dispatch<true, true>(a, m, D, Dv, n_kv_blocks, st)
               : launch_main_dispatch<true, false>(a, m, D, Dv, n_kv_blocks, st);
}
cudaError_t launch_dq_fp16(const MainArgs& a, const MainMaps& m, int D, int Dv, cudaStream_t st) {
  return launch_dq_dispatch<true>(a, m, D, Dv, st);
}
cudaError_t launch_kv_fp16(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, cudaStream_t st) {
  if (D == 64 && Dv == 64) return launch_kv_t<64, 64, true>(a, m, n_kv_blocks, st);
  if (D == 128 && Dv == 128) return launch_kv_t<128, 128, true>(a, m, n_kv_blocks, st);
  if (D == 192 && Dv == 128) return launch_kv_t<192, 128, true>(a, m, n_kv_blocks, st);
  return cudaErrorInvalidValue;
}
cudaError_t launch_bwd_fp16(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, cudaStream_t st) {
  if (D == 64 && Dv == 64) return launch_bwd_t<64, 64, true>(a, m, n_kv_blocks, st);
  if (D == 128 && Dv == 128) return launch_bwd_t<128, 128, true>(a, m, n_kv_blocks, st);
  return cudaErrorInvalidValue;
}
cudaError_t launch_bwd_wide_fp16(const MainArgs& a, const MainMaps& mkv, const MainMaps& mdq, int D, int Dv,
                                  int n_kv_blocks, cudaStream_t st) {
  if (D == 192 && Dv == 128) return launch_bwd_wide_t<192, 128, true>(a, mkv, mdq, n_kv_blocks, st);
  return cudaErrorInvalidValue;
}
cudaError_t launch_fwd_fp16(const MainArgs& a, const MainMaps& m, int D, int Dv, cudaStream_t st) {
  return launch_fwd_dispatch<true>(a, m, D, Dv, st);
}
}  // namespace fabwd
