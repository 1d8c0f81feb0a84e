// The separate dQ mode's two kernels as separate launches (fabwd_run_main: dK/dV; fabwd_run_dq:
// dQ), for one io dtype: compiled once with -DFABWD_INST_FP16=0 (bf16) and once with =1 (fp16).
#ifndef FABWD_INST_FP16
#error "compile with -DFABWD_INST_FP16=0 (bf16) or -DFABWD_INST_FP16=1 (fp16)"
#endif
#include "fabwd_dq.cuh"
#include "fabwd_kv.cuh"

namespace fabwd {

template <bool FP16>
cudaError_t launch_kv(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, cudaStream_t st) {
  if (D == 64 && Dv == 64) return launch_kv_t<64, 64, FP16>(a, m, n_kv_blocks, st);
  if (D == 128 && Dv == 64) return launch_kv_t<128, 64, FP16>(a, m, n_kv_blocks, st);
  if (D == 128 && Dv == 128) return launch_kv_t<128, 128, FP16>(a, m, n_kv_blocks, st);
  if (D == 192 && Dv == 64) return launch_kv_t<192, 64, FP16>(a, m, n_kv_blocks, st);
  if (D == 192 && Dv == 128) return launch_kv_t<192, 128, FP16>(a, m, n_kv_blocks, st);
  if (D == 192 && Dv == 192) return launch_kv_t<192, 192, FP16>(a, m, n_kv_blocks, st);
  return cudaErrorInvalidValue;
}

template <bool FP16>
cudaError_t launch_dq(const MainArgs& a, const MainMaps& m, int D, int Dv, cudaStream_t st) {
  if (D == 64 && Dv == 64) return launch_dq_t<64, 64, FP16>(a, m, st);
  if (D == 128 && Dv == 64) return launch_dq_t<128, 64, FP16>(a, m, st);
  if (D == 128 && Dv == 128) return launch_dq_t<128, 128, FP16>(a, m, st);
  if (D == 192 && Dv == 64) return launch_dq_t<192, 64, FP16>(a, m, st);
  if (D == 192 && Dv == 128) return launch_dq_t<192, 128, FP16>(a, m, st);
  if (D == 192 && Dv == 192) return launch_dq_t<192, 192, FP16>(a, m, st);
  return cudaErrorInvalidValue;
}

template cudaError_t launch_kv<FABWD_INST_FP16 != 0>(const MainArgs&, const MainMaps&, int, int, int, cudaStream_t);
template cudaError_t launch_dq<FABWD_INST_FP16 != 0>(const MainArgs&, const MainMaps&, int, int, cudaStream_t);

}  // namespace fabwd
