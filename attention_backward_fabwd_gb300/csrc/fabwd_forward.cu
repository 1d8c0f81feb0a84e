// The forward kernel (fabwd_forward), for one io dtype: compiled once with -DFABWD_INST_FP16=0
// (bf16) and once with =1 (fp16).
#ifndef FABWD_INST_FP16
#error "compile with -DFABWD_INST_FP16=0 (bf16) or -DFABWD_INST_FP16=1 (fp16)"
#endif
#include "fabwd_fwd.cuh"

namespace fabwd {

template <bool FP16>
cudaError_t launch_fwd(const MainArgs& a, const MainMaps& m, int D, int Dv, cudaStream_t st) {
  if (D == 64 && Dv == 64) return launch_fwd_t<64, 64, FP16>(a, m, st);
  if (D == 128 && Dv == 64) return launch_fwd_t<128, 64, FP16>(a, m, st);
  if (D == 128 && Dv == 128) return launch_fwd_t<128, 128, FP16>(a, m, st);
  if (D == 192 && Dv == 64) return launch_fwd_t<192, 64, FP16>(a, m, st);
  if (D == 192 && Dv == 128) return launch_fwd_t<192, 128, FP16>(a, m, st);
  if (D == 192 && Dv == 192) return launch_fwd_t<192, 192, FP16>(a, m, st);
  return cudaErrorInvalidValue;
}

template cudaError_t launch_fwd<FABWD_INST_FP16 != 0>(const MainArgs&, const MainMaps&, int, int, cudaStream_t);

}  // namespace fabwd
