// The separate dQ mode's dK/dV and dQ CTAs in one launch (fabwd_run), for one io dtype: compiled
// once with -DFABWD_INST_FP16=0 (bf16) and once with =1 (fp16).
#ifndef FABWD_INST_FP16
#error "compile with -DFABWD_INST_FP16=0 (bf16) or -DFABWD_INST_FP16=1 (fp16)"
#endif
#include "fabwd_sep.cuh"

namespace fabwd {

template <bool FP16>
cudaError_t launch_bwd(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, cudaStream_t st) {
  if (D == 64 && Dv == 64) return launch_bwd_t<64, 64, FP16>(a, m, n_kv_blocks, st);
  if (D == 128 && Dv == 64) return launch_bwd_t<128, 64, FP16>(a, m, n_kv_blocks, st);
  if (D == 128 && Dv == 128) return launch_bwd_t<128, 128, FP16>(a, m, n_kv_blocks, st);
  return cudaErrorInvalidValue;
}

template <bool FP16>
cudaError_t launch_bwd_wide(const MainArgs& a, const MainMaps& mkv, const MainMaps& mdq, int D, int Dv,
                            int n_kv_blocks, cudaStream_t st) {
  if (D == 192 && Dv == 64) return launch_bwd_wide_t<192, 64, FP16>(a, mkv, mdq, n_kv_blocks, st);
  if (D == 192 && Dv == 128) return launch_bwd_wide_t<192, 128, FP16>(a, mkv, mdq, n_kv_blocks, st);
  if (D == 192 && Dv == 192) return launch_bwd_wide_t<192, 192, FP16>(a, mkv, mdq, n_kv_blocks, st);
  return cudaErrorInvalidValue;
}

template cudaError_t launch_bwd<FABWD_INST_FP16 != 0>(const MainArgs&, const MainMaps&, int, int, int, cudaStream_t);
template cudaError_t launch_bwd_wide<FABWD_INST_FP16 != 0>(const MainArgs&, const MainMaps&, const MainMaps&, int,
                                                          int, int, cudaStream_t);

}  // namespace fabwd
