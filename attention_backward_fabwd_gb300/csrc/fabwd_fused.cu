// The fused kernel of the atomic dQ mode, for one io dtype: compiled once with
// -DFABWD_INST_FP16=0 (bf16) and once with =1 (fp16).  No (192, 192) kernel: dK and dV would
// take 384 of the 512 TMEM columns, leaving too few for the slot and the second dQᵀ part.
#ifndef FABWD_INST_FP16
#error "compile with -DFABWD_INST_FP16=0 (bf16) or -DFABWD_INST_FP16=1 (fp16)"
#endif
#include "fabwd_main.cuh"

namespace fabwd {

template <bool FP16>
cudaError_t launch_main(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, cudaStream_t st) {
  if (D == 64 && Dv == 64) return launch_main_t<64, 64, FP16>(a, m, n_kv_blocks, st);
  if (D == 128 && Dv == 64) return launch_main_t<128, 64, FP16>(a, m, n_kv_blocks, st);
  if (D == 128 && Dv == 128) return launch_main_t<128, 128, FP16>(a, m, n_kv_blocks, st);
  if (D == 192 && Dv == 64) return launch_main_t<192, 64, FP16>(a, m, n_kv_blocks, st);
  if (D == 192 && Dv == 128) return launch_main_t<192, 128, FP16>(a, m, n_kv_blocks, st);
  return cudaErrorInvalidValue;
}

template cudaError_t launch_main<FABWD_INST_FP16 != 0>(const MainArgs&, const MainMaps&, int, int, int, cudaStream_t);

}  // namespace fabwd
