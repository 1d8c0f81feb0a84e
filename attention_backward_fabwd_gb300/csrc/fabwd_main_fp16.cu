// fp16 instantiations of the main backward kernel.
#include "fabwd_main.cuh"

namespace fabwd {
cudaError_t launch_main_fp16(const MainArgs& a, const MainMaps& m, int D, int Dv, int grid_x, cudaStream_t st) {
  return launch_main_dispatch<true>(a, m, D, Dv, grid_x, st);
}
}  // namespace fabwd
