// One launch for the whole separate-mode backward: the CTAs of the dK/dV kernel
// (heaviest key blocks first) followed by those of the dQ kernel (heaviest query blocks first).
// Both CTA kinds take one SM each (shared memory and all 512 TMEM columns), read only the
// inputs and the preprocess rows, and write disjoint outputs, so they need no ordering between
// them; putting them in one grid lets the dQ CTAs fill the SMs that the short dK/dV CTAs leave
// while the long ones (the first key blocks under a causal mask) are still running, instead of
// the dK/dV grid's tail leaving SMs idle before a second launch.
#pragma once

#include "fabwd_dq.cuh"
#include "fabwd_kv.cuh"

namespace fabwd {

// Launch configuration with programmatic stream serialisation: the grid may start while the
// preceding kernel on the stream (the preprocess) finishes; its CTAs wait for it (griddep_wait)
// after their set-up.  attr is the caller's, valid for the launch call.
inline cudaLaunchConfig_t pdl_config(dim3 grid, int threads, uint32_t smem, cudaStream_t st, cudaLaunchAttribute* attr) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// Which CTA kind and unit blockIdx stands for.  BSND / BNSD (and varlen with many sequences):
// grid (kv_ctas + dQ units, B), the dK/dV units first.  Varlen (FLAT): a flat grid over every
// sequence's dK/dV units and then its dQ units, the sequences back to back (flat_unit), so that
// short sequences leave no CTAs that only exit; CTAs past the last unit return.
struct GridUnit {
  int b, local, nqb;
  bool kv;
};
template <bool FLAT>
__device__ __forceinline__ bool grid_unit(const MainArgs& a, int kv_ctas, int kv_rows, int q_rows, GridUnit& u) {
  if constexpr (FLAT) {
    return flat_unit(a, blockIdx.x, kv_rows, q_rows, u.b, u.local, u.kv, u.nqb);
  } else {
    u.b = blockIdx.y;
    u.kv = (int)blockIdx.x < kv_ctas;
    u.local = u.kv ? (int)blockIdx.x : (int)blockIdx.x - kv_ctas;
    u.nqb = (a.S1 + q_rows - 1) / q_rows;
    return true;
  }
}

// Grid of the one-grid launch: (dK/dV units + dQ units, B), or the flat varlen grid's bound.
inline dim3 one_grid(const MainArgs& a, int n_kv_blocks, int kv_rows, int q_rows) {
  if (flat_grid(a.layout, a.B))
    return dim3((unsigned)(tnd_blocks_bound(a.B, a.S2, a.T2, kv_rows) * a.N2 +
                           tnd_blocks_bound(a.B, a.S1, a.T1, q_rows) * a.N1),
                1);
  return dim3(n_kv_blocks * a.N2 + ((a.S1 + q_rows - 1) / q_rows) * a.N1, a.B);
}

template <int D, int DV, bool FP16, bool FLAT>
__global__ void __launch_bounds__(kMainThreads, 1)
    fabwd_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv, const MainArgs a, int kv_ctas) {
  GridUnit u;
  if (!grid_unit<FLAT>(a, kv_ctas, KvCfg<D, DV>::BC, DqCfg<D, DV>::BM, u)) return;
  if (u.kv)
    kv_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv, a, u.local, u.b);
  else
    dq_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_do, tm_dq, a, u.local, u.b, u.nqb);
}

template <int D, int DV, bool FP16, bool FLAT>
cudaError_t launch_bwd_flat(const MainArgs& a, const MainMaps& m, int n_kv_blocks, cudaStream_t st) {
  static_assert(DqCfg<D, DV>::BN == KvCfg<D, DV>::BC, "one tensor map box for both CTA kinds");
  constexpr uint32_t bytes = KvCfg<D, DV>::bytes > DqCfg<D, DV>::bytes ? KvCfg<D, DV>::bytes : DqCfg<D, DV>::bytes;
  if (cudaError_t e = ensure_smem_limit<fabwd_bwd_kernel<D, DV, FP16, FLAT>>((int)bytes); e != cudaSuccess)
    return e;
  const int kv_ctas = n_kv_blocks * a.N2;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(one_grid(a, n_kv_blocks, KvCfg<D, DV>::BC, DqCfg<D, DV>::BM), kMainThreads,
                                      bytes, st, attr);
  return cudaLaunchKernelEx(&cfg, fabwd_bwd_kernel<D, DV, FP16, FLAT>, m.q, m.k, m.v, m.dout, m.dq, m.dk, m.dv, a,
                            kv_ctas);
}

template <int D, int DV, bool FP16>
cudaError_t launch_bwd_t(const MainArgs& a, const MainMaps& m, int n_kv_blocks, cudaStream_t st) {
  return flat_grid(a.layout, a.B) ? launch_bwd_flat<D, DV, FP16, true>(a, m, n_kv_blocks, st)
                                  : launch_bwd_flat<D, DV, FP16, false>(a, m, n_kv_blocks, st);
}

// D > 128: the two CTA kinds take different tensor-map boxes (the dK/dV CTAs stream 64-row query
// tiles against 128 resident keys, the dQ CTAs 96-key tiles against 128 resident queries), so
// this grid gets both sets of maps.
template <int D, int DV, bool FP16, bool FLAT>
__global__ void __launch_bounds__(kMainThreads, 1)
    fabwd_bwd_wide_kernel(const __grid_constant__ CUtensorMap kq, const __grid_constant__ CUtensorMap kk,
                          const __grid_constant__ CUtensorMap kvv, const __grid_constant__ CUtensorMap kdo,
                          const __grid_constant__ CUtensorMap qq, const __grid_constant__ CUtensorMap qk,
                          const __grid_constant__ CUtensorMap qv, const __grid_constant__ CUtensorMap qdo,
                          const __grid_constant__ CUtensorMap out_dq, const __grid_constant__ CUtensorMap out_dk,
                          const __grid_constant__ CUtensorMap out_dv, const MainArgs a, int kv_ctas) {
  GridUnit u;
  if (!grid_unit<FLAT>(a, kv_ctas, KvCfg<D, DV>::BC, DqCfg<D, DV>::BM, u)) return;
  if (u.kv)
    kv_block<D, DV, FP16>(kq, kk, kvv, kdo, out_dk, out_dv, a, u.local, u.b);
  else
    dq_block<D, DV, FP16>(qq, qk, qv, qdo, out_dq, a, u.local, u.b, u.nqb);
}

template <int D, int DV, bool FP16, bool FLAT>
cudaError_t launch_bwd_wide_flat(const MainArgs& a, const MainMaps& mkv, const MainMaps& mdq, int n_kv_blocks,
                                 cudaStream_t st) {
  constexpr uint32_t kb = KvCfg<D, DV>::bytes, qb = DqCfg<D, DV>::bytes;
  constexpr uint32_t bytes = kb > qb ? kb : qb;
  if (cudaError_t e = ensure_smem_limit<fabwd_bwd_wide_kernel<D, DV, FP16, FLAT>>((int)bytes); e != cudaSuccess)
    return e;
  const int kv_ctas = n_kv_blocks * a.N2;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pdl_config(one_grid(a, n_kv_blocks, KvCfg<D, DV>::BC, DqCfg<D, DV>::BM), kMainThreads,
                                      bytes, st, attr);
  return cudaLaunchKernelEx(&cfg, fabwd_bwd_wide_kernel<D, DV, FP16, FLAT>, mkv.q, mkv.k, mkv.v, mkv.dout, mdq.q,
                            mdq.k, mdq.v, mdq.dout, mdq.dq, mkv.dk, mkv.dv, a, kv_ctas);
}

template <int D, int DV, bool FP16>
cudaError_t launch_bwd_wide_t(const MainArgs& a, const MainMaps& mkv, const MainMaps& mdq, int n_kv_blocks,
                              cudaStream_t st) {
  return flat_grid(a.layout, a.B) ? launch_bwd_wide_flat<D, DV, FP16, true>(a, mkv, mdq, n_kv_blocks, st)
                                  : launch_bwd_wide_flat<D, DV, FP16, false>(a, mkv, mdq, n_kv_blocks, st);
}

}  // namespace fabwd
