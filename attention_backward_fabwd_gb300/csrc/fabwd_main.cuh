// Main FlashAttention backward kernel for sm_103a (tcgen05 + TMEM + TMA).
//
// What it computes is the backward of the page "CANN ops-transformer FlashAttnGrad 算子详解"
// (discosf.com/news/4863418), §一: per kv-block of 128 keys of kv-head n2, over the G q-heads of
// the group and the q-blocks that can see the block,
//     Sᵀ  = K·Qᵀ               (tcgen05, M=128 keys, N=128 queries, K=D)
//     dPᵀ = V·dOᵀ              (tcgen05, K=Dv)
//     Pᵀ  = exp2(Sᵀ·scale·log2e − lse·log2e), masked pairs -> 0          (registers)
//     dSᵀ = Pᵀ ⊙ (dPᵀ − sfmg)                                            (registers)
//     dV += Pᵀ·dO,  dK += dSᵀ·Q  (TMEM accumulators, summed over q-blocks and the G heads)
//     dQ_partial = dS·K  -> added in fp32 into the workspace accumulator (red.global.add)
// The five products are §5.2's MM2, MM1, MM5, MM4, MM3; P/dS are its V2-V4 stages.  Unlike the
// page's Ascend design, K serves as both a K-major (for Sᵀ) and an MN-major (for dQ) operand
// from one shared-memory copy by descriptor choice, and dSᵀ likewise serves dK and dQ.
//
// Shared-memory tiles are 128-byte-swizzled [64-element column block][rows][64] arrays, the
// layout TMA's SWIZZLE_128B writes for a {64, 1, rows, 1} box.
//
// Every mbarrier wait is bounded (MainArgs::wait_ns); on give-up the CTA records
// FABWD_DEV_TIMEOUT, drains what it has in flight (bounded as well), frees TMEM and returns.
#pragma once

#include "fabwd_internal.cuh"
#include "fabwd_ptx.cuh"
#include "../../include/fabwd.h"

namespace fabwd {

constexpr unsigned long long kDrainNs = 200ull * 1000ull * 1000ull;  // 200 ms

template <int D, int DV>
struct MainSmem {
  static constexpr int BR = kBlockQ, BC = kBlockKV;
  static constexpr uint32_t oK = 0;
  static constexpr uint32_t oV = oK + D * BC * 2;
  static constexpr uint32_t oQ = oV + DV * BC * 2;
  static constexpr uint32_t odO = oQ + D * BR * 2;
  static constexpr uint32_t oP = odO + DV * BR * 2;
  static constexpr uint32_t odS = oP + BC * BR * 2;
  static constexpr uint32_t oL = odS + BC * BR * 2;
  static constexpr uint32_t oF = oL + BR * 4;
  static constexpr uint32_t oBar = oF + BR * 4;
  static constexpr uint32_t oTm = oBar + 64;
  static constexpr uint32_t bytes = oTm + 64 + 1024;  // + alignment slack
  // TMEM columns (fp32 accumulators, lane = row)
  static constexpr uint32_t cDK = 0;
  static constexpr uint32_t cDV = D;
  static constexpr uint32_t cS = D + DV;
  static constexpr uint32_t cP = cS + BR;
  static constexpr uint32_t cDQ = (cP + BR + D <= 512) ? cP + BR : cS;  // alias Sᵀ when full
  static_assert(cP + BR <= 512, "TMEM budget");
  static_assert(cS + D <= 512, "TMEM budget for dQ");
};

struct SeqRange {
  int q0, L1, k0, L2;
};

__device__ __forceinline__ bool seq_range(const MainArgs& a, int b, SeqRange& r) {
  if (a.layout == kTND) {
    const long long qa = a.cu_q[b], qb = a.cu_q[b + 1], ka = a.cu_kv[b], kb = a.cu_kv[b + 1];
    if (qa < 0 || qb < qa || qb > a.T1 || qb - qa > a.S1 || ka < 0 || kb < ka || kb > a.T2 || kb - ka > a.S2)
      return false;
    r.q0 = (int)qa;
    r.L1 = (int)(qb - qa);
    r.k0 = (int)ka;
    r.L2 = (int)(kb - ka);
  } else {
    r.q0 = 0;
    r.L1 = a.S1;
    r.k0 = 0;
    r.L2 = a.S2;
  }
  return true;
}

// Visible pairs satisfy lo <= j - i - (L2 - L1) <= hi.
__device__ __forceinline__ void mask_bounds(const MainArgs& a, long long& lo, long long& hi) {
  const long long INF = 1ll << 40;
  lo = -INF;
  hi = INF;
  if (a.mask_mode != 0) {
    if (a.win_left >= 0) lo = -(long long)a.win_left;
    if (a.win_right >= 0) hi = a.win_right;
    if (a.mask_mode == 1 && hi > 0) hi = 0;
  }
}

template <int D, int DV, bool FP16>
__global__ void __launch_bounds__(128, 1)
    fabwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const MainArgs a) {
  using L = MainSmem<D, DV>;
  constexpr int BR = L::BR, BC = L::BC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, warp = tid >> 5;
  const int jb = blockIdx.x, n2 = blockIdx.y, b = blockIdx.z;

  SeqRange sq;
  if (!seq_range(a, b, sq)) return;  // bad cu_seqlens: preprocess reports it
  const int j0 = jb * BC;
  if (j0 >= sq.L2) return;
  const int j1 = min(j0 + BC, sq.L2);
  const long long off = (long long)sq.L2 - sq.L1;
  long long lo, hi;
  mask_bounds(a, lo, hi);
  // q rows that see at least one key of [j0, j1)
  long long ib = (long long)j0 - off - hi, ie = (long long)(j1 - 1) - off - lo;
  if (ib < 0) ib = 0;
  if (ie > sq.L1 - 1) ie = sq.L1 - 1;
  const int qb_begin = ib <= ie ? (int)(ib / BR) : 0;
  const int qb_end = ib <= ie ? (int)(ie / BR) + 1 : 0;
  const bool has_work = qb_begin < qb_end;

  uint8_t* sK = smem + L::oK;
  uint8_t* sV = smem + L::oV;
  uint8_t* sQ = smem + L::oQ;
  uint8_t* sdO = smem + L::odO;
  float* sL = reinterpret_cast<float*>(smem + L::oL);
  float* sF = reinterpret_cast<float*>(smem + L::oF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::oBar);
  uint64_t* kv_bar = bars + 0;
  uint64_t* q_bar = bars + 1;
  uint64_t* mma_bar = bars + 2;
  uint64_t* never_bar = bars + 3;
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + L::oTm);

  if (tid == 0) {
    mbar_init(kv_bar, 1);
    mbar_init(q_bar, 1);
    mbar_init(mma_bar, 1);
    mbar_init(never_bar, 1);
    fence_mbar_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
  }
  __syncwarp();
  if (warp == 0) tmem_alloc(tm_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tm_holder;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  const int kv_row0 = a.layout == kTND ? sq.k0 + j0 : j0;
  const int q_rowbase = a.layout == kTND ? sq.q0 : 0;
  const int bcoord = a.layout == kTND ? 0 : b;
  const bool bnsd = a.layout == kBNSD;  // BNSD maps order their coordinates (d, row, head, batch)

  bool failed = false;
  bool kv_pending = false, q_pending = false, mma_pending = false;
  uint32_t q_parity = 0, mma_parity = 0;

  if (a.inject_timeout) {
    const bool ok = mbar_wait(never_bar, 0, a.wait_ns);
    failed = __syncthreads_or(!ok);
  }

  if (!failed && has_work) {
    if (tid == 0) {
      mbar_arrive_expect_tx(kv_bar, (D + DV) * BC * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_4d(sK + c * BC * 128, &tm_k, kv_bar, c * 64, bnsd ? kv_row0 : n2, bnsd ? n2 : kv_row0, bcoord);
#pragma unroll
      for (int c = 0; c < DV / 64; ++c)
        tma_load_4d(sV + c * BC * 128, &tm_v, kv_bar, c * 64, bnsd ? kv_row0 : n2, bnsd ? n2 : kv_row0, bcoord);
    }
    kv_pending = true;
    {
      const bool ok = mbar_wait(kv_bar, 0, a.wait_ns);
      failed = __syncthreads_or(!ok);
      if (!failed) kv_pending = false;
    }
  }

  // per-thread key row (lane of Sᵀ/dPᵀ/dK/dV) and its visible q-row interval
  const int jr = j0 + tid;
  const bool j_valid = jr < sq.L2;
  long long vlo = (long long)jr - off - hi, vhi = (long long)jr - off - lo;
  const int i_vis_lo = (int)(vlo < -1 ? -1 : (vlo > (1 << 30) ? (1 << 30) : vlo));
  const int i_vis_hi = (int)(vhi < -1 ? -1 : (vhi > (1 << 30) ? (1 << 30) : vhi));

  constexpr bool kBF16 = !FP16;
  constexpr uint32_t ID_S = idesc_f16(BC, BR, kBF16, false, false);
  constexpr uint32_t ID_DV = idesc_f16(BC, DV, kBF16, false, true);
  constexpr uint32_t ID_DK = idesc_f16(BC, D, kBF16, false, true);
  constexpr uint32_t ID_DQ = idesc_f16(BR, D, kBF16, true, true);

  const uint32_t aK = smem_u32(sK), aV = smem_u32(sV), aQ = smem_u32(sQ), adO = smem_u32(sdO);
  const uint32_t aP = smem_u32(smem + L::oP), adS = smem_u32(smem + L::odS);

  bool any_acc = false;  // dK/dV accumulators hold data
  for (int h = 0; h < a.G && !failed && has_work; ++h) {
    const int n1 = n2 * a.G + h;
    const float* lse2_row = a.lse2 + ((long long)b * a.N1 + n1) * a.S1p;
    const float* sfmg_row = a.sfmg + ((long long)b * a.N1 + n1) * a.S1p;
    for (int qb = qb_begin; qb < qb_end && !failed; ++qb) {
      const int i0 = qb * BR;
      // ---- load Q, dO, lse2, sfmg tiles
      if (tid == 0) {
        mbar_arrive_expect_tx(q_bar, (D + DV) * BR * 2 + 2 * BR * 4);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sQ + c * BR * 128, &tm_q, q_bar, c * 64, bnsd ? q_rowbase + i0 : n1, bnsd ? n1 : q_rowbase + i0,
                      bcoord);
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          tma_load_4d(sdO + c * BR * 128, &tm_do, q_bar, c * 64, bnsd ? q_rowbase + i0 : n1,
                      bnsd ? n1 : q_rowbase + i0, bcoord);
        bulk_load(sL, lse2_row + i0, BR * 4, q_bar);
        bulk_load(sF, sfmg_row + i0, BR * 4, q_bar);
      }
      q_pending = true;
      {
        const bool ok = mbar_wait(q_bar, q_parity, a.wait_ns);
        if (__syncthreads_or(!ok)) { failed = true; break; }
        q_pending = false;
        q_parity ^= 1;
      }
      // ---- Sᵀ = K Qᵀ, dPᵀ = V dOᵀ
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(aK + (kk >> 2) * BC * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(aQ + (kk >> 2) * BR * 128 + (kk & 3) * 32, 16, 1024);
          mma_ss(tmem + L::cS, ad, bd, ID_S, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(aV + (kk >> 2) * BC * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(adO + (kk >> 2) * BR * 128 + (kk & 3) * 32, 16, 1024);
          mma_ss(tmem + L::cP, ad, bd, ID_S, kk > 0);
        }
        mma_commit(mma_bar);
      }
      mma_pending = true;
      {
        const bool ok = mbar_wait(mma_bar, mma_parity, a.wait_ns);
        if (__syncthreads_or(!ok)) { failed = true; break; }
        mma_pending = false;
        mma_parity ^= 1;
      }
      tc_fence_after();
      // ---- Pᵀ and dSᵀ rows (thread = key row), written as 128B-swizzled K-major tiles
      {
        const long long dmin = (long long)j0 - (i0 + BR - 1) - off, dmax = (long long)(j1 - 1) - i0 - off;
        const bool full = dmin >= lo && dmax <= hi;
#pragma unroll 1
        for (int c = 0; c < BR / 32; ++c) {
          uint32_t sr[32], pr[32];
          tmem_ld32(tmem + lane_off + L::cS + c * 32, sr);
          tmem_ld32(tmem + lane_off + L::cP + c * 32, pr);
          tmem_wait_ld();
          reg_fence(sr);
          reg_fence(pr);
          uint32_t pp[16], dd[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int col = c * 32 + e;
            float p0 = ex2(fmaf(__uint_as_float(sr[e]), a.scale_log2, -sL[col]));
            float p1 = ex2(fmaf(__uint_as_float(sr[e + 1]), a.scale_log2, -sL[col + 1]));
            if (!full) {
              const int i = i0 + col;
              if (i < i_vis_lo || i > i_vis_hi) p0 = 0.f;
              if (i + 1 < i_vis_lo || i + 1 > i_vis_hi) p1 = 0.f;
            }
            if (!j_valid) p0 = p1 = 0.f;
            const float d0 = p0 * (__uint_as_float(pr[e]) - sF[col]);
            const float d1 = p1 * (__uint_as_float(pr[e + 1]) - sF[col + 1]);
            pp[e >> 1] = pack2<FP16>(p0, p1);
            dd[e >> 1] = pack2<FP16>(d0, d1);
          }
          const uint32_t chunk = (c * 32) >> 6, u0 = ((c * 32) & 63) >> 3;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t rowoff = chunk * BC * 128 + tid * 128 + (((u0 + q) ^ (tid & 7)) << 4);
            st_shared_v4(aP + rowoff, pp[4 * q], pp[4 * q + 1], pp[4 * q + 2], pp[4 * q + 3]);
            st_shared_v4(adS + rowoff, dd[4 * q], dd[4 * q + 1], dd[4 * q + 2], dd[4 * q + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      // ---- dV += Pᵀ dO, dK += dSᵀ Q, dQ = dS K
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(aP + (kk >> 2) * BC * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(adO + kk * 2048, BR * 128, 1024);
          mma_ss(tmem + L::cDV, ad, bd, ID_DV, (any_acc || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(adS + (kk >> 2) * BC * 128 + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(aQ + kk * 2048, BR * 128, 1024);
          mma_ss(tmem + L::cDK, ad, bd, ID_DK, (any_acc || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(adS + kk * 2048, BC * 128, 1024);
          const uint64_t bd = sdesc_sw128(aK + kk * 2048, BC * 128, 1024);
          mma_ss(tmem + L::cDQ, ad, bd, ID_DQ, kk > 0);
        }
        mma_commit(mma_bar);
      }
      any_acc = true;
      mma_pending = true;
      {
        const bool ok = mbar_wait(mma_bar, mma_parity, a.wait_ns);
        if (__syncthreads_or(!ok)) { failed = true; break; }
        mma_pending = false;
        mma_parity ^= 1;
      }
      tc_fence_after();
      // ---- dQ partial (thread = q row) -> fp32 accumulator
      {
        const int ir = i0 + tid;
        const bool i_valid = ir < sq.L1;
        float* dst = a.dq_acc + row_index(a.layout, b, (long long)q_rowbase + (i_valid ? ir : 0), n1, a.N1, a.S1) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + L::cDQ + c * 32, r);
          tmem_wait_ld();
          reg_fence(r);
          if (i_valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              red_add_v4(dst + c * 32 + e, __uint_as_float(r[e]), __uint_as_float(r[e + 1]),
                         __uint_as_float(r[e + 2]), __uint_as_float(r[e + 3]));
          }
        }
      }
      tc_fence_before();
      __syncthreads();
    }
  }

  if (!failed) {
    // ---- epilogue: dK = scale · acc, dV = acc (zeros when no q row sees this block).
    // The TMEM loads are warp-collective: every thread loads, only valid rows store.
    const long long krow =
        row_index(a.layout, b, (long long)(a.layout == kTND ? sq.k0 : 0) + (j_valid ? jr : 0), n2, a.N2, a.S2);
    uint16_t* dk = static_cast<uint16_t*>(a.dk) + krow * D;
    uint16_t* dv = static_cast<uint16_t*>(a.dv) + krow * DV;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + L::cDK + c * 32, r);
      tmem_wait_ld();
      reg_fence(r);
      uint32_t o[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2)
        o[e >> 1] = any_acc ? pack2<FP16>(__uint_as_float(r[e]) * a.scale, __uint_as_float(r[e + 1]) * a.scale) : 0u;
      if (j_valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(dk + c * 32 + q * 8) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      }
    }
#pragma unroll 1
    for (int c = 0; c < DV / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_off + L::cDV + c * 32, r);
      tmem_wait_ld();
      reg_fence(r);
      uint32_t o[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2)
        o[e >> 1] = any_acc ? pack2<FP16>(__uint_as_float(r[e]), __uint_as_float(r[e + 1])) : 0u;
      if (j_valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(dv + c * 32 + q * 8) = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
      }
    }
  } else {
    if (tid == 0) {
      atomicOr(a.status, FABWD_DEV_TIMEOUT);
      if (kv_pending) mbar_wait(kv_bar, 0, kDrainNs);
      if (q_pending) mbar_wait(q_bar, q_parity, kDrainNs);
      if (mma_pending) mbar_wait(mma_bar, mma_parity, kDrainNs);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int DV, bool FP16>
cudaError_t launch_main_t(const MainArgs& a, const MainMaps& m, int grid_x, cudaStream_t st) {
  using L = MainSmem<D, DV>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fabwd_main_kernel<D, DV, FP16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::bytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(grid_x, a.N2, a.B);
  fabwd_main_kernel<D, DV, FP16><<<grid, 128, L::bytes, st>>>(m.q, m.k, m.v, m.dout, a);
  return cudaGetLastError();
}

template <bool FP16>
cudaError_t launch_main_dispatch(const MainArgs& a, const MainMaps& m, int D, int Dv, int grid_x, cudaStream_t st) {
  if (D == 64 && Dv == 64) return launch_main_t<64, 64, FP16>(a, m, grid_x, st);
  if (D == 128 && Dv == 128) return launch_main_t<128, 128, FP16>(a, m, grid_x, st);
  return cudaErrorInvalidValue;
}

}  // namespace fabwd
