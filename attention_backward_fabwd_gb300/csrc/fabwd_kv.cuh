// kv-stationary dK/dV kernel of the separate dQ mode: 128-row query steps up to D = 128, 64-row
// steps at D = 192 (where dK alone takes 192 of the 512 TMEM columns).
//
// What it computes is dK and dV of the page "CANN ops-transformer FlashAttnGrad 算子详解"
// (discosf.com/news/4863418), §一: dV = Pᵀ·dY and dK = scale·dSᵀ·Q with P = exp(scale·QKᵀ − lse)
// and dS = P ⊙ (dY·Vᵀ − sfmg), summed over the query blocks and the G q-heads of a kv-head.
// One CTA owns 128 keys of one kv-head; each step handles BR query rows of one q-head:
//     Sᵀ  = K·Qᵀ     tcgen05 M = 128 keys, N = BR queries (128: a full-rate shape), TMEM slot S
//     dPᵀ = V·dOᵀ    same shape, TMEM slot dP
//     Pᵀ  = exp2(Sᵀ·scale·log2e − lse·log2e) -> 16-bit pairs over the warpgroup's own Sᵀ columns
//     −dSᵀ = Pᵀ ⊙ (sfmg − dPᵀ)              -> 16-bit pairs over its own dPᵀ columns
//     dV += Pᵀ·dO, dK −= (−dSᵀ)·Q            tcgen05 with the A operand read from TMEM; the
//                                           epilogue writes −scale times the accumulator
// The elementwise steps use packed fp32x2 FMA and multiply; the signs are chosen so that no
// per-element negation of the lse and sfmg vectors is needed.
// Warpgroup g (warps 4g..4g+3) handles query columns [NCW·g, NCW·g + NCW) of every step, NCW = BR/2.
// Keeping dSᵀ in
// the dPᵀ columns frees the Sᵀ columns as soon as dV has read Pᵀ, so the MMA warp issues
//     Sᵀ(t), dPᵀ(t), dV(t), Sᵀ(t+1), dK(t), dPᵀ(t+1), dV(t+1), ...
// and the elementwise work of each step overlaps the previous step's dK and the next step's Sᵀ.
// Warp 8 streams Q with lse·log2e through a 3-stage TMA ring and dO with sfmg through a 2-stage
// ring (K and V are loaded once); a Q stage is released by a commit after dK, a dO stage by a commit
// after dV together with an arrival of every compute warp once it has read the stage's sfmg.
// One thread issues every tcgen05.mma, and an MMA of this shape occupies it about as long as the
// tensor pipe takes to run it, so each barrier wait between MMA groups idles the pipe.  The MMA
// thread therefore waits only for the compute warps' P and dS handoffs; the compute warps wait
// for the TMA stages the MMA thread reads next (Q(t+1) before they hand over P(t), dO(t+1) before
// dS(t)), which falls where they would otherwise idle.
// TMEM columns: dK [0, D), dV [D, D+Dv), Sᵀ/Pᵀ [D+Dv, +BR), dPᵀ/dSᵀ [D+Dv+BR, +BR).
// Bounded waits, abort flag, drain and TMEM release as in the fused kernel.
#pragma once

#include "fabwd_internal.cuh"
#include "fabwd_main.cuh"
#include "fabwd_ptx.cuh"
#include "../../include/fabwd.h"

namespace fabwd {

template <int D, int DV>
struct KvCfg {
  // 128 query rows per step up to D = 128; 64 at D = 192, where dK alone takes 192 TMEM columns
  static constexpr int BR = D > 128 ? 64 : 128, BC = kBlockKV, NQ = 3, NO = 2;  // Q ring and dO ring stages
  static constexpr int NCW = BR / 2;  // query columns of each compute warpgroup
  static constexpr uint32_t kK = D * BC * 2, kV = DV * BC * 2, kQ = D * BR * 2, kdO = DV * BR * 2;
  static constexpr uint32_t oK = 0, oV = oK + kK, oQ = oV + kV, odO = oQ + NQ * kQ;
  static constexpr uint32_t oL = odO + NO * kdO;     // [NQ][BR] fp32 lse·log2(e)
  static constexpr uint32_t oF = oL + NQ * BR * 4;   // [NO][BR] fp32 sfmg
  static constexpr uint32_t oBar = oF + NO * BR * 4;
  static constexpr uint32_t oMisc = oBar + 20 * 8;
  static constexpr uint32_t bytes = oMisc + 64;
  static constexpr uint32_t cDK = 0, cDV = D, cS = D + DV, cP = cS + BR;
  static_assert(D % 64 == 0 && DV % 64 == 0 && DV <= D && D <= 192, "head dims");
  static_assert(cP + BR <= 512, "TMEM budget");
  static_assert(DV / 64 * BC * 128 <= NO * kdO, "dV staging fits in the dO ring");
  static_assert(D / 64 * BC * 128 <= NQ * kQ, "dK staging fits in the Q ring");
  static_assert(bytes <= 232448, "shared memory budget");
};

constexpr int kKvKvFull = 0, kKvQFull = 1 /*+3*/, kKvQEmpty = 4 /*+3*/, kKvOFull = 7 /*+2*/, kKvOEmpty = 9 /*+2*/,
              kKvSFull = 11, kKvDpFull = 12, kKvPFull = 13, kKvDsFull = 14, kKvAccDone = 15, kKvNever = 16,
              kKvDrain = 17, kKvNumBars = 18;

// One CTA of the dK/dV kernel: key block bx / N2 of kv-head bx % N2, batch (or sequence) by.
template <int D, int DV, bool FP16>
__device__ __forceinline__ void kv_block(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                         const CUtensorMap& tm_do, const CUtensorMap& tm_dk, const CUtensorMap& tm_dv,
                                         const MainArgs& a, int bx, int by) {
  using C = KvCfg<D, DV>;
  constexpr int BR = C::BR, BC = C::BC, NQ = C::NQ, NO = C::NO;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int jb = bx / a.N2, n2 = bx % a.N2, b = by;
  SeqRange sq;
  if (!seq_range(a, b, sq)) return;  // bad cu_seqlens: the preprocess kernel reports it
  const int j0 = jb * BC;
  if (j0 >= sq.L2) return;
  if ((smem_u32(smem) & 1023u) != 0) {
    griddep_wait();  // the preprocess clears the status word
    if (tid == 0) atomicOr(a.status, FABWD_DEV_INTERNAL);
    return;
  }
  const int j1 = min(j0 + BC, sq.L2);
  const long long off = (long long)sq.L2 - sq.L1;
  long long lo, hi;
  mask_bounds(a, lo, hi);
  long long ib = (long long)j0 - off - hi, ie = (long long)(j1 - 1) - off - lo;
  if (ib < 0) ib = 0;
  if (ie > sq.L1 - 1) ie = sq.L1 - 1;
  const int qb_begin = ib <= ie ? (int)(ib / BR) : 0;
  const int nqb = ib <= ie ? (int)(ie / BR) + 1 - qb_begin : 0;
  const int T = nqb * a.G;  // steps: (head in group, 128-row q-block)

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::oBar);
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + C::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oMisc + 16);
  const bool tnd = a.layout == kTND, bnsd = a.layout == kBNSD;
  const int kv_row0 = tnd ? sq.k0 + j0 : j0;
  const int q_rowbase = tnd ? sq.q0 : 0;
  const int bcoord = tnd ? 0 : b;
  if (warp == 8 && lane == 0) {
    for (int i = 0; i < kKvNumBars; ++i) {
      // P/dS handoffs: one arrival per compute warp; a dO stage: the dV commit + 8 compute warps
      const bool oe = i >= kKvOEmpty && i < kKvOEmpty + NO;
      mbar_init(&bars[i], (i == kKvPFull || i == kKvDsFull) ? 8 : (oe ? 9 : 1));
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
    if (T > 0) {
      // K, V and the Q and dO tiles of step 0 are inputs (the preprocess writes none of them):
      // they load while the CTA allocates TMEM and waits for the preprocess; step 0's lse and
      // sfmg rows follow after that wait (the stages' byte counts include them)
      mbar_arrive_expect_tx(&bars[kKvKvFull], (D + DV) * BC * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_4d(smem + C::oK + c * BC * 128, &tm_k, &bars[kKvKvFull], c * 64, bnsd ? kv_row0 : n2,
                    bnsd ? n2 : kv_row0, bcoord);
#pragma unroll
      for (int c = 0; c < DV / 64; ++c)
        tma_load_4d(smem + C::oV + c * BC * 128, &tm_v, &bars[kKvKvFull], c * 64, bnsd ? kv_row0 : n2,
                    bnsd ? n2 : kv_row0, bcoord);
      const int row = q_rowbase + qb_begin * BR, n1 = n2 * a.G;
      mbar_arrive_expect_tx(&bars[kKvQFull], D * BR * 2 + BR * 4);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_4d(smem + C::oQ + c * BR * 128, &tm_q, &bars[kKvQFull], c * 64, bnsd ? row : n1, bnsd ? n1 : row,
                    bcoord);
      mbar_arrive_expect_tx(&bars[kKvOFull], DV * BR * 2 + BR * 4);
#pragma unroll
      for (int c = 0; c < DV / 64; ++c)
        tma_load_4d(smem + C::odO + c * BR * 128, &tm_do, &bars[kKvOFull], c * 64, bnsd ? row : n1,
                    bnsd ? n1 : row, bcoord);
    }
  }
  __syncwarp();
  if (warp == 9) tmem_alloc(tm_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tm_holder;
  // The set-up above (barriers, tensor memory, tensor-map prefetch) overlaps the tail of the
  // preceding preprocess kernel under programmatic dependent launch; nothing it wrote is read
  // before this point.
  griddep_wait();
  if (a.inject_timeout) {
    if (lane == 0) wait_bar(&bars[kKvNever], 0, abort_flag, a);
    __syncwarp();
  }
  __syncthreads();

  constexpr bool kBF16 = !FP16;

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && T > 0 && !*abort_flag) {
      for (int t = 0; t < T; ++t) {  // step 0's tiles were issued during the set-up (above)
        const int sq_ = t % NQ, so = t % NO;
        const int h = t / nqb, qb = qb_begin + t % nqb;
        const int n1 = n2 * a.G + h, i0 = qb * BR;
        const int row = q_rowbase + i0;
        const long long rbase = ((long long)b * a.N1 + n1) * a.S1p + i0;
        if (t >= NQ && !wait_bar(&bars[kKvQEmpty + sq_], ((t / NQ) - 1) & 1, abort_flag, a)) break;
        uint64_t* qfull = &bars[kKvQFull + sq_];
        if (t > 0) {
          mbar_arrive_expect_tx(qfull, D * BR * 2 + BR * 4);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(smem + C::oQ + sq_ * C::kQ + c * BR * 128, &tm_q, qfull, c * 64, bnsd ? row : n1,
                        bnsd ? n1 : row, bcoord);
        }
        bulk_load(smem + C::oL + sq_ * BR * 4, a.lse2 + rbase, BR * 4, qfull);
        if (t >= NO && !wait_bar(&bars[kKvOEmpty + so], ((t / NO) - 1) & 1, abort_flag, a)) break;
        uint64_t* ofull = &bars[kKvOFull + so];
        if (t > 0) {
          mbar_arrive_expect_tx(ofull, DV * BR * 2 + BR * 4);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_4d(smem + C::odO + so * C::kdO + c * BR * 128, &tm_do, ofull, c * 64, bnsd ? row : n1,
                        bnsd ? n1 : row, bcoord);
        }
        bulk_load(smem + C::oF + so * BR * 4, a.sfmg + rbase, BR * 4, ofull);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t ID_S = idesc_f16(BC, BR, kBF16, false, false);
      constexpr uint32_t ID_DV = idesc_f16(BC, DV, kBF16, false, true);
      constexpr uint32_t ID_DK = idesc_f16(BC, D, kBF16, false, true);
      const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::oK), 16, 1024);
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::oV), 16, 1024);
      // A operand columns of k-step kk (16 queries): warpgroup kk/KPW holds queries NCW·(kk/KPW)..,
      // its 16-bit pairs at the start of its own NCW columns
      constexpr int NCW = C::NCW, KPW = NCW / 16;
      auto a_col = [](int kk) { return (kk / KPW) * NCW + (kk % KPW) * 8; };
      auto issue_s = [&](int t) {  // Q(t) landed: vouched for by the compute warps' P(t-1) handoff
        const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::oQ + (t % NQ) * C::kQ), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::cS, sdesc_at(dK0, (kk >> 2) * BC * 128 + (kk & 3) * 32),
                 sdesc_at(dQ0, (kk >> 2) * BR * 128 + (kk & 3) * 32), ID_S, kk > 0);
        mma_commit(&bars[kKvSFull]);
      };
      auto issue_dp = [&](int t) {  // dO(t) landed: vouched for by the compute warps' dS(t-1) handoff
        const uint64_t ddO0 = sdesc_sw128(smem_u32(smem + C::odO + (t % NO) * C::kdO), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          mma_ss(tmem + C::cP, sdesc_at(dV0, (kk >> 2) * BC * 128 + (kk & 3) * 32),
                 sdesc_at(ddO0, (kk >> 2) * BR * 128 + (kk & 3) * 32), ID_S, kk > 0);
        mma_commit(&bars[kKvDpFull]);
      };
      bool ok = wait_bar(&bars[kKvKvFull], 0, abort_flag, a) && wait_bar(&bars[kKvQFull], 0, abort_flag, a) &&
                wait_bar(&bars[kKvOFull], 0, abort_flag, a);
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int t = 0; ok && t < T; ++t) {
        const int sq_ = t % NQ, so = t % NO;
        const uint64_t dQt = sdesc_sw128(smem_u32(smem + C::oQ + sq_ * C::kQ), BR * 128, 1024);
        const uint64_t ddOt = sdesc_sw128(smem_u32(smem + C::odO + so * C::kdO), BR * 128, 1024);
        if (!(ok = wait_bar(&bars[kKvPFull], t & 1, abort_flag, a))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ts(tmem + C::cDV, tmem + C::cS + a_col(kk), sdesc_at(ddOt, kk * 2048), ID_DV,
                 (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kKvOEmpty + so]);  // dO(t) read; the compute warps add their sfmg arrivals
        // Sᵀ of the next step may overwrite the Pᵀ columns once dV (issued above) has read them
        if (t + 1 < T) issue_s(t + 1);
        if (!(ok = wait_bar(&bars[kKvDsFull], t & 1, abort_flag, a))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ts(tmem + C::cDK, tmem + C::cP + a_col(kk), sdesc_at(dQt, kk * 2048), ID_DK,
                 (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kKvQEmpty + sq_]);
        if (t + 1 < T) issue_dp(t + 1);  // after dK read the dSᵀ held in the dPᵀ columns
      }
      if (ok) {
        mma_commit(&bars[kKvAccDone]);
      } else {
        mma_commit(&bars[kKvDrain]);
        mbar_wait(&bars[kKvDrain], 0, kDrainNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ compute warpgroups 0, 1
    const int q4 = warp & 3, g = warp >> 2;
    const int row = q4 * 32 + lane;  // TMEM lane = key row j0 + row
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    constexpr int NCW = C::NCW;
    constexpr bool W2 = NCW == 64;  // two 32-column halves per thread (else one)
    const uint32_t sS = tmem + lane_off + C::cS + g * NCW, sP = tmem + lane_off + C::cP + g * NCW;
    const int jr = j0 + row;
    const bool j_valid = jr < sq.L2;
    const long long vlo = (long long)jr - off - hi, vhi = (long long)jr - off - lo;
    const int i_vis_lo = (int)(vlo < -1 ? -1 : (vlo > (1 << 30) ? (1 << 30) : vlo));
    const int i_vis_hi = (int)(vhi < -1 ? -1 : (vhi > (1 << 30) ? (1 << 30) : vhi));
    bool ok = true;
    if (T > 0) ok = wait_bar_warp(&bars[kKvQFull], 0, abort_flag, a) && wait_bar_warp(&bars[kKvOFull], 0, abort_flag, a);
    for (int t = 0; ok && t < T; ++t) {
      const int sq_ = t % NQ, so = t % NO;
      const int qb = qb_begin + t % nqb;
      const int i0 = qb * BR, ic0 = i0 + g * NCW;
      // lse(t) and sfmg(t) landed: observed before the previous step's handoffs (or above).  The
      // MMA thread issues Sᵀ(t+1) right after this step's P handoff: its Q stage (loaded long
      // ago) is confirmed here, while the warps would wait for Sᵀ(t) anyway.
      if (t + 1 < T && !(ok = wait_bar_warp(&bars[kKvQFull + (t + 1) % NQ], ((t + 1) / NQ) & 1, abort_flag, a))) break;
      if (!(ok = wait_bar_warp(&bars[kKvSFull], t & 1, abort_flag, a))) break;
      tc_fence_after();
      const float4* sL4 = reinterpret_cast<const float4*>(smem + C::oL + sq_ * BR * 4 + g * NCW * 4);
      const float4* sF4 = reinterpret_cast<const float4*>(smem + C::oF + so * BR * 4 + g * NCW * 4);
      const long long dmin = (long long)j0 - (i0 + BR - 1) - off, dmax = (long long)(j1 - 1) - i0 - off;
      const bool full = dmin >= lo && dmax <= hi;
      uint32_t p0[32], p1[32];  // Sᵀ row (NCW queries), then P (fp32 bits)
      tmem_ld32(sS, p0);
      if constexpr (W2) tmem_ld32(sS + 32, p1);
      tmem_wait_ld();
      reg_fence(p0);
      if constexpr (W2) reg_fence(p1);
      // P = 2^(s·scale_log2 − lse2) as 2^−(lse2 − s·scale_log2): one packed fp32x2 FMA per
      // query pair against the lse vector as stored; the sign goes with the exponential's operand.
      // RN is sign-symmetric, so the value is the one the unpacked form gives, bit for bit.
      const float2 nsc2 = make_float2(-a.scale_log2, -a.scale_log2);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 l0 = sL4[c4];
        const float la[4] = {l0.x, l0.y, l0.z, l0.w};
        float lb[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (W2) {
          const float4 l1 = sL4[c4 + 8];
          lb[0] = l1.x, lb[1] = l1.y, lb[2] = l1.z, lb[3] = l1.w;
        }
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const int c = 4 * c4 + e;
          const float2 y0 = __ffma2_rn(make_float2(__uint_as_float(p0[c]), __uint_as_float(p0[c + 1])), nsc2,
                                       make_float2(la[e], la[e + 1]));
          p0[c] = __float_as_uint(ex2(-y0.x));
          p0[c + 1] = __float_as_uint(ex2(-y0.y));
          if constexpr (W2) {
            const float2 y1 = __ffma2_rn(make_float2(__uint_as_float(p1[c]), __uint_as_float(p1[c + 1])), nsc2,
                                         make_float2(lb[e], lb[e + 1]));
            p1[c] = __float_as_uint(ex2(-y1.x));
            p1[c + 1] = __float_as_uint(ex2(-y1.y));
          }
        }
      }
      if (!full) {
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (ic0 + c < i_vis_lo || ic0 + c > i_vis_hi) p0[c] = 0u;
          if constexpr (W2)
            if (ic0 + 32 + c < i_vis_lo || ic0 + 32 + c > i_vis_hi) p1[c] = 0u;
        }
      }
      if (!j_valid) {
#pragma unroll
        for (int c = 0; c < 32; ++c) p0[c] = p1[c] = 0u;
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          pk[c] = pack2<FP16>(__uint_as_float(p0[2 * c]), __uint_as_float(p0[2 * c + 1]));
          if constexpr (W2) pk[16 + c] = pack2<FP16>(__uint_as_float(p1[2 * c]), __uint_as_float(p1[2 * c + 1]));
        }
        // Pᵀ over this warpgroup's own (already read) Sᵀ columns
        if constexpr (W2) tmem_st32(sS, pk);
        else tmem_st16(sS, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kKvPFull]);
      // and dPᵀ(t+1) right after the dS handoff: its dO stage must have landed
      if (t + 1 < T && !(ok = wait_bar_warp(&bars[kKvOFull + (t + 1) % NO], ((t + 1) / NO) & 1, abort_flag, a))) break;
      if (!(ok = wait_bar_warp(&bars[kKvDpFull], t & 1, abort_flag, a))) break;
      tc_fence_after();
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(sP, r0);
        if constexpr (W2) tmem_ld32(sP + 32, r1);
        tmem_wait_ld();
        reg_fence(r0);
        if constexpr (W2) reg_fence(r1);
        // −dS = P ⊙ (sfmg − dP), packed: (sfmg − dP) as one fp32x2 FMA with −1 (exactly the
        // negated difference), then a packed multiply.  dK accumulates −dS·Q and its epilogue
        // scales by −scale.
        const float2 m1 = make_float2(-1.f, -1.f);
        uint32_t dk[32];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 f0 = sF4[c4];
          const float fa[4] = {f0.x, f0.y, f0.z, f0.w};
          float fb[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (W2) {
            const float4 f1 = sF4[c4 + 8];
            fb[0] = f1.x, fb[1] = f1.y, fb[2] = f1.z, fb[3] = f1.w;
          }
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int c = 4 * c4 + e;
            const float2 n0 = __fmul2_rn(make_float2(__uint_as_float(p0[c]), __uint_as_float(p0[c + 1])),
                                         __ffma2_rn(make_float2(__uint_as_float(r0[c]), __uint_as_float(r0[c + 1])), m1,
                                                    make_float2(fa[e], fa[e + 1])));
            dk[c >> 1] = pack2<FP16>(n0.x, n0.y);
            if constexpr (W2) {
              const float2 n1 = __fmul2_rn(make_float2(__uint_as_float(p1[c]), __uint_as_float(p1[c + 1])),
                                           __ffma2_rn(make_float2(__uint_as_float(r1[c]), __uint_as_float(r1[c + 1])),
                                                      m1, make_float2(fb[e], fb[e + 1])));
              dk[16 + (c >> 1)] = pack2<FP16>(n1.x, n1.y);
            }
          }
        }
        // −dSᵀ over this warpgroup's own (already read) dPᵀ columns
        if constexpr (W2) tmem_st32(sP, dk);
        else tmem_st16(sP, *reinterpret_cast<uint32_t(*)[16]>(&dk[0]));
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kKvDsFull]);
        mbar_arrive(&bars[kKvOEmpty + so]);  // this warp's sfmg reads of stage so are done
      }
    }
    // ---- epilogue: dK = scale · acc, dV = acc; zeros when no query sees this block
    // A block whose 128 rows lie inside its sequence is staged in shared memory (the drained
    // Q/dO rings) as 128-byte-swizzled 64-column tiles and written by TMA stores, one per tile;
    // the last block of a TND sequence, whose box would reach into the next sequence's rows,
    // is written row by row.  A thread's 16-byte stores to rows 2 KB or more apart would
    // otherwise take one request each.  dV is final once the last dV product has completed
    // (the commit on its dO stage, which also frees the dO ring): its tiles are staged in the dO
    // ring and stored while the last dK product still runs; dK follows through the Q ring.
    const bool staged = !tnd || j0 + BC <= sq.span_k;  // the same in every thread of the CTA
    if (staged) {
      auto put = [&](uint8_t* stage, int tile, int unit0, const uint32_t (&o)[16]) {
        uint8_t* rowp = stage + tile * BC * 128 + row * 128;
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          st_shared_v4(smem_u32(rowp + (((unit0 + v4) ^ (row & 7)) << 4)), o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2],
                       o[4 * v4 + 3]);
      };
      if (ok && T > 0) ok = wait_bar_warp(&bars[kKvOEmpty + (T - 1) % NO], ((T - 1) / NO) & 1, abort_flag, a);
      tc_fence_after();
      uint8_t* vstage = smem + C::odO;  // Dv/64 dV tiles, BC·128 bytes each
#pragma unroll 1
      for (int c = 0; ok && c < DV / 64; ++c) {
        const int col = g * (DV / 2) + c * 32;
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::cDV + col, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          o[e >> 1] = T > 0 ? pack2<FP16>(__uint_as_float(r[e]), __uint_as_float(r[e + 1])) : 0u;
        put(vstage, col / 64, (col % 64) / 8, o);
      }
      fence_proxy_async_smem();
      // every compute thread reaches these barriers (staged is CTA-uniform); tiles are stored
      // only if every warp wrote its part
      const bool v_ok = compute_warps_all(ok);
      if (v_ok && warp == 0 && lane == 0) {
#pragma unroll 1
        for (int c = 0; c < DV / 64; ++c)
          tma_store_4d(&tm_dv, vstage + c * BC * 128, c * 64, bnsd ? kv_row0 : n2, bnsd ? n2 : kv_row0, bcoord);
        bulk_commit_group();
      }
      if (ok && T > 0) ok = wait_bar_warp(&bars[kKvAccDone], 0, abort_flag, a);
      tc_fence_after();
      uint8_t* kstage = smem + C::oQ;  // D/64 dK tiles
#pragma unroll 1
      for (int c = 0; ok && c < D / 64; ++c) {
        const int col = g * (D / 2) + c * 32;
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::cDK + col, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          o[e >> 1] = T > 0 ? pack2<FP16>(__uint_as_float(r[e]) * -a.scale, __uint_as_float(r[e + 1]) * -a.scale) : 0u;
        put(kstage, col / 64, (col % 64) / 8, o);
      }
      fence_proxy_async_smem();
      const bool k_ok = compute_warps_all(ok);
      if (k_ok && warp == 0 && lane == 0) {
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c)
          tma_store_4d(&tm_dk, kstage + c * BC * 128, c * 64, bnsd ? kv_row0 : n2, bnsd ? n2 : kv_row0, bcoord);
        bulk_commit_group();
      }
    } else if (ok && (T == 0 || (ok = wait_bar_warp(&bars[kKvAccDone], 0, abort_flag, a)))) {
      tc_fence_after();
      const long long krow = row_index(a.layout, b, (long long)(tnd ? sq.k0 : 0) + (j_valid ? jr : 0), n2, a.N2, a.S2);
      uint16_t* dk = static_cast<uint16_t*>(a.dk) + krow * a.io_d;
      uint16_t* dv = static_cast<uint16_t*>(a.dv) + krow * a.io_dv;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        const int col = g * (D / 2) + c * 32;
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::cDK + col, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          o[e >> 1] = T > 0 ? pack2<FP16>(__uint_as_float(r[e]) * -a.scale, __uint_as_float(r[e + 1]) * -a.scale) : 0u;
        if (j_valid) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            if (col + v4 * 8 < a.io_d)
              *reinterpret_cast<uint4*>(dk + col + v4 * 8) = make_uint4(o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2], o[4 * v4 + 3]);
        }
      }
#pragma unroll 1
      for (int c = 0; c < DV / 64; ++c) {
        const int col = g * (DV / 2) + c * 32;
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::cDV + col, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          o[e >> 1] = T > 0 ? pack2<FP16>(__uint_as_float(r[e]), __uint_as_float(r[e + 1])) : 0u;
        if (j_valid) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            if (col + v4 * 8 < a.io_dv)
              *reinterpret_cast<uint4*>(dv + col + v4 * 8) = make_uint4(o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2], o[4 * v4 + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < kGraceNs) {
    }
  }
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // the TMA stores issued in the epilogue read their tiles before the CTA's shared memory is
  // released; that drain overlaps the tensor-memory release above
  if (warp == 0 && lane == 0) bulk_wait_group_read0();
}

template <int D, int DV, bool FP16, bool FLAT>
__global__ void __launch_bounds__(kMainThreads, 1)
    fabwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const MainArgs a) {
  if constexpr (FLAT) {  // varlen: the sequences' own key blocks back to back
    int b, local, nqb;
    bool kv;
    if (!flat_unit(a, blockIdx.x, KvCfg<D, DV>::BC, 0, b, local, kv, nqb)) return;
    kv_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv, a, local, b);
  } else {
    kv_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv, a, blockIdx.x, blockIdx.y);
  }
}

template <int D, int DV, bool FP16, bool FLAT>
cudaError_t launch_kv_flat(const MainArgs& a, const MainMaps& m, dim3 grid, cudaStream_t st) {
  using C = KvCfg<D, DV>;
  if (cudaError_t e = ensure_smem_limit<fabwd_kv_kernel<D, DV, FP16, FLAT>>((int)C::bytes); e != cudaSuccess)
    return e;
  fabwd_kv_kernel<D, DV, FP16, FLAT><<<grid, kMainThreads, C::bytes, st>>>(m.q, m.k, m.v, m.dout, m.dk, m.dv, a);
  return cudaGetLastError();
}

template <int D, int DV, bool FP16>
cudaError_t launch_kv_t(const MainArgs& a, const MainMaps& m, int n_kv_blocks, cudaStream_t st) {
  using C = KvCfg<D, DV>;
  if (flat_grid(a.layout, a.B))
    return launch_kv_flat<D, DV, FP16, true>(
        a, m, dim3((unsigned)(tnd_blocks_bound(a.B, a.S2, a.T2, C::BC) * a.N2), 1), st);
  return launch_kv_flat<D, DV, FP16, false>(a, m, dim3(n_kv_blocks * a.N2, a.B), st);
}

}  // namespace fabwd
