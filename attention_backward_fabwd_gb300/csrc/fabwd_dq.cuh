// q-stationary dQ kernel for sm_103a (the deterministic dQ mode).
//
// What it computes is dQ of the page "CANN ops-transformer FlashAttnGrad 算子详解"
// (discosf.com/news/4863418), §一: dQ = scale · dS · K with dS = P ⊙ (dP − sfmg),
// P = exp(scale·QKᵀ − lse), dP = dY·Vᵀ.  One CTA owns 128 query rows of one q-head and loops
// over the key blocks that row block can see:
//     S  = Q·Kᵀ       tcgen05 (M = 128 queries, N = BN keys, K = D), double-buffered in TMEM
//     dP = dO·Vᵀ      tcgen05 (K = Dv)
//     dS = exp2(S·scale·log2e − lse·log2e) ⊙ (dP − sfmg), masked pairs -> 0, bf16/fp16 in TMEM
//     dQ += dS·K      tcgen05, A operand read from TMEM, accumulated in TMEM over all key blocks
// and writes dq = scale · dQ in the io dtype once.  Every dQ element is summed by one CTA in a
// fixed order: no atomics, no fp32 workspace, bitwise reproducible.  dK and dV come from the
// kv-stationary kernel run without its dQ product.  The lane of every TMEM accumulator is the
// query row, so the per-row lse and sfmg are per-thread scalars.
//
// Warp roles (320 threads): warps 0-7 compute (warp w reads TMEM lanes 32·(w%4)..+31; warps 0-3
// take key columns [0, BN/2), warps 4-7 [BN/2, BN)), warp 8 issues TMA loads (Q, dO once; K
// through a 3-stage ring released after dQ, V through a ring of NV stages released after dP), warp 9
// allocates TMEM and issues the MMAs.  BN = 128 keys and NV = 2 up to D = 128; at D = 192, BN = 96
// and NV = 1 at Dv = 128 (a second V stage does not fit beside Q, dO and three 36 KB K stages).
// One thread issues every tcgen05.mma, and an MMA of these
// shapes occupies it about as long as the tensor pipe takes to run it, so each barrier wait
// between MMA groups idles the pipe.  The MMA thread therefore issues
//     [dS(t) written] dP(t+1), dQ(t), [K(t+2) landed] S(t+2)
// (S is double-buffered, so S(t+2) reuses the buffer whose dS dQ(t) has just read), and the
// compute warps, not the MMA thread, wait for V(t+1) before they signal dS(t): that wait falls
// while the warps wait for dP anyway.  K(t+2) stays with the MMA thread: its stage is freed by
// dQ(t-1), too late for the compute warps to vouch for it by dS(t).  With one V stage, V(t+1)
// can load only once dP(t) has read V(t), so the order is [dS(t)] dQ(t), [V(t+1)] dP(t+1),
// [K(t+2)] S(t+2): the load overlaps dQ(t) and the MMA thread, not the compute warps, waits for
// it (a phase trace had the compute warps waiting ~1000 clk per step for V(t+1) before dS(t)).
// TMEM columns: dQ [0, D), S buffer 0 [D, D+BN), S buffer 1 [D+BN, D+2BN), dP [D+2BN, D+3BN).
// Every mbarrier wait is bounded as in the kv-stationary kernel.
#pragma once

#include "fabwd_internal.cuh"
#include "fabwd_main.cuh"
#include "fabwd_ptx.cuh"
#include "../../include/fabwd.h"

namespace fabwd {

template <int D, int DV>
struct DqCfg {
  static constexpr int BM = 128;                 // query rows per CTA (TMEM lanes)
  static constexpr int BN = dq_block_kv(D, DV);  // keys per step
  static constexpr int NK = 3;                   // K ring stages
  static constexpr uint32_t kQ = D * BM * 2, kdO = DV * BM * 2, kK = D * BN * 2, kV = DV * BN * 2;
  // V ring stages: two where they fit beside Q, dO and the K ring (one at D = 192, Dv = 128)
  static constexpr int NV = kQ + kdO + NK * kK + 2 * kV + 20 * 8 + 64 <= 232448 ? 2 : 1;
  static constexpr int NC = BN / 2;              // key columns per compute thread
  static_assert(NC % 16 == 0, "dS k-steps of 16 keys stay within one warpgroup's columns");
  static constexpr uint32_t oQ = 0, odO = oQ + kQ, oK = odO + kdO, oV = oK + NK * kK;
  static constexpr uint32_t oBar = oV + NV * kV;
  static constexpr uint32_t oMisc = oBar + 20 * 8;
  static constexpr uint32_t bytes = oMisc + 64;
  static constexpr uint32_t cDQ = 0, cS0 = D, cP = D + 2 * BN;  // S buffer b at cS0 + b·BN
  static_assert(cP + BN <= 512, "TMEM budget");
  static_assert(D / 64 * BM * 128 <= NK * kK, "dQ staging fits in the K ring");
  static_assert(bytes <= 232448, "shared memory budget");
};

constexpr int kDqQdoFull = 0, kDqKFull = 1 /*+3*/, kDqKEmpty = 4 /*+3*/, kDqVFull = 7 /*+2*/, kDqVEmpty = 9 /*+2*/,
              kDqSFull = 11 /*+2*/, kDqDpFull = 13, kDqDsFull = 14, kDqAccDone = 15, kDqNever = 16, kDqDrain = 17,
              kDqNumBars = 18;

// One CTA of the dQ kernel: query block nqb - 1 - bx / N1 (latest first) of q-head bx % N1,
// batch by; nqb counts the BM-row query blocks of the batch row (or sequence) that bx runs over.
template <int D, int DV, bool FP16>
__device__ __forceinline__ void dq_block(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                         const CUtensorMap& tm_do, const CUtensorMap& tm_dq, const MainArgs& a, int bx,
                                         int by, int nqb) {
  using C = DqCfg<D, DV>;
  constexpr int BM = C::BM, BN = C::BN, NK = C::NK, NV = C::NV, NC = C::NC;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = by;
  SeqRange sq;
  if (!seq_range(a, b, sq)) return;  // bad cu_seqlens: the preprocess kernel reports it
  const int qb = nqb - 1 - bx / a.N1, n1 = bx % a.N1;  // latest query blocks first
  const int i0 = qb * BM;
  if (qb < 0 || i0 >= sq.L1) return;
  if ((smem_u32(smem) & 1023u) != 0) {
    griddep_wait();  // the preprocess clears the status word
    if (tid == 0) atomicOr(a.status, FABWD_DEV_INTERNAL);
    return;
  }
  const int n2 = n1 / a.G;
  const int i1 = min(i0 + BM, sq.L1);
  const long long off = (long long)sq.L2 - sq.L1;
  long long lo, hi;
  mask_bounds(a, lo, hi);
  // keys seen by at least one row of [i0, i1)
  long long jb_ = (long long)i0 + off + lo, je_ = (long long)(i1 - 1) + off + hi;
  if (jb_ < 0) jb_ = 0;
  if (je_ > sq.L2 - 1) je_ = sq.L2 - 1;
  const int kb_begin = jb_ <= je_ ? (int)(jb_ / BN) : 0;
  const int T = jb_ <= je_ ? (int)(je_ / BN) + 1 - kb_begin : 0;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::oBar);
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + C::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oMisc + 16);
  const bool tnd = a.layout == kTND, bnsd = a.layout == kBNSD;
  const int q_row = (tnd ? sq.q0 : 0) + i0;
  const int kv_rowbase = tnd ? sq.k0 : 0;
  const int bcoord = tnd ? 0 : b;
  // key-block steps whose K and V tiles load during the set-up (the first NV: no stage to wait for)
  const int early = T < NV ? T : NV;
  auto load_k = [&](int t) {
    const int sk = t % NK;
    const int row = kv_rowbase + (kb_begin + t) * BN;
    uint64_t* kfull = &bars[kDqKFull + sk];
    mbar_arrive_expect_tx(kfull, D * BN * 2);
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      tma_load_4d(smem + C::oK + sk * C::kK + c * BN * 128, &tm_k, kfull, c * 64, bnsd ? row : n2, bnsd ? n2 : row,
                  bcoord);
  };
  auto load_v = [&](int t) {
    const int sv = t % NV;
    const int row = kv_rowbase + (kb_begin + t) * BN;
    uint64_t* vfull = &bars[kDqVFull + sv];
    mbar_arrive_expect_tx(vfull, DV * BN * 2);
#pragma unroll
    for (int c = 0; c < DV / 64; ++c)
      tma_load_4d(smem + C::oV + sv * C::kV + c * BN * 128, &tm_v, vfull, c * 64, bnsd ? row : n2, bnsd ? n2 : row,
                  bcoord);
  };
  if (warp == 8 && lane == 0) {
    for (int i = 0; i < kDqNumBars; ++i) mbar_init(&bars[i], i == kDqDsFull ? 8 : 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
    if (T > 0) {
      // Q, dO and the first K, V tiles are inputs (the preprocess writes none of them): they load
      // while the CTA allocates TMEM and waits for the preprocess
      mbar_arrive_expect_tx(&bars[kDqQdoFull], (D + DV) * BM * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_4d(smem + C::oQ + c * BM * 128, &tm_q, &bars[kDqQdoFull], c * 64, bnsd ? q_row : n1,
                    bnsd ? n1 : q_row, bcoord);
#pragma unroll
      for (int c = 0; c < DV / 64; ++c)
        tma_load_4d(smem + C::odO + c * BM * 128, &tm_do, &bars[kDqQdoFull], c * 64, bnsd ? q_row : n1,
                    bnsd ? n1 : q_row, bcoord);
      for (int t = 0; t < early; ++t) {
        load_k(t);
        load_v(t);
      }
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
    if (lane == 0) wait_bar(&bars[kDqNever], 0, abort_flag, a);
    __syncwarp();
  }
  __syncthreads();

  constexpr bool kBF16 = !FP16;

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && T > 0 && !*abort_flag) {
      for (int t = early; t < T; ++t) {  // the first `early` steps' tiles were issued above
        const int sk = t % NK, sv = t % NV;
        if (t >= NK && !wait_bar(&bars[kDqKEmpty + sk], ((t / NK) - 1) & 1, abort_flag, a)) break;
        load_k(t);
        if (t >= NV && !wait_bar(&bars[kDqVEmpty + sv], ((t / NV) - 1) & 1, abort_flag, a)) break;
        load_v(t);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t ID_S = idesc_f16(BM, BN, kBF16, false, false);
      constexpr uint32_t ID_DQ = idesc_f16(BM, D, kBF16, false, true);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::oQ), 16, 1024);
      const uint64_t ddO0 = sdesc_sw128(smem_u32(smem + C::odO), 16, 1024);
      auto issue_s = [&](int t) {  // K(t) landed (see above)
        const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::oK + (t % NK) * C::kK), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::cS0 + (t & 1) * BN, sdesc_at(dQ0, (kk >> 2) * BM * 128 + (kk & 3) * 32),
                 sdesc_at(dK0, (kk >> 2) * BN * 128 + (kk & 3) * 32), ID_S, kk > 0);
        mma_commit(&bars[kDqSFull + (t & 1)]);
      };
      auto issue_dp = [&](int t) {  // V(t) landed (see above)
        const int sv = t % NV;
        const uint64_t dV0 = sdesc_sw128(smem_u32(smem + C::oV + sv * C::kV), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          mma_ss(tmem + C::cP, sdesc_at(ddO0, (kk >> 2) * BM * 128 + (kk & 3) * 32),
                 sdesc_at(dV0, (kk >> 2) * BN * 128 + (kk & 3) * 32), ID_S, kk > 0);
        mma_commit(&bars[kDqDpFull]);
        mma_commit(&bars[kDqVEmpty + sv]);
      };
      bool ok = wait_bar(&bars[kDqQdoFull], 0, abort_flag, a) && wait_bar(&bars[kDqKFull], 0, abort_flag, a) &&
                wait_bar(&bars[kDqVFull], 0, abort_flag, a) && (T < 2 || wait_bar(&bars[kDqKFull + 1], 0, abort_flag, a));
      // from here on V(t+1) is vouched for by the compute warps' dS(t) arrival
      if (ok) {
        tc_fence_after();
        issue_s(0);
        issue_dp(0);
        if (T > 1) issue_s(1);
      }
      for (int t = 0; ok && t < T; ++t) {
        // dS(t) written, dP(t) read by every compute warp (and, with two V stages, V(t+1) landed)
        if (!(ok = wait_bar(&bars[kDqDsFull], t & 1, abort_flag, a))) break;
        tc_fence_after();
        if (NV > 1 && t + 1 < T) issue_dp(t + 1);
        const uint64_t dKt = sdesc_sw128(smem_u32(smem + C::oK + (t % NK) * C::kK), BN * 128, 1024);
        const uint32_t sb = tmem + C::cS0 + (t & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)  // dS of warpgroup kk/(NC/16) sits in its own S columns
          mma_ts(tmem + C::cDQ, sb + (kk / (NC / 16)) * NC + (kk % (NC / 16)) * 8,
                 sdesc_at(dKt, kk * 2048), ID_DQ, (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kDqKEmpty + (t % NK)]);
        if (NV == 1 && t + 1 < T) {  // one V stage: V(t+1) has loaded while dQ(t) runs
          if (!(ok = wait_bar(&bars[kDqVFull], (t + 1) & 1, abort_flag, a))) break;
          tc_fence_after();
          issue_dp(t + 1);
        }
        if (t + 2 < T) {  // into the S buffer whose dS the dQ product above has read
          if (!(ok = wait_bar(&bars[kDqKFull + (t + 2) % NK], ((t + 2) / NK) & 1, abort_flag, a))) break;
          tc_fence_after();
          issue_s(t + 2);
        }
      }
      if (ok) {
        mma_commit(&bars[kDqAccDone]);
      } else {
        mma_commit(&bars[kDqDrain]);
        mbar_wait(&bars[kDqDrain], 0, kDrainNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ compute warpgroups 0, 1
    const int q4 = warp & 3, g = warp >> 2;
    const int row = q4 * 32 + lane;  // TMEM lane = query row i0 + row
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int ir = i0 + row;
    const float* lse2_row = a.lse2 + ((long long)b * a.N1 + n1) * a.S1p;
    const float* sfmg_row = a.sfmg + ((long long)b * a.N1 + n1) * a.S1p;
    const float lse2 = lse2_row[ir];  // +inf beyond the sequence: P = 0 there
    const float sf = sfmg_row[ir];
    const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nl2 = make_float2(-lse2, -lse2);
    const float2 nsf2 = make_float2(-sf, -sf);
    // keys visible to this row: j - ir - off in [lo, hi]
    const long long vlo = (long long)ir + off + lo, vhi = (long long)ir + off + hi;
    const int j_vis_lo = (int)(vlo < -1 ? -1 : (vlo > (1 << 30) ? (1 << 30) : vlo));
    const int j_vis_hi = (int)min((long long)sq.L2 - 1, vhi < -1 ? -1ll : (vhi > (1 << 30) ? (long long)(1 << 30) : vhi));
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int j0 = (kb_begin + t) * BN;
      const uint32_t sb = tmem + lane_off + C::cS0 + (t & 1) * BN + g * NC;
      const long long dmin = (long long)j0 - (i0 + BM - 1) - off, dmax = (long long)(j0 + BN - 1) - i0 - off;
      const bool full = j0 + BN <= sq.L2 && dmin >= lo && dmax <= hi;
      if (!(ok = wait_bar_warp(&bars[kDqSFull + (t & 1)], (t >> 1) & 1, abort_flag, a))) break;
      tc_fence_after();
      uint32_t p[NC];
      tmem_ld32(sb, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
      if constexpr (NC == 64) tmem_ld32(sb + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
      if constexpr (NC == 48) tmem_ld16(sb + 32, *reinterpret_cast<uint32_t(*)[16]>(&p[32]));
      tmem_wait_ld();
      reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&p[0]));
      if constexpr (NC == 64) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&p[32]));
      if constexpr (NC == 48) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(&p[32]));
      // P = 2^(s·scale_log2 − lse2): one packed fp32x2 FMA per key pair (lse2 is this row's)
#pragma unroll
      for (int c = 0; c < NC; c += 2) {
        const float2 y = __ffma2_rn(make_float2(__uint_as_float(p[c]), __uint_as_float(p[c + 1])), sc2, nl2);
        p[c] = __float_as_uint(ex2(y.x));
        p[c + 1] = __float_as_uint(ex2(y.y));
      }
      if (!full) {
        const int jc = j0 + g * NC;
#pragma unroll
        for (int c = 0; c < NC; ++c)
          if (jc + c < j_vis_lo || jc + c > j_vis_hi) p[c] = 0u;
      }
      // with two V stages the MMA thread issues dP(t+1) right after the dS(t) handoff below: its V
      // stage must have landed
      if (NV > 1 && t + 1 < T && !(ok = wait_bar_warp(&bars[kDqVFull + (t + 1) % NV], ((t + 1) / NV) & 1, abort_flag, a)))
        break;
      if (!(ok = wait_bar_warp(&bars[kDqDpFull], t & 1, abort_flag, a))) break;
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < NC / 32; ++hh) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::cP + g * NC + hh * 32, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t ds[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {  // dS = P ⊙ (dP − sfmg), packed
          const float2 d = __fmul2_rn(make_float2(__uint_as_float(p[hh * 32 + c]), __uint_as_float(p[hh * 32 + c + 1])),
                                      __fadd2_rn(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), nsf2));
          ds[c >> 1] = pack2<FP16>(d.x, d.y);
        }
        tmem_st16(sb + hh * 16, ds);  // dS over this warpgroup's own (already read) S columns
      }
      if constexpr (NC % 32 == 16) {  // the last 16 key columns
        constexpr int c0 = NC - 16;
        uint32_t r[16];
        tmem_ld16(tmem + lane_off + C::cP + g * NC + c0, r);
        tmem_wait_ld();
        reg_fence16(r);
        uint32_t ds[8];
#pragma unroll
        for (int c = 0; c < 16; c += 2) {
          const float2 d = __fmul2_rn(make_float2(__uint_as_float(p[c0 + c]), __uint_as_float(p[c0 + c + 1])),
                                      __fadd2_rn(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), nsf2));
          ds[c >> 1] = pack2<FP16>(d.x, d.y);
        }
        tmem_st8(sb + c0 / 2, ds);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kDqDsFull]);
    }
    // ---- epilogue: dq = scale · dQ (zeros when the row block sees no key)
    if (ok && T > 0) ok = wait_bar_warp(&bars[kDqAccDone], 0, abort_flag, a);
    // As in the dK/dV CTAs: a block whose 128 rows lie inside its sequence is staged in the
    // drained K ring as 128-byte-swizzled 64-column tiles and written by TMA stores; the last
    // block of a TND sequence is written row by row.
    const bool staged = !tnd || i0 + BM <= sq.span_q;  // the same in every thread of the CTA
    if (staged) {
      tc_fence_after();
      uint8_t* stage = smem + C::oK;  // D/64 tiles of BM·128 bytes
#pragma unroll 1
      for (int c = 0; ok && c < D / 64; ++c) {
        const int col = g * (D / 2) + c * 32;
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::cDQ + col, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          o[e >> 1] = T > 0 ? pack2<FP16>(__uint_as_float(r[e]) * a.scale, __uint_as_float(r[e + 1]) * a.scale) : 0u;
        uint8_t* rowp = stage + (col / 64) * BM * 128 + row * 128;
        const int unit0 = (col % 64) / 8;
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          st_shared_v4(smem_u32(rowp + (((unit0 + v4) ^ (row & 7)) << 4)), o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2],
                       o[4 * v4 + 3]);
      }
      fence_proxy_async_smem();
      // every compute thread reaches this barrier; the tiles are stored only if every warp wrote
      // its part
      const bool all_ok = compute_warps_all(ok);
      if (all_ok && warp == 0 && lane == 0) {
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c)
          tma_store_4d(&tm_dq, stage + c * BM * 128, c * 64, bnsd ? q_row : n1, bnsd ? n1 : q_row, bcoord);
        bulk_commit_group();
      }
    } else if (ok) {
      tc_fence_after();
      const bool i_valid = ir < sq.L1;
      const long long qrow = row_index(a.layout, b, (long long)(tnd ? sq.q0 : 0) + (i_valid ? ir : 0), n1, a.N1, a.S1);
      uint16_t* dq = static_cast<uint16_t*>(a.dq) + qrow * a.io_d;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        const int col = g * (D / 2) + c * 32;
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + C::cDQ + col, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          o[e >> 1] = T > 0 ? pack2<FP16>(__uint_as_float(r[e]) * a.scale, __uint_as_float(r[e + 1]) * a.scale) : 0u;
        if (i_valid) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            if (col + v4 * 8 < a.io_d)
              *reinterpret_cast<uint4*>(dq + col + v4 * 8) = make_uint4(o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2], o[4 * v4 + 3]);
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
    fabwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const MainArgs a) {
  using C = DqCfg<D, DV>;
  if constexpr (FLAT) {  // varlen: the sequences' own query blocks back to back
    int b, local, nqb;
    bool kv;
    if (!flat_unit(a, blockIdx.x, 0, C::BM, b, local, kv, nqb)) return;
    dq_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_do, tm_dq, a, local, b, nqb);
  } else {
    dq_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_do, tm_dq, a, blockIdx.x, blockIdx.y, (a.S1 + C::BM - 1) / C::BM);
  }
}

template <int D, int DV, bool FP16, bool FLAT>
cudaError_t launch_dq_flat(const MainArgs& a, const MainMaps& m, dim3 grid, cudaStream_t st) {
  using C = DqCfg<D, DV>;
  if (cudaError_t e = ensure_smem_limit<fabwd_dq_kernel<D, DV, FP16, FLAT>>((int)C::bytes); e != cudaSuccess)
    return e;
  fabwd_dq_kernel<D, DV, FP16, FLAT><<<grid, kMainThreads, C::bytes, st>>>(m.q, m.k, m.v, m.dout, m.dq, a);
  return cudaGetLastError();
}

template <int D, int DV, bool FP16>
cudaError_t launch_dq_t(const MainArgs& a, const MainMaps& m, cudaStream_t st) {
  using C = DqCfg<D, DV>;
  if (flat_grid(a.layout, a.B))
    return launch_dq_flat<D, DV, FP16, true>(
        a, m, dim3((unsigned)(tnd_blocks_bound(a.B, a.S1, a.T1, C::BM) * a.N1), 1), st);
  return launch_dq_flat<D, DV, FP16, false>(a, m, dim3(((a.S1 + C::BM - 1) / C::BM) * a.N1, a.B), st);
}

}  // namespace fabwd
