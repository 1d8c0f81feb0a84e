// q-stationary forward kernel for sm_103a: the attn_out and softmax_lse that the backward takes.
//
// What it computes is the forward of the page "CANN ops-transformer FlashAttnGrad 算子详解"
// (discosf.com/news/4863418), §一: S = scale·QKᵀ, lse_i = ln Σ_j exp(S_ij) over the visible keys,
// P = exp(S − lse), Y = P·V; a row with no visible key gets Y = 0 and lse = +inf.  One CTA owns
// 128 query rows of one q-head and loops over the key blocks those rows can see:
//     S = Q·Kᵀ        tcgen05 (M = 128 queries, N = BN keys, K = D), double-buffered in TMEM
//     P = exp2(S·scale·log2e − m) with a running row maximum m, written back over S as 16-bit pairs
//     O_g += P_g·V_g  tcgen05 with the A operand read from TMEM
// Warpgroup g (warps 4g..4g+3, lane = query row) takes key columns [g·BN/2, (g+1)·BN/2) of every
// block and keeps its own online softmax (m_g, l_g) and its own accumulator O_g in TMEM; the two
// halves are combined once at the end: m = max(m_0, m_1), O = Σ_g O_g·2^(m_g − m), l likewise.
// The running maximum is updated lazily: O_g and l_g are rescaled only when a block's row
// maximum exceeds the reference by more than 8 (in log2 units), so P stays below 2^8 and most
// blocks need no pass over O_g.  After the first block, P is formed against the current
// reference in the same pass that finds the block's row maximum (packed fp32x2 FMA and adds),
// and formed again only when the reference moves.  The MMA warp shares its scheduler with two
// compute warps, so fewer compute instructions leave it more issue slots.
// Warp 8 issues TMA loads (Q once; K and V through 3-stage rings, a K stage released after its S
// product, a V stage after its O product); warp 9 allocates TMEM and issues the MMAs
//     S(0), S(1), [P(t) written] O(t), S(t+2), ...
// The compute warps confirm V(t) before they hand over P(t); the MMA thread waits for K itself.
// TMEM columns: S buffer 0 [0, BN), S buffer 1 [BN, 2BN), O_0 [2BN, 2BN+Dv), O_1 [2BN+Dv, 2BN+2Dv).
// Bounded waits, abort flag, drain and TMEM release as in the backward kernels.
#pragma once
#include <type_traits>

#include "fabwd_internal.cuh"
#include "fabwd_main.cuh"
#include "fabwd_ptx.cuh"
#include "../../include/fabwd.h"

namespace fabwd {

template <int D, int DV>
struct FwdCfg {
  static constexpr int BM = 128;                 // query rows per CTA (TMEM lanes)
  static constexpr int BN = D > 128 ? 64 : 128;  // keys per step
  static constexpr int NK = 3, NV = 3;           // K ring and V ring stages
  static constexpr int NC = BN / 2;              // key columns per compute thread
  static constexpr uint32_t kQ = D * BM * 2, kK = D * BN * 2, kV = DV * BN * 2;
  static constexpr uint32_t oQ = 0, oK = oQ + kQ, oV = oK + NK * kK;
  static constexpr uint32_t oStat = oV + NV * kV;  // [2 halves][m, l][BM] fp32
  static constexpr uint32_t oBar = oStat + 2 * 2 * BM * 4;
  static constexpr uint32_t oMisc = oBar + 20 * 8;
  static constexpr uint32_t bytes = oMisc + 64;
  static constexpr uint32_t cS0 = 0, cO = 2 * BN;  // O_g at cO + g·DV
  static_assert(cO + 2 * DV <= 512, "TMEM budget");
  static_assert(bytes <= 232448, "shared memory budget");
  static_assert(NC % 16 == 0 && DV % 64 == 0, "tile shapes");
  static_assert(DV / 64 * BM * 128 <= NK * kK, "attn_out staging fits in the K ring");
};

constexpr int kFwQFull = 0, kFwKFull = 1 /*+3*/, kFwKEmpty = 4 /*+3*/, kFwVFull = 7 /*+3*/, kFwVEmpty = 10 /*+3*/,
              kFwSFull = 13 /*+2*/, kFwPFull = 15, kFwOFull = 16, kFwNever = 17, kFwDrain = 18, kFwNumBars = 19;

// One CTA of the forward: query block nqb - 1 - bx / N1 (latest first) of q-head bx % N1, batch (or
// sequence) by; nqb counts the BM-row query blocks of the batch row (or sequence) that bx runs over.
template <int D, int DV, bool FP16>
__device__ __forceinline__ void fwd_block(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                          const CUtensorMap& tm_y, const MainArgs& a, int bx, int by, int nqb) {
  using C = FwdCfg<D, DV>;
  constexpr int BM = C::BM, BN = C::BN, NK = C::NK, NV = C::NV, NC = C::NC;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = by;
  SeqRange sq;
  if (!seq_range(a, b, sq)) {  // bad cu_seqlens: reported, nothing touched
    if (tid == 0) atomicOr(a.status, FABWD_DEV_BAD_SEQLENS);
    return;
  }
  const int qb = nqb - 1 - bx / a.N1, n1 = bx % a.N1;  // latest query blocks first
  const int i0 = qb * BM;
  if (qb < 0 || i0 >= sq.L1) return;
  if ((smem_u32(smem) & 1023u) != 0) {
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
  auto load_k = [&](int t) {
    const int sk = t % NK, row = kv_rowbase + (kb_begin + t) * BN;
    mbar_arrive_expect_tx(&bars[kFwKFull + sk], D * BN * 2);
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      tma_load_4d(smem + C::oK + sk * C::kK + c * BN * 128, &tm_k, &bars[kFwKFull + sk], c * 64, bnsd ? row : n2,
                  bnsd ? n2 : row, bcoord);
  };
  auto load_v = [&](int t) {
    const int sv = t % NV, row = kv_rowbase + (kb_begin + t) * BN;
    mbar_arrive_expect_tx(&bars[kFwVFull + sv], DV * BN * 2);
#pragma unroll
    for (int c = 0; c < DV / 64; ++c)
      tma_load_4d(smem + C::oV + sv * C::kV + c * BN * 128, &tm_v, &bars[kFwVFull + sv], c * 64, bnsd ? row : n2,
                  bnsd ? n2 : row, bcoord);
  };
  if (warp == 8 && lane == 0) {
    for (int i = 0; i < kFwNumBars; ++i) mbar_init(&bars[i], i == kFwPFull ? 8 : 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    if (T > 0) {  // Q and the first K, V tiles load while the CTA allocates TMEM
      mbar_arrive_expect_tx(&bars[kFwQFull], D * BM * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_4d(smem + C::oQ + c * BM * 128, &tm_q, &bars[kFwQFull], c * 64, bnsd ? q_row : n1,
                    bnsd ? n1 : q_row, bcoord);
      load_k(0);
      load_v(0);
    }
  }
  __syncwarp();
  if (warp == 9) tmem_alloc(tm_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tm_holder;
  if (a.inject_timeout) {
    if (lane == 0) wait_bar(&bars[kFwNever], 0, abort_flag, a);
    __syncwarp();
  }
  __syncthreads();

  constexpr bool kBF16 = !FP16;

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && T > 0 && !*abort_flag) {
      for (int t = 1; t < T; ++t) {  // Q and step 0's K, V were issued during the set-up
        const int sk = t % NK, sv = t % NV;
        if (t >= NK && !wait_bar(&bars[kFwKEmpty + sk], ((t / NK) - 1) & 1, abort_flag, a)) break;
        load_k(t);
        if (t >= NV && !wait_bar(&bars[kFwVEmpty + sv], ((t / NV) - 1) & 1, abort_flag, a)) break;
        load_v(t);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t ID_S = idesc_f16(BM, BN, kBF16, false, false);
      constexpr uint32_t ID_O = idesc_f16(BM, DV, kBF16, false, true);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(smem + C::oQ), 16, 1024);
      auto issue_s = [&](int t) -> bool {  // into S buffer t & 1
        const int sk = t % NK;
        const uint64_t dK0 = sdesc_sw128(smem_u32(smem + C::oK + sk * C::kK), 16, 1024);
        if (!wait_bar(&bars[kFwKFull + sk], (t / NK) & 1, abort_flag, a)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + C::cS0 + (t & 1) * BN, sdesc_at(dQ0, (kk >> 2) * BM * 128 + (kk & 3) * 32),
                 sdesc_at(dK0, (kk >> 2) * BN * 128 + (kk & 3) * 32), ID_S, kk > 0);
        mma_commit(&bars[kFwSFull + (t & 1)]);
        mma_commit(&bars[kFwKEmpty + sk]);  // K(t) is read by S(t) only
        return true;
      };
      bool ok = wait_bar(&bars[kFwQFull], 0, abort_flag, a) && issue_s(0) && (T < 2 || issue_s(1));
      for (int t = 0; ok && t < T; ++t) {
        // P(t) written by both warpgroups; V(t) landed (confirmed by them before the handoff)
        if (!(ok = wait_bar(&bars[kFwPFull], t & 1, abort_flag, a))) break;
        tc_fence_after();
        const int sv = t % NV;
        const uint64_t dVt = sdesc_sw128(smem_u32(smem + C::oV + sv * C::kV), BN * 128, 1024);
        const uint32_t sb = tmem + C::cS0 + (t & 1) * BN;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
#pragma unroll
          for (int kk = 0; kk < NC / 16; ++kk)  // keys 16·kk.. of half g: P pairs at +8·kk of its columns
            mma_ts(tmem + C::cO + g * DV, sb + g * NC + kk * 8,
                   sdesc_at(dVt, (g * (NC / 16) + kk) * 2048), ID_O, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bars[kFwOFull]);
        mma_commit(&bars[kFwVEmpty + sv]);
        // S(t+2) may overwrite this buffer once O(t) (issued above) has read its P
        if (t + 2 < T && !(ok = issue_s(t + 2))) break;
      }
      if (!ok) {
        mma_commit(&bars[kFwDrain]);
        mbar_wait(&bars[kFwDrain], 0, kDrainNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ compute warpgroups 0, 1
    const int q4 = warp & 3, g = warp >> 2;
    const int row = q4 * 32 + lane;  // TMEM lane = query row i0 + row
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t oG = tmem + lane_off + C::cO + g * DV;
    const int ir = i0 + row;
    // keys visible to this row: j - ir - off in [lo, hi]
    const long long vlo = (long long)ir + off + lo, vhi = (long long)ir + off + hi;
    const int j_vis_lo = (int)(vlo < -1 ? -1 : (vlo > (1 << 30) ? (1 << 30) : vlo));
    const int j_vis_hi = (int)min((long long)sq.L2 - 1, vhi < -1 ? -1ll : (vhi > (1 << 30) ? (long long)(1 << 30) : vhi));
    const bool i_valid = ir < sq.L1;
    float m = -INFINITY, l = 0.f;  // running reference maximum (log2 units) and row sum of this half
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int j0 = (kb_begin + t) * BN;
      const uint32_t sb = tmem + lane_off + C::cS0 + (t & 1) * BN + g * NC;
      const long long dmin = (long long)j0 - (i0 + BM - 1) - off, dmax = (long long)(j0 + BN - 1) - i0 - off;
      const bool full = j0 + BN <= sq.L2 && dmin >= lo && dmax <= hi;
      if (!(ok = wait_bar_warp(&bars[kFwSFull + (t & 1)], (t >> 1) & 1, abort_flag, a))) break;
      tc_fence_after();
      uint32_t p[NC];
      tmem_ld32(sb, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
      if constexpr (NC == 64) tmem_ld32(sb + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
      tmem_wait_ld();
      reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&p[0]));
      if constexpr (NC == 64) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&p[32]));
      const int jc = j0 + g * NC;
      // The scores stay as loaded (natural units, unscaled).  P = 2^(s·scale_log2 − ref) is one
      // packed fp32x2 FMA per key pair and two ex2; the row sum runs on packed adds over two
      // accumulator pairs.  P goes out in the io dtype, two keys per 32-bit column, over this
      // half's S columns in 16-column pieces as they are ready.
      const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
      uint32_t pk[NC / 2];
      float2 ls2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      auto exp_pair = [&](int c, float2 nref2) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(p[c]), __uint_as_float(p[c + 1])), sc2, nref2);
        const float e0 = ex2(x.x), e1 = ex2(x.y);
        ls2[(c >> 1) & 1] = __fadd2_rn(ls2[(c >> 1) & 1], make_float2(e0, e1));
        pk[c >> 1] = pack2<FP16>(e0, e1);
        if ((c & 31) == 30) tmem_st16(sb + (c >> 5) * 16, *reinterpret_cast<uint32_t(*)[16]>(&pk[(c >> 5) * 16]));
      };
      auto exps = [&](float mref) {
        ls2[0] = ls2[1] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < NC; c += 2) exp_pair(c, make_float2(-mref, -mref));
      };
      // One pass: hide the keys a row does not see (skipped on tiles every row sees whole,
      // `full`, the same for the whole CTA), reduce the row (three-input max over 4 chains; min
      // when the scale is negative, so that the scaled maximum is scale times it) and, after the
      // first tile, form P against the reference maximum of the earlier tiles in the same loop
      // (OPT), so the exponentials need not wait for this tile's maximum.
      const bool neg = a.scale_log2 < 0.f;
      const float hide = neg ? INFINITY : -INFINITY;  // scaled, it is -inf either way
      float red[4] = {hide, hide, hide, hide};
      const float mref_prev = m == -INFINITY ? 0.f : m;
      auto pass = [&](auto full_c, auto opt_c, auto neg_c) {
        constexpr bool kFull = decltype(full_c)::value, kOpt = decltype(opt_c)::value;
        constexpr bool kNeg = decltype(neg_c)::value;
#pragma unroll
        for (int c = 0; c < NC; c += 2) {
          if constexpr (!kFull) {
            if (jc + c < j_vis_lo || jc + c > j_vis_hi) p[c] = __float_as_uint(hide);
            if (jc + c + 1 < j_vis_lo || jc + c + 1 > j_vis_hi) p[c + 1] = __float_as_uint(hide);
          }
          const float r0 = __uint_as_float(p[c]), r1 = __uint_as_float(p[c + 1]);
          if constexpr (kNeg) {
            red[(c >> 1) & 3] = fmin3(red[(c >> 1) & 3], r0, r1);
          } else {
            red[(c >> 1) & 3] = fmax3(red[(c >> 1) & 3], r0, r1);
          }
          if constexpr (kOpt) exp_pair(c, make_float2(-mref_prev, -mref_prev));
        }
      };
      using kT = std::true_type;
      using kF = std::false_type;
      const bool opt = t > 0;  // at t = 0 no row has a reference yet
      auto pass_sign = [&](auto full_c, auto opt_c) {
        if (neg) pass(full_c, opt_c, kT{}); else pass(full_c, opt_c, kF{});
      };
      if (full) {
        if (opt) pass_sign(kT{}, kT{}); else pass_sign(kT{}, kF{});
      } else {
        if (opt) pass_sign(kF{}, kT{}); else pass_sign(kF{}, kF{});
      }
      const float mx = (neg ? fmin3(red[0], red[1], fminf(red[2], red[3]))
                            : fmax3(red[0], red[1], fmaxf(red[2], red[3]))) * a.scale_log2;
      // New reference maximum when a row's block maximum exceeds it by more than 8 (P <= 2^8 in
      // the io dtype otherwise).  The decision is taken per warp (the TMEM loads and stores below
      // are warp-collective); every row of the warp then moves to its own max(m, mx), and P is
      // formed again from the kept scores.
      const bool grow = __any_sync(0xffffffffu, mx > m + 8.f);
      if (grow) {
        const float mnew = fmaxf(m, mx);
        const float alpha = mnew == -INFINITY ? 1.f : ex2(m - mnew);  // 0 while nothing was seen
        l *= alpha;
        if (t > 0) {
          // O(t-1) must be complete; O(t) waits for this step's P handoff below
          if (!(ok = wait_bar_warp(&bars[kFwOFull], (t - 1) & 1, abort_flag, a))) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DV; c += 32) {
            uint32_t r[32];
            tmem_ld32(oG + c, r);
            tmem_wait_ld();
            reg_fence(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
            tmem_st32(oG + c, r);
          }
        }
        m = mnew;
      }
      if (grow || !opt) {
        tmem_wait_st();  // the first P stores of this tile land before these overwrite them
        exps(m == -INFINITY ? 0.f : m);  // every x is -inf when m is: P = 0
      }
      l += (ls2[0].x + ls2[0].y) + (ls2[1].x + ls2[1].y);
      tmem_wait_st();
      // the MMA thread issues O(t) right after this handoff: its V stage must have landed
      if (!(ok = wait_bar_warp(&bars[kFwVFull + t % NV], (t / NV) & 1, abort_flag, a))) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kFwPFull]);
    }
    // ---- epilogue: combine the halves, Y = O / l in the io dtype, lse = ln-sum-exp (+inf: no key)
    if (ok && T > 0) ok = wait_bar_warp(&bars[kFwOFull], (T - 1) & 1, abort_flag, a);
    float* st_m = reinterpret_cast<float*>(smem + C::oStat);
    float* st_l = st_m + 2 * BM;
    st_m[g * BM + row] = m;
    st_l[g * BM + row] = l;
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the eight compute warps
    if (ok) {
      tc_fence_after();
      const float mo = st_m[(1 - g) * BM + row], lo_ = st_l[(1 - g) * BM + row];
      const float m0 = g == 0 ? m : mo, m1 = g == 0 ? mo : m, l0 = g == 0 ? l : lo_, l1 = g == 0 ? lo_ : l;
      float M = fmaxf(m0, m1);
      float c0 = m0 == -INFINITY ? 0.f : ex2(m0 - M), c1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
      float L = l0 * c0 + l1 * c1;
      if (a.sinks) {
        // the q-head's sink logit joins the normaliser with no value: in the log2 units of M,
        // L·2^(M − M') + 2^(sink·log2e − M') with M' = max(M, sink·log2e)
        const float ks = a.sinks[n1] * 1.4426950408889634f;
        const float Mn = fmaxf(M, ks);
        if (Mn != -INFINITY) {
          const float cs = M == -INFINITY ? 0.f : ex2(M - Mn);
          c0 *= cs;
          c1 *= cs;
          L = L * cs + ex2(ks - Mn);
          M = Mn;
        }
      }
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const long long qrow = row_index(a.layout, b, (long long)(tnd ? sq.q0 : 0) + (i_valid ? ir : 0), n1, a.N1, a.S1);
      uint16_t* y = static_cast<uint16_t*>(a.dq) + qrow * a.io_dv;
      // A block whose 128 rows lie inside its sequence is staged in the drained K ring as
      // 128-byte-swizzled 64-column tiles and written by TMA stores (as the backward's epilogues);
      // the last block of a TND sequence is written row by row.
      const bool staged = !tnd || i0 + BM <= sq.span_q;
      uint8_t* stage = smem + C::oK;
#pragma unroll 1
      for (int c = 0; c < DV / 64; ++c) {
        const int col = g * (DV / 2) + c * 32;
        uint32_t r0[32], r1[32];
        if (T > 0) {
          tmem_ld32(tmem + lane_off + C::cO + col, r0);
          tmem_ld32(tmem + lane_off + C::cO + DV + col, r1);
          tmem_wait_ld();
          reg_fence(r0);
          reg_fence(r1);
        }
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          o[e >> 1] = T > 0 ? pack2<FP16>((__uint_as_float(r0[e]) * c0 + __uint_as_float(r1[e]) * c1) * inv,
                                          (__uint_as_float(r0[e + 1]) * c0 + __uint_as_float(r1[e + 1]) * c1) * inv)
                            : 0u;
        if (staged) {
          uint8_t* rowp = stage + (col / 64) * BM * 128 + row * 128;
          const int unit0 = (col % 64) / 8;
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            st_shared_v4(smem_u32(rowp + (((unit0 + v4) ^ (row & 7)) << 4)), o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2],
                         o[4 * v4 + 3]);
        } else if (i_valid) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            if (col + v4 * 8 < a.io_dv)
              *reinterpret_cast<uint4*>(y + col + v4 * 8) = make_uint4(o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2], o[4 * v4 + 3]);
        }
      }
      if (staged) fence_proxy_async_smem();
      if (g == 0 && i_valid) {
        const long long li = tnd ? (long long)n1 * a.T1 + sq.q0 + ir : ((long long)b * a.N1 + n1) * a.S1 + ir;
        a.lse_out[li] = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : INFINITY;
      }
    }
    // every compute thread reaches this barrier; the tiles are stored only if every warp wrote
    // its part (staged is the same in every thread of the CTA)
    if (!tnd || i0 + BM <= sq.span_q) {
      const bool all_ok = compute_warps_all(ok);
      if (all_ok && warp == 0 && lane == 0) {
#pragma unroll 1
        for (int c = 0; c < DV / 64; ++c)
          tma_store_4d(&tm_y, smem + C::oK + c * BM * 128, c * 64, bnsd ? q_row : n1, bnsd ? n1 : q_row, bcoord);
        bulk_commit_group();
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
    fabwd_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_y,
                     const MainArgs a) {
  using C = FwdCfg<D, DV>;
  if constexpr (FLAT) {  // varlen: the sequences' own query blocks back to back
    if (blockIdx.x == 0) {
      // a sequence with a negative span owns no CTA: its cu_seqlens are checked here
      for (int s = threadIdx.x; s < a.B; s += blockDim.x) {
        SeqRange r;
        if (!seq_range(a, s, r)) atomicOr(a.status, FABWD_DEV_BAD_SEQLENS);
      }
    }
    int b, local, nqb;
    bool kv;
    if (!flat_unit(a, blockIdx.x, 0, C::BM, b, local, kv, nqb)) return;
    fwd_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_y, a, local, b, nqb);
  } else {
    fwd_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_y, a, blockIdx.x, blockIdx.y, (a.S1 + C::BM - 1) / C::BM);
  }
}

template <int D, int DV, bool FP16, bool FLAT>
cudaError_t launch_fwd_flat(const MainArgs& a, const MainMaps& m, dim3 grid, cudaStream_t st) {
  using C = FwdCfg<D, DV>;
  if (cudaError_t e = ensure_smem_limit<fabwd_fwd_kernel<D, DV, FP16, FLAT>>((int)C::bytes); e != cudaSuccess)
    return e;
  fabwd_fwd_kernel<D, DV, FP16, FLAT><<<grid, kMainThreads, C::bytes, st>>>(m.q, m.k, m.v, m.dq, a);
  return cudaGetLastError();
}

template <int D, int DV, bool FP16>
cudaError_t launch_fwd_t(const MainArgs& a, const MainMaps& m, cudaStream_t st) {
  using C = FwdCfg<D, DV>;
  if (flat_grid(a.layout, a.B))
    return launch_fwd_flat<D, DV, FP16, true>(
        a, m, dim3((unsigned)(tnd_blocks_bound(a.B, a.S1, a.T1, C::BM) * a.N1), 1), st);
  return launch_fwd_flat<D, DV, FP16, false>(a, m, dim3(((a.S1 + C::BM - 1) / C::BM) * a.N1, a.B), st);
}

}  // namespace fabwd
