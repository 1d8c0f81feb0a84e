// Fused FlashAttention backward kernel of the atomic dQ mode for sm_103a: warp-specialised
// tcgen05 + TMEM + TMA with two ping-ponged TMEM slots; all five products in one CTA, dQ reduced
// into an fp32 workspace accumulator.  It also holds the helpers (sequence ranges, mask bounds,
// bounded waits) that the other backward kernels share.
//
// What it computes is the backward of the page "CANN ops-transformer FlashAttnGrad 算子详解"
// (discosf.com/news/4863418), §一.  One CTA owns a block of 128 keys of one kv-head and loops
// over steps t = (q-head of the group, 64-row q-block that can see the block):
//     Sᵀ  = K·Qᵀ                 tcgen05 (M = 128 keys, N = 64 queries, K = D)
//     dPᵀ = V·dOᵀ                tcgen05 (K = Dv)
//     Pᵀ  = exp2(Sᵀ·scale·log2e − lse·log2e), masked pairs -> 0, written back to TMEM (bf16/fp16)
//     dSᵀ = Pᵀ ⊙ (dPᵀ − sfmg)    -> TMEM and shared memory (bf16/fp16)
//     dV += Pᵀ·dO                tcgen05, A operand read from TMEM
//     dK += dSᵀ·Q                tcgen05, A operand read from TMEM; accumulated over all steps
//     dQᵀ = Kᵀ·dSᵀ               tcgen05 (M = 128 head-dim rows) -> fp32 reduce-add into the
//                                workspace accumulator, one coalesced 128-byte line per warp
// The five products are §5.2's MM2, MM1, MM5, MM4, MM3 and the elementwise steps its V2-V4.
// K is read K-major (Sᵀ) and MN-major (dQᵀ) from one shared-memory copy; Q and dO likewise
// serve two products each, and dSᵀ serves dK (K-major) and dQᵀ (MN-major).
//
// Schedule (D <= 128).  Steps alternate between two TMEM slots (Sᵀ/Pᵀ and dPᵀ/dQᵀ per slot) and
// two compute warpgroups: warpgroup g (warps 4g..4g+3, warp w reading TMEM lanes 32·(w%4)..+31)
// handles the steps t ≡ g (mod 2).  The MMA warp issues, for step t, the Sᵀ/dPᵀ products of step
// t+1 (other slot) and then dV, dK, dQᵀ of step t, so each warpgroup's softmax/dS work overlaps
// the other slot's products.  Warp 8 streams Q, dO, lse and sfmg through a 4-stage ring (K and V
// once).  With D = 192 (dK alone takes 192 TMEM columns) there is one slot: both warpgroups work
// on every step, 32 query columns each, and dQᵀ is two M = 128 products (head-dim rows 0..127
// and 64..191, of which rows 128..191 are kept).
//
// TMEM columns: dK [0, D), dV [D, D+Dv), slot g at D+Dv+128g: Sᵀ [+0, +64) overwritten by Pᵀ
// [+0, +32) and dSᵀ [+32, +64) (16-bit pairs), dPᵀ/dQᵀ [+64, +128).
// Shared memory: K (padded to 128 head-dim columns), V, 4×(Q, dO, lse, sfmg), 2×dSᵀ.  Tiles are
// 128-byte-swizzled [64-column block][rows][64] arrays (TMA SWIZZLE_128B, box {64,1,rows,1}).
//
// Every mbarrier wait is bounded (MainArgs::wait_ns).  A wait that gives up sets a CTA abort
// flag and FABWD_DEV_TIMEOUT; the other roles see the flag and leave their loops, the MMA
// issuer drains its MMAs, TMA loads in flight get a bounded grace period, and TMEM is freed.
#pragma once

#include "fabwd_internal.cuh"
#include "fabwd_ptx.cuh"
#include "../../include/fabwd.h"

namespace fabwd {

constexpr unsigned long long kDrainNs = 100ull * 1000ull * 1000ull;  // 100 ms
constexpr unsigned long long kGraceNs = 2ull * 1000ull * 1000ull;    // 2 ms
constexpr int kMainThreads = 320;

template <int D, int DV>
struct MainCfg {
  static constexpr int BR = kBlockQ, BC = kBlockKV;
  // Head dims up to 128 leave TMEM room for two slots (ping-pong between the warpgroups); D = 192
  // (dK alone takes 192 columns) leaves room for one, which both warpgroups share, 32 query
  // columns each.
  static constexpr int NSLOT = D > 128 ? 1 : 2;
  static constexpr int NC = NSLOT == 2 ? 64 : 32;       // query columns per compute thread per step
  static constexpr int NS = D > 128 ? 3 : 4;            // Q/dO/lse/sfmg ring stages
  static constexpr bool DQ2 = D > 128;               // second dQᵀ product for head-dim rows 128..D-1
  static constexpr int DK = D < 128 ? 128 : D;           // K rows padded so dQᵀ = Kᵀ·dSᵀ has M = 128
  static constexpr uint32_t kK = DK * BC * 2, kV = DV * BC * 2, kQ = D * BR * 2, kdO = DV * BR * 2;
  static constexpr uint32_t kdS = BC * BR * 2;
  static constexpr uint32_t oK = 0, oV = oK + kK, oQ = oV + kV, odO = oQ + NS * kQ, odS = odO + NS * kdO;
  static constexpr uint32_t oL = odS + NSLOT * kdS;  // [NS][BR] fp32 lse·log2(e)
  static constexpr uint32_t oF = oL + NS * BR * 4;    // [NS][BR] fp32 sfmg
  static constexpr uint32_t oBar = oF + NS * BR * 4;  // mbarriers
  static constexpr uint32_t oMisc = oBar + 48 * 8;    // TMEM base holder, abort flag
  static constexpr uint32_t bytes = oMisc + 64;
  static constexpr uint32_t cDK = 0, cDV = D, cSlot = D + DV;  // slot g: cSlot + 128 g
  static constexpr uint32_t cDQ2 = cSlot + 128 * NSLOT;       // second dQᵀ part (D = 192)
  static_assert(BR == 64, "the slot layout assumes 64-row q-blocks");
  static_assert(D % 64 == 0 && DV % 64 == 0 && (D <= 128 || (D == 192 && DV <= 128)) && DV <= D, "head dims");
  static_assert(cDQ2 + (DQ2 ? 64 : 0) <= 512, "TMEM budget");
  static_assert(bytes <= 232448, "shared memory budget");
  static_assert((D / 64 + DV / 64) * BC * 128 <= NS * (kQ + kdO), "dK/dV staging fits in the Q/dO ring");
};

// mbarrier indices
constexpr int kKvFull = 0, kQFull = 1 /*+NS*/, kQEmpty = 5 /*+NS*/, kSFull = 9 /*+2*/, kDpFull = 11 /*+2*/,
              kDqFull = 13 /*+2*/, kPFull = 15 /*+2*/, kDsFull = 17 /*+2*/, kDqEmpty = 19 /*+2*/, kAccDone = 21,
              kNever = 22, kDrain = 23, kNumBars = 24;

struct SeqRange {
  int q0, L1, k0, L2;
  int span_q, span_k;  // the sequence's rows (TND: from cu_seqlens; else S1, S2), before seqused
};

// Rows of sequence (TND) or batch row b: its first q row and key row, and the lengths that take
// part, after seqused when given.  False when cu_seqlens or seqused are inconsistent (the
// preprocess kernel reports that; the caller touches nothing).
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
  r.span_q = r.L1;
  r.span_k = r.L2;
  if (a.used_q) {
    const int u = a.used_q[b];
    if (u < 0 || u > r.L1) return false;
    r.L1 = u;
  }
  if (a.used_kv) {
    const int u = a.used_kv[b];
    if (u < 0 || u > r.L2) return false;
    r.L2 = u;
  }
  return true;
}

// Work unit f of a varlen grid.  Sequence b owns ceil(L2_b / kv_rows) · N2 dK/dV units (none
// when kv_rows is 0) followed by ceil(L1_b / q_rows) · N1 dQ units (none when q_rows is 0), the
// sequences back to back, L1_b / L2_b their cu_seqlens spans clamped to [0, max_seqlen].  Gives
// the sequence, whether the unit is a dK/dV one, its index among that kind's units of the
// sequence and the sequence's count of q_rows-row query blocks; false past the last unit.  Each
// warp scans the sequences 32 at a time (lane = sequence), so every thread of the CTA gets the
// result without shared memory; called by whole warps.
__device__ __forceinline__ bool flat_unit(const MainArgs& a, long long f, int kv_rows, int q_rows, int& b,
                                          int& local, bool& kv, int& nqb) {
  const int lane = threadIdx.x & 31;
  long long base = 0;  // units of the sequences before this group of 32
  for (int c0 = 0; c0 < a.B; c0 += 32) {
    const int s = c0 + lane;
    long long lq = 0, lk = 0;
    if (s < a.B) {
      lq = (long long)a.cu_q[s + 1] - a.cu_q[s];
      lk = (long long)a.cu_kv[s + 1] - a.cu_kv[s];
      lq = lq < 0 ? 0 : (lq > a.S1 ? a.S1 : lq);
      lk = lk < 0 ? 0 : (lk > a.S2 ? a.S2 : lk);
    }
    const long long nk = kv_rows > 0 ? (lk + kv_rows - 1) / kv_rows * a.N2 : 0;
    const long long nq = q_rows > 0 ? (lq + q_rows - 1) / q_rows * a.N1 : 0;
    long long incl = nk + nq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const long long excl = incl - nk - nq;
    const unsigned hit = __ballot_sync(0xffffffffu, f >= base + excl && f < base + incl);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const long long r = f - base - __shfl_sync(0xffffffffu, excl, src);
      const long long nks = __shfl_sync(0xffffffffu, nk, src);
      b = c0 + src;
      kv = r < nks;
      local = (int)(kv ? r : r - nks);
      nqb = q_rows > 0 ? (int)((__shfl_sync(0xffffffffu, lq, src) + q_rows - 1) / q_rows) : 0;
      return true;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return false;
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

// Bounded wait shared by all roles: gives up on the CTA abort flag or after wait_ns.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, const MainArgs& a) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > a.wait_ns) {
      *abort_flag = 1;
      atomicOr(a.status, FABWD_DEV_TIMEOUT);
      return false;
    }
  }
}

// Warp-uniform variant: the warp proceeds only if every lane saw the phase complete.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              const MainArgs& a) {
  const bool ok = wait_bar(bar, parity, abort_flag, a);
  return __all_sync(0xffffffffu, ok);
}

// One CTA of the fused kernel (atomic dQ mode): key block bx / N2 of kv-head bx % N2, batch (or
// sequence) by; dK and dV into the outputs, dQᵀ reduced into the fp32 workspace accumulator.
template <int D, int DV, bool FP16>
__device__ __forceinline__ void main_block(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                           const CUtensorMap& tm_do, const CUtensorMap& tm_dk, const CUtensorMap& tm_dv,
                                           const MainArgs& a, int bx, int by) {
  using C = MainCfg<D, DV>;
  constexpr int BR = C::BR, BC = C::BC, NS = C::NS;
  extern __shared__ __align__(1024) uint8_t smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int jb = bx / a.N2, n2 = bx % a.N2, b = by;

  SeqRange sq;
  if (!seq_range(a, b, sq)) return;  // bad cu_seqlens: the preprocess kernel reports it
  const int j0 = jb * BC;
  if (j0 >= sq.L2) return;
  if ((smem_u32(smem) & 1023u) != 0) {  // swizzled tiles need 1024-byte alignment
    griddep_wait();  // the preprocess clears the status word
    if (tid == 0) atomicOr(a.status, FABWD_DEV_INTERNAL);
    return;
  }
  const int j1 = min(j0 + BC, sq.L2);
  const long long off = (long long)sq.L2 - sq.L1;
  long long lo, hi;
  mask_bounds(a, lo, hi);
  // q rows that see at least one key of [j0, j1)
  long long ib = (long long)j0 - off - hi, ie = (long long)(j1 - 1) - off - lo;
  if (ib < 0) ib = 0;
  if (ie > sq.L1 - 1) ie = sq.L1 - 1;
  const int qb_begin = ib <= ie ? (int)(ib / BR) : 0;
  const int nqb = ib <= ie ? (int)(ie / BR) + 1 - qb_begin : 0;
  const int T = nqb * a.G;  // steps: (head in group, q-block)

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::oBar);
  uint32_t* tm_holder = reinterpret_cast<uint32_t*>(smem + C::oMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::oMisc + 16);

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool per_warp = (i >= kPFull && i < kPFull + 2) || (i >= kDsFull && i < kDsFull + 2) ||
                            (i >= kDqEmpty && i < kDqEmpty + 2);
      mbar_init(&bars[i], per_warp ? (C::NSLOT == 2 ? 4 : 8) : 1);  // one arrival per compute warp of the slot
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
  }
  if (D < C::DK && warp < 8) {  // zero the K padding columns (read by the dQᵀ product only)
    uint4* z = reinterpret_cast<uint4*>(smem + C::oK + (D / 64) * BC * 128);
    const int n16 = (C::DK - D) / 64 * BC * 128 / 16;
    for (int x = tid; x < n16; x += 256) z[x] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
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

  if (a.inject_timeout) {  // fault injection for tests: a wait that nothing completes
    if (lane == 0) wait_bar(&bars[kNever], 0, abort_flag, a);
    __syncwarp();
  }
  __syncthreads();

  const bool tnd = a.layout == kTND, bnsd = a.layout == kBNSD;
  const int kv_row0 = tnd ? sq.k0 + j0 : j0;
  const int q_rowbase = tnd ? sq.q0 : 0;
  const int bcoord = tnd ? 0 : b;
  constexpr bool kBF16 = !FP16;

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0 && T > 0 && !*abort_flag) {
      mbar_arrive_expect_tx(&bars[kKvFull], (D + DV) * BC * 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_4d(smem + C::oK + c * BC * 128, &tm_k, &bars[kKvFull], c * 64, bnsd ? kv_row0 : n2,
                    bnsd ? n2 : kv_row0, bcoord);
#pragma unroll
      for (int c = 0; c < DV / 64; ++c)
        tma_load_4d(smem + C::oV + c * BC * 128, &tm_v, &bars[kKvFull], c * 64, bnsd ? kv_row0 : n2,
                    bnsd ? n2 : kv_row0, bcoord);
      for (int t = 0; t < T; ++t) {
        const int st = t % NS;
        const int h = t / nqb, qb = qb_begin + t % nqb;
        const int n1 = n2 * a.G + h, i0 = qb * BR;
        if (t >= NS && !wait_bar(&bars[kQEmpty + st], ((t / NS) - 1) & 1, abort_flag, a)) break;
        uint64_t* full = &bars[kQFull + st];
        mbar_arrive_expect_tx(full, (D + DV) * BR * 2 + 2 * BR * 4);
        const int row = q_rowbase + i0;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(smem + C::oQ + st * C::kQ + c * BR * 128, &tm_q, full, c * 64, bnsd ? row : n1,
                      bnsd ? n1 : row, bcoord);
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          tma_load_4d(smem + C::odO + st * C::kdO + c * BR * 128, &tm_do, full, c * 64, bnsd ? row : n1,
                      bnsd ? n1 : row, bcoord);
        const long long rbase = ((long long)b * a.N1 + n1) * a.S1p + i0;
        bulk_load(smem + C::oL + st * BR * 4, a.lse2 + rbase, BR * 4, full);
        bulk_load(smem + C::oF + st * BR * 4, a.sfmg + rbase, BR * 4, full);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && T > 0) {
      constexpr uint32_t ID_S = idesc_f16(BC, BR, kBF16, false, false);
      constexpr uint32_t ID_DV = idesc_f16(BC, DV, kBF16, false, true);
      constexpr uint32_t ID_DK = idesc_f16(BC, D, kBF16, false, true);
      constexpr uint32_t ID_DQ = idesc_f16(128, BR, kBF16, true, true);
      const uint32_t aK = smem_u32(smem + C::oK), aV = smem_u32(smem + C::oV);
      // Sᵀ(t) and dPᵀ(t) into slot t % NSLOT
      auto issue_s_dp = [&](int t) -> bool {
        const int g = t % C::NSLOT, st = t % NS, use = t / C::NSLOT;
        const uint32_t aQ = smem_u32(smem + C::oQ + st * C::kQ), adO = smem_u32(smem + C::odO + st * C::kdO);
        const uint32_t slot = tmem + C::cSlot + g * 128;
        if (!wait_bar(&bars[kQFull + st], (t / NS) & 1, abort_flag, a)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(slot, sdesc_sw128(aK + (kk >> 2) * BC * 128 + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(aQ + (kk >> 2) * BR * 128 + (kk & 3) * 32, 16, 1024), ID_S, kk > 0);
        mma_commit(&bars[kSFull + g]);
        // dPᵀ reuses the slot's dPᵀ/dQᵀ columns: wait until the previous dQᵀ was read
        if (use >= 1 && !wait_bar(&bars[kDqEmpty + g], (use - 1) & 1, abort_flag, a)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          mma_ss(slot + 64, sdesc_sw128(aV + (kk >> 2) * BC * 128 + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(adO + (kk >> 2) * BR * 128 + (kk & 3) * 32, 16, 1024), ID_S, kk > 0);
        mma_commit(&bars[kDpFull + g]);
        return true;
      };
      // Pᵀ / dSᵀ TMEM columns of k-step kk (16 queries): with two slots one warpgroup owns all 64
      // queries (Pᵀ at +0, dSᵀ at +32); with one slot warpgroup kk/2 owns 32 (Pᵀ at +0, dSᵀ at +16
      // within its own 32 Sᵀ columns)
      auto p_col = [](int kk) { return C::NSLOT == 2 ? kk * 8 : (kk >> 1) * 32 + (kk & 1) * 8; };
      auto ds_col = [](int kk) { return C::NSLOT == 2 ? 32 + kk * 8 : (kk >> 1) * 32 + 16 + (kk & 1) * 8; };
      // dV, dK, dQᵀ of step t
      auto issue_grads = [&](int t) -> bool {
        const int g = t % C::NSLOT, st = t % NS;
        const uint32_t aQ = smem_u32(smem + C::oQ + st * C::kQ), adO = smem_u32(smem + C::odO + st * C::kdO);
        const uint32_t adS = smem_u32(smem + C::odS + g * C::kdS);
        const uint32_t slot = tmem + C::cSlot + g * 128;
        const uint32_t u = (t / C::NSLOT) & 1;
        if (!wait_bar(&bars[kPFull + g], u, abort_flag, a)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)
          mma_ts(tmem + C::cDV, slot + p_col(kk), sdesc_sw128(adO + kk * 2048, BR * 128, 1024), ID_DV,
                 (t > 0 || kk > 0) ? 1u : 0u);
        if (!wait_bar(&bars[kDsFull + g], u, abort_flag, a)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BR / 16; ++kk)  // dSᵀ from TMEM (next to Pᵀ)
          mma_ts(tmem + C::cDK, slot + ds_col(kk), sdesc_sw128(aQ + kk * 2048, BR * 128, 1024), ID_DK,
                 (t > 0 || kk > 0) ? 1u : 0u);
        {
#pragma unroll
          for (int kk = 0; kk < BC / 16; ++kk)
            mma_ss(slot + 64, sdesc_sw128(aK + kk * 2048, BC * 128, 1024), sdesc_sw128(adS + kk * 2048, BC * 128, 1024),
                   ID_DQ, kk > 0);
          if constexpr (C::DQ2) {  // head-dim rows 64..191 (rows 64..127 again; only 128..191 are used)
#pragma unroll
            for (int kk = 0; kk < BC / 16; ++kk)
              mma_ss(tmem + C::cDQ2, sdesc_sw128(aK + BC * 128 + kk * 2048, BC * 128, 1024),
                     sdesc_sw128(adS + kk * 2048, BC * 128, 1024), ID_DQ, kk > 0);
          }
          mma_commit(&bars[kDqFull + g]);
        }
        mma_commit(&bars[kQEmpty + st]);
        return true;
      };
      bool ok = wait_bar(&bars[kKvFull], 0, abort_flag, a) && issue_s_dp(0);
      for (int t = 0; ok && t < T; ++t) {
        if (C::NSLOT == 2) {  // the other slot's Sᵀ/dPᵀ go first, overlapping this slot's dS work
          if (t + 1 < T && !(ok = issue_s_dp(t + 1))) break;
          ok = issue_grads(t);
        } else {
          if (!(ok = issue_grads(t))) break;
          if (t + 1 < T) ok = issue_s_dp(t + 1);
        }
      }
      if (ok) {
        mma_commit(&bars[kAccDone]);
      } else {
        mma_commit(&bars[kDrain]);
        mbar_wait(&bars[kDrain], 0, kDrainNs);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ compute warpgroups 0, 1
    const int q4 = warp & 3, g = warp >> 2;
    const int row = q4 * 32 + lane;  // TMEM lane: key row (Sᵀ, dPᵀ, dK, dV) or head-dim row (dQᵀ)
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    constexpr int NC = C::NC;
    const int cb = C::NSLOT == 2 ? 0 : 32 * g;  // this warpgroup's first query column of a step
    const int jr = j0 + row;
    const bool j_valid = jr < sq.L2;
    const long long vlo = (long long)jr - off - hi, vhi = (long long)jr - off - lo;
    const int i_vis_lo = (int)(vlo < -1 ? -1 : (vlo > (1 << 30) ? (1 << 30) : vlo));
    const int i_vis_hi = (int)(vhi < -1 ? -1 : (vhi > (1 << 30) ? (1 << 30) : vhi));
    const uint32_t adS_row = smem_u32(smem + C::odS) + row * 128;
    const long long i_stride = bnsd ? a.io_d : (long long)a.N1 * a.io_d;
    bool ok = true;
    const int sg = C::NSLOT == 2 ? g : 0;  // the slot this warpgroup works on
    const uint32_t slot = tmem + lane_off + C::cSlot + sg * 128;
    const uint32_t adS = adS_row + sg * C::kdS;
    constexpr int kTStep = C::NSLOT == 2 ? 2 : 1;
    for (int t = C::NSLOT == 2 ? g : 0; t < T; t += kTStep) {
      const int st = t % NS;
      const uint32_t u = (C::NSLOT == 2 ? (t >> 1) : t) & 1;
      const int h = t / nqb, qb = qb_begin + t % nqb;
      const int n1 = n2 * a.G + h, i0 = qb * BR;
      if (!(ok = wait_bar_warp(&bars[kQFull + st], (t / NS) & 1, abort_flag, a))) break;
      if (!(ok = wait_bar_warp(&bars[kSFull + sg], u, abort_flag, a))) break;
      tc_fence_after();
      const float4* sL4 = reinterpret_cast<const float4*>(smem + C::oL + st * BR * 4 + cb * 4);
      const float4* sF4 = reinterpret_cast<const float4*>(smem + C::oF + st * BR * 4 + cb * 4);
      const long long dmin = (long long)j0 - (i0 + BR - 1) - off, dmax = (long long)(j1 - 1) - i0 - off;
      const bool full = dmin >= lo && dmax <= hi;
      uint32_t p[NC];  // Sᵀ row, then P (fp32 bits)
#pragma unroll
      for (int k = 0; k < NC / 32; ++k) tmem_ld32(slot + cb + 32 * k, *reinterpret_cast<uint32_t(*)[32]>(&p[32 * k]));
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < NC / 32; ++k) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&p[32 * k]));
#pragma unroll
      for (int c4 = 0; c4 < NC / 4; ++c4) {
        const float4 l = sL4[c4];
        const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 4 * c4 + e;
          p[c] = __float_as_uint(ex2(fmaf(__uint_as_float(p[c]), a.scale_log2, -lv[e])));
        }
      }
      if (!full) {
#pragma unroll
        for (int c = 0; c < NC; ++c)
          if (i0 + cb + c < i_vis_lo || i0 + cb + c > i_vis_hi) p[c] = 0u;
      }
      if (!j_valid) {
#pragma unroll
        for (int c = 0; c < NC; ++c) p[c] = 0u;
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < NC / 2; ++c) pk[c] = pack2<FP16>(__uint_as_float(p[2 * c]), __uint_as_float(p[2 * c + 1]));
        if constexpr (NC == 64) tmem_st32(slot, pk);  // Pᵀ over this warpgroup's own Sᵀ columns
        else tmem_st16(slot + cb, *reinterpret_cast<uint32_t(*)[16]>(&pk[0]));
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kPFull + sg]);
      if (!(ok = wait_bar_warp(&bars[kDpFull + sg], u, abort_flag, a))) break;
      tc_fence_after();
      const uint32_t ds_tmem = slot + (C::NSLOT == 2 ? 32 : cb + 16);
#pragma unroll
      for (int hh = 0; hh < NC / 32; ++hh) {
        uint32_t r[32];
        tmem_ld32(slot + 64 + cb + hh * 32, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t dk[16];
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 f = sF4[hh * 8 + c4];
          const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int c = 4 * c4 + e;
            const float d0 = __uint_as_float(p[hh * 32 + c]) * (__uint_as_float(r[c]) - fv[e]);
            const float d1 = __uint_as_float(p[hh * 32 + c + 1]) * (__uint_as_float(r[c + 1]) - fv[e + 1]);
            dk[c >> 1] = pack2<FP16>(d0, d1);
          }
        }
        tmem_st16(ds_tmem + hh * 16, dk);  // dSᵀ (A operand of dK) next to Pᵀ
        {  // dSᵀ also in shared memory: the B operand of dQᵀ
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            st_shared_v4(adS + ((((cb / 8 + hh * 4 + v4) ^ (row & 7))) << 4), dk[4 * v4], dk[4 * v4 + 1],
                         dk[4 * v4 + 2], dk[4 * v4 + 3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kDsFull + sg]);
      if (!(ok = wait_bar_warp(&bars[kDqFull + sg], u, abort_flag, a))) break;
      tc_fence_after();
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(slot + 64 + cb, r0);
        if constexpr (NC == 64) tmem_ld32(slot + 96 + cb, r1);
        tmem_wait_ld();
        reg_fence(r0);
        if constexpr (NC == 64) reg_fence(r1);
        if constexpr (!C::DQ2) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kDqEmpty + sg]);
        }
        const int nvalid = min(NC, sq.L1 - (i0 + cb));
        if (row < a.io_d) {  // lane = head-dim index d; columns = queries i0 + cb .. + NC - 1
          float* dst = a.dq_acc +
                       row_index(a.layout, b, (long long)q_rowbase + (nvalid > 0 ? i0 + cb : 0), n1, a.N1, a.S1) * a.io_d + row;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c < nvalid) red_add_f32(dst + c * i_stride, __uint_as_float(r0[c]));
          if constexpr (NC == 64) {
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c + 32 < nvalid) red_add_f32(dst + (c + 32) * i_stride, __uint_as_float(r1[c]));
          }
        }
        if constexpr (C::DQ2) {  // lanes 64..127 of the second part hold head-dim rows 128..191
          if (q4 >= 2) {
            tmem_ld32(tmem + lane_off + C::cDQ2 + cb, r0);
            tmem_wait_ld();
            reg_fence(r0);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kDqEmpty + sg]);
          if (q4 >= 2 && 64 + row < a.io_d) {
            float* dst = a.dq_acc +
                         row_index(a.layout, b, (long long)q_rowbase + (nvalid > 0 ? i0 + cb : 0), n1, a.N1, a.S1) * a.io_d +
                         64 + row;
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c < nvalid) red_add_f32(dst + c * i_stride, __uint_as_float(r0[c]));
          }
        }
      }
    }
    // ---- epilogue: dK = scale · acc, dV = acc; zeros when no query sees this block.  Blocks
    // inside their sequence are staged in the drained Q/dO ring and written by TMA stores, the
    // last block of a TND sequence row by row (as in the separate mode's dK/dV CTAs).
    if (ok && T > 0) ok = wait_bar_warp(&bars[kAccDone], 0, abort_flag, a);
    const bool staged = !tnd || j0 + BC <= sq.span_k;  // the same in every thread of the CTA
    if (staged) {
      tc_fence_after();
      uint8_t* stage = smem + C::oQ;  // D/64 dK tiles, then Dv/64 dV tiles, BC·128 bytes each
#pragma unroll 1
      for (int c = 0; ok && c < D / 64 + DV / 64; ++c) {
        const bool kpart = c < D / 64;
        const int col = kpart ? g * (D / 2) + c * 32 : g * (DV / 2) + (c - D / 64) * 32;
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + (kpart ? C::cDK : C::cDV) + col, r);
        tmem_wait_ld();
        reg_fence(r);
        const float s = kpart ? a.scale : 1.f;
        uint32_t o[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2)
          o[e >> 1] = T > 0 ? pack2<FP16>(__uint_as_float(r[e]) * s, __uint_as_float(r[e + 1]) * s) : 0u;
        uint8_t* rowp = stage + ((kpart ? 0 : D / 64) + col / 64) * BC * 128 + row * 128;
        const int unit0 = (col % 64) / 8;
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4)
          st_shared_v4(smem_u32(rowp + (((unit0 + v4) ^ (row & 7)) << 4)), o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2],
                       o[4 * v4 + 3]);
      }
      fence_proxy_async_smem();
      const bool all_ok = compute_warps_all(ok);  // every compute thread reaches this barrier
      if (all_ok && warp == 0 && lane == 0) {
#pragma unroll 1
        for (int c = 0; c < D / 64 + DV / 64; ++c) {
          const CUtensorMap* m = c < D / 64 ? &tm_dk : &tm_dv;
          const int x = (c < D / 64 ? c : c - D / 64) * 64;
          tma_store_4d(m, stage + c * BC * 128, x, bnsd ? kv_row0 : n2, bnsd ? n2 : kv_row0, bcoord);
        }
        bulk_commit_group();
      }
    } else if (ok) {
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
          o[e >> 1] = T > 0 ? pack2<FP16>(__uint_as_float(r[e]) * a.scale, __uint_as_float(r[e + 1]) * a.scale) : 0u;
        if (j_valid) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            if (col + v4 * 8 < a.io_d)
              *reinterpret_cast<uint4*>(dk + col + v4 * 8) =
                  make_uint4(o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2], o[4 * v4 + 3]);
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
              *reinterpret_cast<uint4*>(dv + col + v4 * 8) =
                  make_uint4(o[4 * v4], o[4 * v4 + 1], o[4 * v4 + 2], o[4 * v4 + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) {  // bounded grace period for TMA loads still in flight
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
    fabwd_main_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                      const MainArgs a) {
  if constexpr (FLAT) {  // varlen: the sequences' own key blocks back to back
    int b, local, nqb;
    bool kv;
    if (!flat_unit(a, blockIdx.x, kBlockKV, 0, b, local, kv, nqb)) return;
    main_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv, a, local, b);
  } else {
    main_block<D, DV, FP16>(tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv, a, blockIdx.x, blockIdx.y);
  }
}

template <int D, int DV, bool FP16, bool FLAT>
cudaError_t launch_main_flat(const MainArgs& a, const MainMaps& m, dim3 grid, cudaStream_t st) {
  using C = MainCfg<D, DV>;
  if (cudaError_t e = ensure_smem_limit<fabwd_main_kernel<D, DV, FP16, FLAT>>((int)C::bytes); e != cudaSuccess)
    return e;
  fabwd_main_kernel<D, DV, FP16, FLAT><<<grid, kMainThreads, C::bytes, st>>>(m.q, m.k, m.v, m.dout, m.dk, m.dv, a);
  return cudaGetLastError();
}

template <int D, int DV, bool FP16>
cudaError_t launch_main_t(const MainArgs& a, const MainMaps& m, int n_kv_blocks, cudaStream_t st) {
  // blockIdx.x = kv-block * N2 + kv-head: the heaviest kv-blocks (earliest keys under a causal
  // mask) of every head launch first.
  if (flat_grid(a.layout, a.B))
    return launch_main_flat<D, DV, FP16, true>(
        a, m, dim3((unsigned)(tnd_blocks_bound(a.B, a.S2, a.T2, kBlockKV) * a.N2), 1), st);
  return launch_main_flat<D, DV, FP16, false>(a, m, dim3(n_kv_blocks * a.N2, a.B), st);
}

}  // namespace fabwd
