// HBM-bound kernels around the main backward kernel:
//   preprocess: sfmg = rowsum(dout ⊙ attn_out) (the V1 "softmaxGradFront" stage of the page
//               "CANN ops-transformer FlashAttnGrad 算子详解", §5.2 data flow), lse · log2(e)
//               into padded rows, the fp32 dQ accumulator zeroed, device status cleared and
//               the cu_seqlens checked;
//   convert:    dq = cast(scale · dQ accumulator) (the fp32-workspace dQ of the same page's
//               bn2gs1s2 template, §5.2).
#include "fabwd_internal.cuh"
#include "fabwd_ptx.cuh"
#include "../../include/fabwd.h"

#include <cmath>
#include <type_traits>

namespace fabwd {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <bool FP16, int DV, bool SMALL>
__global__ void __launch_bounds__(256) preprocess_kernel(PreArgs a) {
  // the backward kernel that follows may start its set-up now; it waits for this grid to finish
  // before it reads the rows written here
  griddep_launch_dependents();
  if (blockIdx.x == 0) {
    // block 0 clears the status word, then its threads check the sequences in parallel
    if (threadIdx.x == 0) {
      unsigned st = 0;
      if (a.layout == kTND && (a.cu_q[0] != 0 || a.cu_kv[0] != 0 || a.cu_q[a.B] != a.T1 || a.cu_kv[a.B] != a.T2))
        st |= FABWD_DEV_BAD_SEQLENS;
      *a.status = st;
    }
    __syncthreads();
    unsigned bad = 0;
    for (int s = threadIdx.x; s < a.B; s += blockDim.x) {
      long long lq = a.S1, lk = a.S2;
      if (a.layout == kTND) {
        lq = (long long)a.cu_q[s + 1] - a.cu_q[s];
        lk = (long long)a.cu_kv[s + 1] - a.cu_kv[s];
        if (lq < 0 || lq > a.S1 || lk < 0 || lk > a.S2) bad = 1;
      }
      if (a.used_q && (a.used_q[s] < 0 || a.used_q[s] > lq)) bad = 1;
      if (a.used_kv && (a.used_kv[s] < 0 || a.used_kv[s] > lk)) bad = 1;
    }
    if (bad) atomicOr(a.status, FABWD_DEV_BAD_SEQLENS);
  }

  // Grid-stride over iterations of RPI consecutive rows (b, n1, i0 .. i0 + RPI - 1), i over the
  // padded length S1p: the order of the lse, lse2 and sfmg rows, so that a warp's 4-byte reads
  // and writes of them are contiguous (a row's dout and attn_out, 2·Dv bytes each, are whole
  // 128-byte lines in any order).  Iterations go heads fastest, (b, i0, n1), so that the warps
  // resident together read the rows of a few positions across all heads: in BSND and TND those
  // are contiguous stretches of dout and attn_out.  An iteration is UN groups of RPW rows with
  // LPR lanes per row, whose dout, attn_out and lse loads are all issued before the arithmetic.
  // RPI divides S1p (a multiple of 128), so the rows of an iteration share (b, n1) and one
  // 128-row block: the index split, the sequence bounds and the first row's addresses are worked
  // out once per iteration and stepped per row.  SMALL: every row index fits 32 bits, so the
  // split uses 32-bit division.
  // DV is the kernel's row width (64, 128 or 192); a.Dv (a multiple of 8, at most DV) the rows'
  // own length: chunks past it are not read.
  constexpr int CPL = DV == 192 ? 3 : 1;  // 16-byte chunks (8 elements) per lane and row
  constexpr int LPR = DV / (8 * CPL);     // lanes per row (a power of two)
  constexpr int RPW = 32 / LPR;           // rows per warp step
  constexpr int UN = 4;                   // row groups per iteration
  constexpr int RPI = RPW * UN;           // rows per warp iteration
  static_assert(kRowPad % RPI == 0, "an iteration's rows stay within one padded row block");
  long long ngroups = (long long)a.B * a.N1 * a.S1p / RPI;
  const long long gwarp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarp = ((long long)gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, part = lane % LPR;
  const bool tnd = a.layout == kTND;
  const long long rstep = a.layout == kBNSD ? 1 : a.N1;  // row_index step from row i to i + 1
  // Varlen with up to 64 sequences: the iterations run over each sequence's own rows up to its
  // last 128-row block only (lanes s and s + 32 of every warp hold sequences s and s + 32: their
  // counts of iterations and running sums), instead of max_seqlen rows per sequence of which the
  // excess is skipped.
  const bool compact = tnd && a.B <= 64;
  long long cnt0 = 0, cnt1 = 0, incl0 = 0, incl1 = 0;
  if (compact) {
    auto count = [&](int s) -> long long {  // iterations of sequence s (0 past the last one)
      if (s >= a.B) return 0;
      const long long s0 = a.cu_q[s];
      long long L = (long long)a.cu_q[s + 1] - s0;
      if (s0 < 0 || s0 > a.T1) L = 0;
      L = L < 0 ? 0 : (L > a.S1 ? a.S1 : L);
      if (s0 + L > a.T1) L = a.T1 - s0 < 0 ? 0 : a.T1 - s0;
      if (a.used_q) {
        const long long us = a.used_q[s];
        L = us < 0 ? 0 : (us < L ? us : L);
      }
      return (L + 127) / 128 * (128 / RPI) * a.N1;
    };
    cnt0 = count(lane);
    cnt1 = count(lane + 32);
    incl0 = cnt0;
    incl1 = cnt1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v0 = __shfl_up_sync(0xffffffffu, incl0, o), v1 = __shfl_up_sync(0xffffffffu, incl1, o);
      if (lane >= o) {
        incl0 += v0;
        incl1 += v1;
      }
    }
    incl1 += __shfl_sync(0xffffffffu, incl0, 31);
    ngroups = __shfl_sync(0xffffffffu, incl1, 31);
  }
  for (long long grp = gwarp; grp < ngroups; grp += nwarp) {
    int b, n1;
    long long i0;
    const int ipb = a.S1p / RPI;  // iterations per (b, n1)
    if (compact) {
      // the sequences that end at or before grp
      b = __popc(__ballot_sync(0xffffffffu, incl0 <= grp)) + __popc(__ballot_sync(0xffffffffu, incl1 <= grp));
      const int src = b & 31;
      const long long ib = b < 32 ? __shfl_sync(0xffffffffu, incl0, src) : __shfl_sync(0xffffffffu, incl1, src);
      const long long cb = b < 32 ? __shfl_sync(0xffffffffu, cnt0, src) : __shfl_sync(0xffffffffu, cnt1, src);
      const long long local = grp - (ib - cb);
      n1 = (int)(local % a.N1);
      i0 = (local / a.N1) * RPI;
    } else if (SMALL) {
      const uint32_t g32 = (uint32_t)grp, N1 = (uint32_t)a.N1;
      const uint32_t t = g32 / N1;
      n1 = (int)(g32 - t * N1);
      const uint32_t bb = t / (uint32_t)ipb;
      b = (int)bb;
      i0 = (long long)(t - bb * (uint32_t)ipb) * RPI;
    } else {
      n1 = (int)(grp % a.N1);
      const long long t = grp / a.N1;
      b = (int)(t / ipb);
      i0 = (t % ipb) * RPI;
    }
    const long long base = ((long long)b * a.N1 + n1) * a.S1p + i0;  // first lse2 / sfmg row
    long long q0 = 0, L1 = a.S1;
    if (tnd) {
      q0 = a.cu_q[b];
      L1 = (long long)a.cu_q[b + 1] - q0;
      if (q0 < 0 || q0 > a.T1) L1 = 0;                 // bad cu_seqlens: touch nothing
      L1 = L1 < 0 ? 0 : (L1 > a.S1 ? a.S1 : L1);
      if (q0 + L1 > a.T1) L1 = a.T1 - q0 < 0 ? 0 : a.T1 - q0;
    }
    if (a.used_q) {  // rows past seqused are padding: lse2 = +inf, sfmg = 0
      const long long us = a.used_q[b];
      L1 = us < 0 ? 0 : (us < L1 ? us : L1);
    }
    // rows past the sequence's last 128-row block are never read by the backward kernels
    if (tnd && i0 >= ((L1 + 127) / 128) * 128) continue;
    const long long r0 = row_index(a.layout, b, q0 + i0, n1, a.N1, a.S1);
    const long long li0 = tnd ? (long long)n1 * a.T1 + q0 + i0 : ((long long)b * a.N1 + n1) * a.S1 + i0;
    uint4 x[UN][CPL], y[UN][CPL];
    float l[UN];
    bool val[UN];
#pragma unroll
    for (int u = 0; u < UN; ++u) {
      const int di = u * RPW + sub;  // this lane group's row: i0 + di
      val[u] = i0 + di < L1;
#pragma unroll
      for (int k = 0; k < CPL; ++k) x[u][k] = y[u][k] = make_uint4(0u, 0u, 0u, 0u);
      l[u] = 0.f;
      if (val[u]) {
        const long long r = r0 + di * rstep;
#pragma unroll
        for (int k = 0; k < CPL; ++k) {
          const int col = (k * LPR + part) * 8;
          if (col < a.Dv) {
            x[u][k] = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.dout) + r * a.Dv + col);
            y[u][k] = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.attn_out) + r * a.Dv + col);
          }
        }
        if (part == 0) {
          const long long li = li0 + di;
          if (a.smax) {
            // (row maximum, row sum of exp(S - max)) -> lse; no visible key (sum <= 0) -> +inf
            const float m = a.smax[li * a.stat_stride], sm = a.ssum[li * a.stat_stride];
            l[u] = sm > 0.f ? m + logf(sm) : INFINITY;
          } else {
            l[u] = a.lse[li];
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < UN; ++u) {
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        const uint32_t xs[4] = {x[u][k].x, x[u][k].y, x[u][k].z, x[u][k].w};
        const uint32_t ys[4] = {y[u][k].x, y[u][k].y, y[u][k].z, y[u][k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 xf = unpack2<FP16>(xs[e]), yf = unpack2<FP16>(ys[e]);
          acc = fmaf(xf.x, yf.x, acc);
          acc = fmaf(xf.y, yf.y, acc);
        }
      }
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (part == 0) {
        const long long o = base + u * RPW + sub;
        a.lse2[o] = val[u] ? l[u] * kLog2e : INFINITY;
        a.sfmg[o] = val[u] ? acc : 0.f;
      }
    }
  }

  float4* z = reinterpret_cast<float4*>(a.dq_acc);
  const long long n4 = a.dq_acc_elems / 4;
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n4; x += (long long)gridDim.x * blockDim.x)
    z[x] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Sequence s holding global token t: the last s with cu[s] <= t (cu non-decreasing from 0).
__device__ __forceinline__ int seq_of(const int* cu, int B, long long t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cu[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// One thread per (row, head) of the q side, then of the kv side; a row past its sequence's
// seqused gets its output row written (see UnusedArgs).  Rows are located like the main kernels
// do; with inconsistent cu_seqlens or seqused nothing is written (the preprocess reports it).
__global__ void __launch_bounds__(256) unused_rows_kernel(UnusedArgs a) {
  const bool tnd = a.layout == kTND;
  const long long rq = tnd ? a.T1 : (long long)a.B * a.S1, rk = tnd ? a.T2 : (long long)a.B * a.S2;
  const long long nq = a.used_q ? rq * a.N1 : 0, nk = a.used_kv && !a.fwd ? rk * a.N2 : 0;
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < nq + nk;
       x += (long long)gridDim.x * blockDim.x) {
    const bool qside = x < nq;
    const long long u = qside ? x : x - nq;
    const int N = qside ? a.N1 : a.N2;
    const long long S = qside ? a.S1 : a.S2;
    const int* cu = qside ? a.cu_q : a.cu_kv;
    const int* used = qside ? a.used_q : a.used_kv;
    int b, n;
    long long i, t;
    if (a.layout == kBNSD) {
      i = u % S;
      n = (int)((u / S) % N);
      b = (int)(u / (S * N));
    } else {
      n = (int)(u % N);
      t = u / N;
      b = tnd ? seq_of(cu, a.B, t) : (int)(t / S);
      i = tnd ? t - cu[b] : t % S;
    }
    const long long span = tnd ? (long long)cu[b + 1] - cu[b] : S;
    const int us = used[b];
    if (i < 0 || i >= span || us < 0 || us > span || i < us) continue;
    const long long r = row_index(a.layout, b, tnd ? cu[b] + i : i, n, N, S);
    if (qside) {
      const int dim = a.fwd ? a.Dv : a.D;
      uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dq) + r * dim);
      for (int c = 0; c < dim / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
      if (a.fwd) a.lse_out[tnd ? (long long)n * a.T1 + cu[b] + i : ((long long)b * a.N1 + n) * a.S1 + i] = INFINITY;
    } else {
      uint4* k = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dk) + r * a.D);
      uint4* v = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dv) + r * a.Dv);
      for (int c = 0; c < a.D / 8; ++c) k[c] = make_uint4(0u, 0u, 0u, 0u);
      for (int c = 0; c < a.Dv / 8; ++c) v[c] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

template <bool FP16>
__global__ void __launch_bounds__(256) convert_kernel(ConvArgs a) {
  const long long n8 = a.elems / 8;
  const float4* src = reinterpret_cast<const float4*>(a.dq_acc);
  uint4* dst = reinterpret_cast<uint4*>(a.dq);
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n8; x += (long long)gridDim.x * blockDim.x) {
    const float4 u = __ldcs(src + 2 * x), v = __ldcs(src + 2 * x + 1);
    uint4 o;
    o.x = pack2<FP16>(u.x * a.scale, u.y * a.scale);
    o.y = pack2<FP16>(u.z * a.scale, u.w * a.scale);
    o.z = pack2<FP16>(v.x * a.scale, v.y * a.scale);
    o.w = pack2<FP16>(v.z * a.scale, v.w * a.scale);
    dst[x] = o;
  }
}

__global__ void __launch_bounds__(256) zero_kernel(uint4* p, long long n16) {
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n16; x += (long long)gridDim.x * blockDim.x)
    p[x] = make_uint4(0u, 0u, 0u, 0u);
}

__global__ void __launch_bounds__(256) fill_f32_kernel(float* p, long long n, float v) {
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long long)gridDim.x * blockDim.x)
    p[x] = v;
}

__global__ void __launch_bounds__(256) fill_lse_sinks_kernel(float* lse, const float* sinks, long long S, int N1,
                                                              long long n, bool tnd) {
  for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long long)gridDim.x * blockDim.x)
    lse[x] = sinks[tnd ? x / S : (x / S) % N1];
}

int grid_for(long long work_items, int per_block) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long want = (work_items + per_block - 1) / per_block;
  long long cap = (long long)sms * 8;
  if (want > cap) want = cap;
  if (want < 1) want = 1;
  return (int)want;
}

}  // namespace

cudaError_t kernel_binary_version(int* version) {
  cudaFuncAttributes at;
  const cudaError_t e = cudaFuncGetAttributes(&at, zero_kernel);
  if (e == cudaSuccess) *version = at.binaryVersion;
  return e;
}

cudaError_t launch_zero(void* p, long long bytes, cudaStream_t st) {
  if (bytes <= 0) return cudaSuccess;
  const long long n16 = bytes / 16;
  zero_kernel<<<grid_for(n16, 256), 256, 0, st>>>(static_cast<uint4*>(p), n16);
  return cudaGetLastError();
}

cudaError_t launch_fill_f32(float* p, long long n, float v, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  fill_f32_kernel<<<grid_for(n, 256), 256, 0, st>>>(p, n, v);
  return cudaGetLastError();
}

cudaError_t launch_fill_lse_sinks(float* lse, const float* sinks, long long S, int N1, long long n, bool tnd,
                                  cudaStream_t st) {
  if (n <= 0 || S <= 0) return cudaSuccess;
  fill_lse_sinks_kernel<<<grid_for(n, 256), 256, 0, st>>>(lse, sinks, S, N1, n, tnd);
  return cudaGetLastError();
}

cudaError_t launch_preprocess(const PreArgs& a, bool fp16, cudaStream_t st) {
  const long long rows = (long long)a.B * a.N1 * a.S1p;
  const int dv = pad_dim(a.Dv);
  const long long lanes = rows * (dv == 192 ? 8 : dv / 8);
  const long long work = lanes > a.dq_acc_elems / 4 ? lanes : a.dq_acc_elems / 4;
  const bool small = rows < (1ll << 31);
  const int grid = grid_for(work, 256);
  if (a.Dv % 8 != 0 || a.Dv > 192) return cudaErrorInvalidValue;
  auto go = [&](auto fp16_c, auto dv_c) {
    constexpr bool F = decltype(fp16_c)::value;
    constexpr int V = decltype(dv_c)::value;
    if (small) preprocess_kernel<F, V, true><<<grid, 256, 0, st>>>(a);
    else preprocess_kernel<F, V, false><<<grid, 256, 0, st>>>(a);
  };
  using T = std::true_type;
  using Fa = std::false_type;
  if (dv == 64) fp16 ? go(T{}, std::integral_constant<int, 64>{}) : go(Fa{}, std::integral_constant<int, 64>{});
  else if (dv == 128) fp16 ? go(T{}, std::integral_constant<int, 128>{}) : go(Fa{}, std::integral_constant<int, 128>{});
  else fp16 ? go(T{}, std::integral_constant<int, 192>{}) : go(Fa{}, std::integral_constant<int, 192>{});
  return cudaGetLastError();
}

cudaError_t launch_unused_rows(const UnusedArgs& a, cudaStream_t st) {
  const bool tnd = a.layout == kTND;
  const long long rq = tnd ? a.T1 : (long long)a.B * a.S1, rk = tnd ? a.T2 : (long long)a.B * a.S2;
  const long long n = (a.used_q ? rq * a.N1 : 0) + (a.used_kv && !a.fwd ? rk * a.N2 : 0);
  if (n <= 0) return cudaSuccess;
  unused_rows_kernel<<<grid_for(n, 256), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_convert(const ConvArgs& a, bool fp16, cudaStream_t st) {
  if (a.elems <= 0) return cudaSuccess;
  const int grid = grid_for(a.elems / 8, 256);
  if (fp16) convert_kernel<true><<<grid, 256, 0, st>>>(a);
  else convert_kernel<false><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace fabwd
