// Internal kernel arguments and launchers shared by the libfabwd translation units.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fabwd {

// Raises the dynamic shared-memory limit of `Kernel` to `bytes` on the current device.  The
// attribute belongs to a (function, device) pair, so it is set once per device: devices 0-63
// are remembered in a bit mask, others get it before every launch.  Host threads may race here;
// both then set the same value, which is harmless.
template <auto Kernel>
cudaError_t ensure_smem_limit(int bytes) {
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

constexpr int kBlockKV = 128;  // kv rows per CTA of the main kernel (M of the kv-side MMAs)
constexpr int kBlockQ = 64;    // q rows per main-loop step (N of S^T / dP^T / dQ^T)
constexpr int kRowPad = 128;   // padding of the per-(sequence, q-head) lse2 / sfmg rows
constexpr int kDqBlockQ = 128; // q rows per CTA of the q-stationary dQ kernel
// Head dims are built as 64, 128 and 192; any other D (or Dv), a multiple of 8, runs in the next
// larger kernel: its TMA boxes read zeros past the row's last element, which add nothing to any
// product, and the epilogues write the row's own elements only.
constexpr int pad_dim(int d) { return d <= 64 ? 64 : d <= 128 ? 128 : 192; }
// keys per step of the q-stationary dQ kernel: 96 at D = 192, where the dQ accumulator leaves
// 320 TMEM columns for the two S buffers and dP; 64 when Dv = 192 as well (the 48 KB dO tile
// leaves shared memory for three 24 KB K stages and two V stages only)
constexpr int dq_block_kv(int D, int DV) { return D > 128 ? (DV > 128 ? 64 : 96) : 128; }

enum Layout : int { kBSND = 0, kTND = 1, kBNSD = 2 };

// Varlen (TND) grids of up to kFlatMaxSeqs sequences run over the sequences' own work units back
// to back instead of B times the units of the longest sequence.  Each CTA finds its unit with a
// warp scan of the cu_seqlens spans, 32 sequences per pass, each pass about one cu_seqlens
// load latency (what an empty CTA of the B-by-units grid costs): kept to two passes, more
// sequences keep that grid.
constexpr int kFlatMaxSeqs = 64;
inline bool flat_grid(int layout, long long B) { return layout == kTND && B <= kFlatMaxSeqs; }
// Upper bound of sum over sequences of ceil(L_b / blk) for B sequences of at most S rows and T
// rows in all: each term is at most (L_b + blk - 1) / blk and at most ceil(S / blk).
inline long long tnd_blocks_bound(long long B, long long S, long long T, int blk) {
  const long long by_max = B * ((S + blk - 1) / blk), by_total = (T + (long long)(blk - 1) * B) / blk;
  return by_max < by_total ? by_max : by_total;
}

// Element offset of row `row` (sequence-local for BSND/BNSD, global token index for TND) of
// head n in a [B,S,N,dim] / [T,N,dim] / [B,N,S,dim] tensor, in units of `dim`-element rows.
__host__ __device__ __forceinline__ long long row_index(int layout, int b, long long row, int n, int N,
                                                        long long S) {
  if (layout == kBSND) return ((long long)b * S + row) * N + n;
  if (layout == kBNSD) return ((long long)b * N + n) * S + row;
  return row * N + n;
}

struct PreArgs {
  int layout, B, N1, D, Dv;
  long long S1, S2, T1, T2;  // S1/S2: sequence lengths (BSND/BNSD) or max_seqlen (TND)
  int S1p;                   // padded row count per (sequence, q-head)
  const void* dout;
  const void* attn_out;
  const float* lse;
  const float* smax;         // non-null: lse = smax + ln(ssum) per row, read at stride stat_stride
  const float* ssum;
  long long stat_stride;
  const int* cu_q;
  const int* cu_kv;
  const int* used_q;         // seqused_q / seqused_kv (B entries) or null
  const int* used_kv;
  float* lse2;               // [B][N1][S1p]: lse * log2(e), +inf on padding rows
  float* sfmg;               // [B][N1][S1p]: rowsum(dout * attn_out), 0 on padding rows
  float* dq_acc;             // fp32, q's shape with D
  long long dq_acc_elems;
  unsigned* status;
};

struct ConvArgs {
  const float* dq_acc;
  void* dq;
  long long elems;
  float scale;
};

struct MainArgs {
  int layout, B, N1, N2, G;
  int io_d, io_dv;           // head dims of the io tensors: their row lengths (the kernel's
                             // template dims are these rounded up by pad_dim)
  int S1, S2;                // sequence lengths (BSND/BNSD) or max_seqlen (TND)
  long long T1, T2;
  const int* cu_q;
  const int* cu_kv;
  const int* used_q;         // seqused_q / seqused_kv (B entries) or null: used rows per sequence
  const int* used_kv;
  const float* sinks;        // forward only: per-q-head sink logits or null
  int mask_mode, win_left, win_right;
  float scale, scale_log2;   // scale and scale * log2(e)
  int S1p;
  const float* lse2;
  const float* sfmg;
  float* dq_acc;              // fp32 accumulator (atomic dQ mode), else null
  void* dq;                   // io-dtype dq (written by the q-stationary dQ kernel); attn_out for the forward
  float* lse_out;             // forward only: softmax_lse output
  void* dk;
  void* dv;
  unsigned* status;
  unsigned long long wait_ns;
  int inject_timeout;
};

// Rows outside every sequence's used rows (seqused): their output rows are set here.  Backward:
// dq rows (D elements) and dk / dv rows (D / Dv) to 0.  Forward (fwd = true): attn_out rows
// (held in dq, Dv elements) to 0 and their lse entries to +inf.
struct UnusedArgs {
  int layout, B, N1, N2, D, Dv;
  long long S1, S2, T1, T2;
  const int* cu_q;
  const int* cu_kv;
  const int* used_q;
  const int* used_kv;
  void* dq;
  void* dk;
  void* dv;
  float* lse_out;
  bool fwd;
};

struct MainMaps {
  CUtensorMap q, k, v, dout;
  CUtensorMap dq, dk, dv;  // outputs: dq with q's box, dk and dv with k's (TMA-stored epilogues)
};

cudaError_t launch_preprocess(const PreArgs& a, bool fp16, cudaStream_t st);
cudaError_t launch_convert(const ConvArgs& a, bool fp16, cudaStream_t st);
// Writes the output rows of UnusedArgs; nothing when neither seqused pointer is given.
cudaError_t launch_unused_rows(const UnusedArgs& a, cudaStream_t st);
// Zero `bytes` (a multiple of 16) at a 16-byte-aligned device address.
cudaError_t launch_zero(void* p, long long bytes, cudaStream_t st);
// Set n fp32 values to v.
cudaError_t launch_fill_f32(float* p, long long n, float v, cudaStream_t st);
// Set the n entries of an lse array ([B][N1][S] or, tnd, [N1][S]) to their q-head's sink logit.
cudaError_t launch_fill_lse_sinks(float* lse, const float* sinks, long long S, int N1, long long n, bool tnd,
                                  cudaStream_t st);
// Kernel launchers, one explicit instantiation per io dtype (FP16: fp16, else bf16), each in its
// own translation unit.  D and Dv are kernel dims (pad_dim of the io dims); a launcher returns
// cudaErrorInvalidValue when no kernel is built for them.
// The fused kv-stationary kernel of the atomic dQ mode: dK, dV and the fp32 dQ accumulator.
template <bool FP16>
cudaError_t launch_main(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, cudaStream_t st);
// The dK/dV kernel of the separate dQ mode; q-side maps with 128-row boxes up to D = 128 and
// 64-row boxes at D = 192, kv-side maps with 128-row boxes.
template <bool FP16>
cudaError_t launch_kv(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, cudaStream_t st);
// The q-stationary dQ kernel; q-side maps with 128-row boxes, kv-side with dq_block_kv(D, Dv).
template <bool FP16>
cudaError_t launch_dq(const MainArgs& a, const MainMaps& m, int D, int Dv, cudaStream_t st);
// Both separate-mode kernels in one launch (dK/dV CTAs, then dQ CTAs); D <= 128, maps with
// 128-row boxes on both sides.
template <bool FP16>
cudaError_t launch_bwd(const MainArgs& a, const MainMaps& m, int D, int Dv, int n_kv_blocks, cudaStream_t st);
// The same for D = 192: mkv are the dK/dV CTAs' maps (64-row query, 128-row key boxes), mdq the
// dQ CTAs' (128-row query boxes, dq_block_kv(D, Dv)-row key boxes).
template <bool FP16>
cudaError_t launch_bwd_wide(const MainArgs& a, const MainMaps& mkv, const MainMaps& mdq, int D, int Dv,
                            int n_kv_blocks, cudaStream_t st);
// Forward kernel (attn_out and softmax_lse); a.dq is attn_out, a.lse_out the lse rows, a.status the
// status word.  Maps: q with 128-row boxes, k and v with 128-row (D <= 128) or 64-row boxes.
template <bool FP16>
cudaError_t launch_fwd(const MainArgs& a, const MainMaps& m, int D, int Dv, cudaStream_t st);
// A kernel exists for (D, Dv) (before rounding by pad_dim); atomic: the fused dQ-reducing kernel,
// whose TMEM plan leaves no room for Dv > 128 beside a dK of more than 128 columns.
bool dims_supported(int D, int Dv, bool atomic);
// binaryVersion (major * 10 + minor) of the library's kernels as loaded on the current device.
cudaError_t kernel_binary_version(int* version);

}  // namespace fabwd
