// libfabwd host side: argument validation, workspace planning, TMA descriptors and launches.
// The argument rules are those of the page "CANN ops-transformer FlashAttnGrad 算子详解"
// (discosf.com/news/4863418), §4.6 constraints; the two-phase workspace protocol follows the
// page "CANN Floyd注意力梯度算子" (jsqmd.com/news/783980), §函数原型.
#include "../../include/fabwd.h"
#include "fabwd_internal.cuh"

#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

namespace {

using namespace fabwd;

uint64_t g_wait_ns = 2000000000ull;
int g_inject_timeout = 0;

struct Plan {
  bool separate = false;   // dQ by the q-stationary kernel (no fp32 accumulator, no atomics)
  long long S1p = 0;       // padded rows per (sequence, q-head)
  long long rowsQ = 0;     // q rows over all batches/sequences
  long long rowsK = 0;
  size_t off_status = 0, off_lse2 = 0, off_sfmg = 0, off_dqacc = 0, total = 0;
  double scale = 0.0;
  long long dq_elems = 0;
};

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fabwd_status plan_and_check(const fabwd_params* p, Plan* pl, bool check_ptrs) {
  if (!p) return FABWD_ERR_NULLPTR;
  if (p->dtype != FABWD_BF16 && p->dtype != FABWD_FP16) return FABWD_ERR_INVALID;
  if (p->layout != FABWD_BSND && p->layout != FABWD_TND && p->layout != FABWD_BNSD) return FABWD_ERR_INVALID;
  if (p->mask_mode < 0 || p->mask_mode > 2) return FABWD_ERR_INVALID;
  // [FAG] §4.6: B in (0, 65536); N1 a multiple of N2; 0 < Dv <= D <= 192
  if (p->B <= 0 || p->B >= 65536) return FABWD_ERR_INVALID;
  if (p->N1 <= 0 || p->N2 <= 0 || p->N1 % p->N2 != 0) return FABWD_ERR_INVALID;
  if (p->D <= 0 || p->Dv <= 0 || p->Dv > p->D || p->D > 192) return FABWD_ERR_INVALID;
  if (p->S1 < 0 || p->S2 < 0 || p->S1 >= (1ll << 30) || p->S2 >= (1ll << 30)) return FABWD_ERR_INVALID;
  if (p->N1 > 65535 || p->N2 > 65535) return FABWD_ERR_INVALID;
  // windows: -1 = unbounded; the dense preset (mode 0) takes none ([FAG] §4.6)
  if (p->win_left < -1 || p->win_right < -1 || p->win_left >= (1ll << 30) || p->win_right >= (1ll << 30))
    return FABWD_ERR_INVALID;
  if (p->mask_mode == FABWD_MASK_NONE && (p->win_left >= 0 || p->win_right >= 0)) return FABWD_ERR_INVALID;
  if (!(p->softmax_scale == p->softmax_scale) || std::isinf(p->softmax_scale)) return FABWD_ERR_INVALID;
  if (p->dq_mode != FABWD_DQ_AUTO && p->dq_mode != FABWD_DQ_ATOMIC && p->dq_mode != FABWD_DQ_SEPARATE)
    return FABWD_ERR_INVALID;
  // TND requires cu_seqlens; the other layouts forbid them ([FAG] §4.6)
  const bool tnd = p->layout == FABWD_TND;
  if (tnd) {
    if (!p->cu_seqlens_q || !p->cu_seqlens_kv) return FABWD_ERR_INVALID;
    if (p->T1 < 0 || p->T2 < 0 || p->T1 >= (1ll << 31) || p->T2 >= (1ll << 31)) return FABWD_ERR_INVALID;
    if ((p->T1 > 0 && p->S1 == 0) || (p->T2 > 0 && p->S2 == 0)) return FABWD_ERR_INVALID;
  } else {
    if (p->cu_seqlens_q || p->cu_seqlens_kv) return FABWD_ERR_INVALID;
    if (p->B * p->S1 >= (1ll << 31) || p->B * p->S2 >= (1ll << 31)) return FABWD_ERR_INVALID;
  }
  if (!dims_supported((int)p->D, (int)p->Dv, p->dq_mode == FABWD_DQ_ATOMIC)) return FABWD_ERR_UNSUPPORTED;
  // The workspace holds B·N1·roundup(S1, 128) fp32 rows twice.  With TND, B, N1 and the
  // max_seqlen_q bound S1 are limited only one by one, so the product could wrap size_t;
  // refuse more than 2^40 rows (4 TiB each) before any size is computed.
  {
    const long long s1p = (p->S1 + kRowPad - 1) / kRowPad * kRowPad;
    if (s1p > 0 && (p->B * p->N1 > (1ll << 40) / s1p)) return FABWD_ERR_INVALID;
  }
  // Each batch is one grid row of 128-row query blocks over N1 heads plus 128-row key blocks
  // over N2 heads; that count must fit a launch's x dimension (and the int the launches use).
  if ((p->S1 + 127) / 128 * p->N1 + (p->S2 + 127) / 128 * p->N2 > 0x7fffffffll) return FABWD_ERR_UNSUPPORTED;
  // Flat varlen grids run over every sequence's units in one x dimension.
  if (flat_grid(p->layout, p->B) && tnd_blocks_bound(p->B, p->S1, p->T1, 128) * p->N1 + tnd_blocks_bound(p->B, p->S2, p->T2, 128) * p->N2 >
                 0x7fffffffll)
    return FABWD_ERR_UNSUPPORTED;

  pl->rowsQ = tnd ? p->T1 : p->B * p->S1;
  pl->rowsK = tnd ? p->T2 : p->B * p->S2;
  pl->S1p = (p->S1 + kRowPad - 1) / kRowPad * kRowPad;
  pl->scale = p->softmax_scale != 0.0 ? p->softmax_scale : 1.0 / std::sqrt((double)p->D);
  // AUTO: the separate pass (measured faster than the fused atomic pass on the GB300 workloads)
  pl->separate = p->dq_mode != FABWD_DQ_ATOMIC;
  pl->dq_elems = pl->separate ? 0 : pl->rowsQ * p->N1 * p->D;
  pl->off_status = 0;
  pl->off_lse2 = 256;
  const size_t rowbytes = round_up((size_t)p->B * p->N1 * pl->S1p * sizeof(float), 256);
  pl->off_sfmg = pl->off_lse2 + rowbytes;
  pl->off_dqacc = pl->off_sfmg + rowbytes;
  pl->total = pl->off_dqacc + round_up((size_t)pl->dq_elems * sizeof(float), 256);

  if (check_ptrs) {
    const bool q_nonempty = pl->rowsQ > 0, k_nonempty = pl->rowsK > 0;
    // attn_out and softmax_lse are read by the preprocess only (which checks softmax_lse itself)
    if (q_nonempty && (!p->q || !p->dout || !p->attn_out || !p->dq)) return FABWD_ERR_NULLPTR;
    if (k_nonempty && (!p->k || !p->v || !p->dk || !p->dv)) return FABWD_ERR_NULLPTR;
    if (q_nonempty && (!aligned16(p->q) || !aligned16(p->dout) || !aligned16(p->attn_out) || !aligned16(p->dq) ||
                       (reinterpret_cast<uintptr_t>(p->softmax_lse) & 3u)))
      return FABWD_ERR_INVALID;
    if (k_nonempty && (!aligned16(p->k) || !aligned16(p->v) || !aligned16(p->dk) || !aligned16(p->dv)))
      return FABWD_ERR_INVALID;
  }
  // the optional inputs: int32 / fp32 device arrays
  if ((reinterpret_cast<uintptr_t>(p->seqused_q) | reinterpret_cast<uintptr_t>(p->seqused_kv) |
       reinterpret_cast<uintptr_t>(p->sinks)) & 3u)
    return FABWD_ERR_INVALID;
  return FABWD_OK;
}

// Output rows past seqused (both entry points set them; the kernels never write them).
cudaError_t unused_rows(const fabwd_params* p, void* dq, float* lse_out, bool fwd, cudaStream_t st) {
  if (!p->seqused_q && (fwd || !p->seqused_kv)) return cudaSuccess;
  UnusedArgs u;
  u.layout = p->layout;
  u.B = (int)p->B;
  u.N1 = (int)p->N1;
  u.N2 = (int)p->N2;
  u.D = (int)p->D;
  u.Dv = (int)p->Dv;
  u.S1 = p->S1;
  u.S2 = p->S2;
  u.T1 = p->T1;
  u.T2 = p->T2;
  u.cu_q = p->cu_seqlens_q;
  u.cu_kv = p->cu_seqlens_kv;
  u.used_q = p->seqused_q;
  u.used_kv = p->seqused_kv;
  u.dq = dq;
  u.dk = p->dk;
  u.dv = p->dv;
  u.lse_out = lse_out;
  u.fwd = fwd;
  return launch_unused_rows(u, st);
}

fabwd_status check_ws(const Plan& pl, const void* ws, size_t ws_bytes) {
  if (!ws || ws_bytes < pl.total) return FABWD_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return FABWD_ERR_WORKSPACE;
  return FABWD_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 4-D map over a q/k/v/dout tensor with a {64, 1, rows, 1} box (BSND, TND) or {64, rows, 1, 1}
// box (BNSD), 128-byte swizzle.  Coordinates: (d, head, row, batch) for BSND/TND and
// (d, row, head, batch) for BNSD; TND is a single batch of T rows.
bool make_map(CUtensorMap* m, const void* base, bool fp16, int layout, long long dim, long long N, long long S,
              long long Bn, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const long long e = 2;
  cuuint64_t gdim[4], gstr[3];
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  if (layout == kBNSD) {
    gdim[0] = dim; gdim[1] = S; gdim[2] = N; gdim[3] = Bn;
    gstr[0] = dim * e; gstr[1] = S * dim * e; gstr[2] = N * S * dim * e;
    box[1] = box_rows;
    box[2] = 1;
  } else {
    gdim[0] = dim; gdim[1] = N; gdim[2] = S; gdim[3] = Bn;
    gstr[0] = dim * e; gstr[1] = N * dim * e; gstr[2] = S * N * dim * e;
  }
  cuuint32_t estr[4] = {1, 1, 1, 1};
  std::memset(m, 0, sizeof(*m));
  CUresult r = enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(base), gdim, gstr, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

namespace fabwd {
bool dims_supported(int D, int Dv, bool atomic) {
  // row strides of D·2 and Dv·2 bytes must be multiples of 16 for the TMA tensor maps and the
  // 16-byte row stores
  if (D % 8 != 0 || Dv % 8 != 0) return false;
  return !(atomic && pad_dim(D) == 192 && pad_dim(Dv) == 192);
}
}  // namespace fabwd

namespace {
fabwd_status preprocess_impl(const fabwd_params* p, const float* smax, const float* ssum, int64_t stat_stride,
                             void* ws, size_t ws_bytes, void* stream);
}  // namespace

extern "C" {

fabwd_status fabwd_workspace_size(const fabwd_params* p, size_t* bytes) {
  if (!p || !bytes) return FABWD_ERR_NULLPTR;
  Plan pl;
  fabwd_status s = plan_and_check(p, &pl, false);
  if (s != FABWD_OK) return s;
  *bytes = pl.total;
  return FABWD_OK;
}

fabwd_status fabwd_workspace_layout(const fabwd_params* p, size_t* off_sfmg, size_t* off_lse2, size_t* off_dq_accum,
                                    int64_t* row_stride) {
  if (!p || !off_sfmg || !off_lse2 || !off_dq_accum || !row_stride) return FABWD_ERR_NULLPTR;
  Plan pl;
  fabwd_status s = plan_and_check(p, &pl, false);
  if (s != FABWD_OK) return s;
  *off_sfmg = pl.off_sfmg;
  *off_lse2 = pl.off_lse2;
  *off_dq_accum = pl.off_dqacc;
  *row_stride = pl.S1p;
  return FABWD_OK;
}

fabwd_status fabwd_resolve_dq_mode(const fabwd_params* p, int32_t* mode) {
  if (!p || !mode) return FABWD_ERR_NULLPTR;
  Plan pl;
  fabwd_status s = plan_and_check(p, &pl, false);
  if (s != FABWD_OK) return s;
  *mode = pl.separate ? FABWD_DQ_SEPARATE : FABWD_DQ_ATOMIC;
  return FABWD_OK;
}

fabwd_status fabwd_preprocess(const fabwd_params* p, void* ws, size_t ws_bytes, void* stream) {
  return preprocess_impl(p, nullptr, nullptr, 0, ws, ws_bytes, stream);
}

fabwd_status fabwd_preprocess_stats(const fabwd_params* p, const float* softmax_max, const float* softmax_sum,
                                    int64_t stat_stride, void* ws, size_t ws_bytes, void* stream) {
  if (!p) return FABWD_ERR_NULLPTR;
  fabwd_params q = *p;
  q.softmax_lse = softmax_max;  // the statistics replace softmax_lse: checked like it
  const bool rows = q.S1 > 0 && q.B > 0 && q.N1 > 0 && (q.layout != FABWD_TND || q.T1 > 0);
  if (rows && (!softmax_max || !softmax_sum)) return FABWD_ERR_NULLPTR;
  if (stat_stride < 1 || stat_stride > 1024 ||
      (rows && (reinterpret_cast<uintptr_t>(softmax_sum) & 3u)))
    return FABWD_ERR_INVALID;
  return preprocess_impl(&q, softmax_max, softmax_sum, stat_stride, ws, ws_bytes, stream);
}

}  // extern "C"

namespace {
fabwd_status preprocess_impl(const fabwd_params* p, const float* smax, const float* ssum, int64_t stat_stride,
                             void* ws, size_t ws_bytes, void* stream) {
  Plan pl;
  fabwd_status s = plan_and_check(p, &pl, true);
  if (s != FABWD_OK) return s;
  if (pl.rowsQ > 0 && !p->softmax_lse) return FABWD_ERR_NULLPTR;
  if ((s = check_ws(pl, ws, ws_bytes)) != FABWD_OK) return s;
  uint8_t* w = static_cast<uint8_t*>(ws);
  PreArgs a;
  a.layout = p->layout;
  a.B = (int)p->B;
  a.N1 = (int)p->N1;
  a.D = (int)p->D;
  a.Dv = (int)p->Dv;
  a.S1 = p->S1;
  a.S2 = p->S2;
  a.T1 = p->T1;
  a.T2 = p->T2;
  a.S1p = (int)pl.S1p;
  a.dout = p->dout;
  a.attn_out = p->attn_out;
  a.lse = p->softmax_lse;
  a.smax = smax;
  a.ssum = ssum;
  a.stat_stride = stat_stride;
  a.cu_q = p->cu_seqlens_q;
  a.cu_kv = p->cu_seqlens_kv;
  a.used_q = p->seqused_q;
  a.used_kv = p->seqused_kv;
  a.lse2 = reinterpret_cast<float*>(w + pl.off_lse2);
  a.sfmg = reinterpret_cast<float*>(w + pl.off_sfmg);
  a.dq_acc = reinterpret_cast<float*>(w + pl.off_dqacc);
  a.dq_acc_elems = pl.dq_elems;
  a.status = reinterpret_cast<unsigned*>(w + pl.off_status);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_preprocess(a, p->dtype == FABWD_FP16, st);
  if (e == cudaSuccess) e = unused_rows(p, p->dq, nullptr, false, st);
  return e == cudaSuccess ? FABWD_OK : FABWD_ERR_CUDA;
}
}  // namespace

namespace {

MainArgs main_args(const fabwd_params* p, const Plan& pl, uint8_t* w, int inject) {
  MainArgs a;
  a.layout = p->layout;
  a.B = (int)p->B;
  a.N1 = (int)p->N1;
  a.N2 = (int)p->N2;
  a.G = (int)(p->N1 / p->N2);
  a.io_d = (int)p->D;
  a.io_dv = (int)p->Dv;
  a.S1 = (int)p->S1;
  a.S2 = (int)p->S2;
  a.T1 = p->T1;
  a.T2 = p->T2;
  a.cu_q = p->cu_seqlens_q;
  a.cu_kv = p->cu_seqlens_kv;
  a.used_q = p->seqused_q;
  a.used_kv = p->seqused_kv;
  a.sinks = nullptr;  // the backward does not read sinks (they are inside softmax_lse)
  a.mask_mode = p->mask_mode;
  a.win_left = (int)p->win_left;
  a.win_right = (int)p->win_right;
  a.scale = (float)pl.scale;
  a.scale_log2 = (float)(pl.scale * 1.4426950408889634);
  a.S1p = (int)pl.S1p;
  a.lse2 = reinterpret_cast<const float*>(w + pl.off_lse2);
  a.sfmg = reinterpret_cast<const float*>(w + pl.off_sfmg);
  a.dq_acc = pl.separate ? nullptr : reinterpret_cast<float*>(w + pl.off_dqacc);
  a.dq = p->dq;
  a.lse_out = nullptr;
  a.dk = p->dk;
  a.dv = p->dv;
  a.status = reinterpret_cast<unsigned*>(w + pl.off_status);
  a.wait_ns = g_wait_ns;
  a.inject_timeout = inject;
  return a;
}

bool any_pair(const fabwd_params* p, const Plan& pl) {
  return pl.rowsQ > 0 && pl.rowsK > 0 && p->S1 > 0 && p->S2 > 0;
}

// Tensor maps with the given q-side and kv-side box heights.
bool make_maps(const fabwd_params* p, MainMaps* maps, int q_rows, int kv_rows) {
  const bool fp16 = p->dtype == FABWD_FP16, tnd = p->layout == FABWD_TND;
  const long long Sq = tnd ? p->T1 : p->S1, Sk = tnd ? p->T2 : p->S2, Bn = tnd ? 1 : p->B;
  return make_map(&maps->q, p->q, fp16, p->layout, p->D, p->N1, Sq, Bn, q_rows) &&
         make_map(&maps->dout, p->dout, fp16, p->layout, p->Dv, p->N1, Sq, Bn, q_rows) &&
         make_map(&maps->k, p->k, fp16, p->layout, p->D, p->N2, Sk, Bn, kv_rows) &&
         make_map(&maps->v, p->v, fp16, p->layout, p->Dv, p->N2, Sk, Bn, kv_rows) &&
         make_map(&maps->dq, p->dq, fp16, p->layout, p->D, p->N1, Sq, Bn, q_rows) &&
         make_map(&maps->dk, p->dk, fp16, p->layout, p->D, p->N2, Sk, Bn, kv_rows) &&
         make_map(&maps->dv, p->dv, fp16, p->layout, p->Dv, p->N2, Sk, Bn, kv_rows);
}

}  // namespace

extern "C" {

fabwd_status fabwd_run_main(const fabwd_params* p, void* ws, size_t ws_bytes, void* stream) {
  Plan pl;
  fabwd_status s = plan_and_check(p, &pl, true);
  if (s != FABWD_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != FABWD_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int inject = g_inject_timeout;
  g_inject_timeout = 0;
  if (any_pair(p, pl)) {
    // separate mode: the dK/dV kernel (128-row query steps up to D = 128, 64-row at D = 192);
    // atomic mode: the fused kv-stationary kernel with 64-row steps, which also reduces dQ
    const int D = pad_dim((int)p->D), Dv = pad_dim((int)p->Dv);
    MainMaps maps;
    if (!make_maps(p, &maps, pl.separate && D <= 128 ? 128 : kBlockQ, kBlockKV)) return FABWD_ERR_CUDA;
    const MainArgs a = main_args(p, pl, static_cast<uint8_t*>(ws), inject);
    const int n_kv_blocks = (int)((p->S2 + kBlockKV - 1) / kBlockKV);
    const bool fp16 = p->dtype == FABWD_FP16;
    cudaError_t e = pl.separate ? (fp16 ? launch_kv<true>(a, maps, D, Dv, n_kv_blocks, st)
                                        : launch_kv<false>(a, maps, D, Dv, n_kv_blocks, st))
                                : (fp16 ? launch_main<true>(a, maps, D, Dv, n_kv_blocks, st)
                                        : launch_main<false>(a, maps, D, Dv, n_kv_blocks, st));
    if (e != cudaSuccess) return FABWD_ERR_CUDA;
  } else if (pl.rowsK > 0) {
    // no visible pair at all: dk = dv = 0
    if (launch_zero(p->dk, pl.rowsK * p->N2 * p->D * 2, st) != cudaSuccess ||
        launch_zero(p->dv, pl.rowsK * p->N2 * p->Dv * 2, st) != cudaSuccess)
      return FABWD_ERR_CUDA;
  }
  return FABWD_OK;
}

fabwd_status fabwd_run_dq(const fabwd_params* p, void* ws, size_t ws_bytes, void* stream) {
  Plan pl;
  fabwd_status s = plan_and_check(p, &pl, true);
  if (s != FABWD_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != FABWD_OK) return s;
  uint8_t* w = static_cast<uint8_t*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (!pl.separate) {
    ConvArgs c;
    c.dq_acc = reinterpret_cast<const float*>(w + pl.off_dqacc);
    c.dq = p->dq;
    c.elems = pl.dq_elems;
    c.scale = (float)pl.scale;
    e = launch_convert(c, p->dtype == FABWD_FP16, st);
  } else if (any_pair(p, pl)) {
    MainMaps maps;
    const int D = pad_dim((int)p->D), Dv = pad_dim((int)p->Dv);
    if (!make_maps(p, &maps, kDqBlockQ, dq_block_kv(D, Dv))) return FABWD_ERR_CUDA;
    const MainArgs a = main_args(p, pl, w, 0);
    e = p->dtype == FABWD_FP16 ? launch_dq<true>(a, maps, D, Dv, st) : launch_dq<false>(a, maps, D, Dv, st);
  } else if (pl.rowsQ > 0) {
    e = launch_zero(p->dq, pl.rowsQ * p->N1 * p->D * 2, st);  // no visible pair: dq = 0
  }
  return e == cudaSuccess ? FABWD_OK : FABWD_ERR_CUDA;
}

fabwd_status fabwd_run(const fabwd_params* p, void* ws, size_t ws_bytes, void* stream) {
  Plan pl;
  fabwd_status s = plan_and_check(p, &pl, true);
  if (s != FABWD_OK) return s;
  if ((s = check_ws(pl, ws, ws_bytes)) != FABWD_OK) return s;
  if (pl.separate && any_pair(p, pl)) {
    // separate mode: the dK/dV and dQ CTAs as one grid (one set of tensor maps for D <= 128,
    // one per CTA kind above)
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int inject = g_inject_timeout;
    g_inject_timeout = 0;
    const MainArgs a = main_args(p, pl, static_cast<uint8_t*>(ws), inject);
    const int n_kv_blocks = (int)((p->S2 + kBlockKV - 1) / kBlockKV);
    const bool fp16 = p->dtype == FABWD_FP16;
    const int D = pad_dim((int)p->D), Dv = pad_dim((int)p->Dv);
    cudaError_t e;
    if (D <= 128) {
      MainMaps maps;
      if (!make_maps(p, &maps, 128, kBlockKV)) return FABWD_ERR_CUDA;
      e = fp16 ? launch_bwd<true>(a, maps, D, Dv, n_kv_blocks, st) : launch_bwd<false>(a, maps, D, Dv, n_kv_blocks, st);
    } else {
      MainMaps mkv, mdq;
      if (!make_maps(p, &mkv, kBlockQ, kBlockKV) || !make_maps(p, &mdq, kDqBlockQ, dq_block_kv(D, Dv)))
        return FABWD_ERR_CUDA;
      e = fp16 ? launch_bwd_wide<true>(a, mkv, mdq, D, Dv, n_kv_blocks, st)
               : launch_bwd_wide<false>(a, mkv, mdq, D, Dv, n_kv_blocks, st);
    }
    return e == cudaSuccess ? FABWD_OK : FABWD_ERR_CUDA;
  }
  s = fabwd_run_main(p, ws, ws_bytes, stream);
  if (s != FABWD_OK) return s;
  return fabwd_run_dq(p, ws, ws_bytes, stream);
}

fabwd_status fabwd_forward(const fabwd_params* p, void* attn_out, float* softmax_lse, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!p) return FABWD_ERR_NULLPTR;
  fabwd_params f = *p;  // the backward-only fields are not used: fill them so the shared checks pass
  f.attn_out = attn_out;
  f.softmax_lse = softmax_lse;
  f.dout = attn_out;
  f.dq = attn_out;  // non-null stand-ins: these fields are not read here
  f.dk = const_cast<void*>(f.k);
  f.dv = const_cast<void*>(f.v);
  f.dq_mode = FABWD_DQ_SEPARATE;
  Plan pl;
  fabwd_status s = plan_and_check(&f, &pl, true);
  if (s != FABWD_OK) return s;
  if (pl.rowsQ > 0 && !softmax_lse) return FABWD_ERR_NULLPTR;
  if (!ws) return FABWD_ERR_NULLPTR;
  if (ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u)) return FABWD_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_zero(ws, 256, st) != cudaSuccess) return FABWD_ERR_CUDA;  // status word
  if (pl.rowsQ == 0) return FABWD_OK;
  if (!any_pair(&f, pl)) {  // no key at all: Y = 0, lse = +inf (or the row's sink logit)
    const long long rows = pl.rowsQ * p->N1;
    const bool ok = launch_zero(attn_out, rows * p->Dv * 2, st) == cudaSuccess &&
                    (p->sinks ? launch_fill_lse_sinks(softmax_lse, p->sinks, p->layout == FABWD_TND ? p->T1 : p->S1,
                                                      (int)p->N1, rows, p->layout == FABWD_TND, st)
                              : launch_fill_f32(softmax_lse, rows, INFINITY, st)) == cudaSuccess &&
                    unused_rows(p, attn_out, softmax_lse, true, st) == cudaSuccess;
    return ok ? FABWD_OK : FABWD_ERR_CUDA;
  }
  const int inject = g_inject_timeout;
  g_inject_timeout = 0;
  MainArgs a = main_args(&f, pl, static_cast<uint8_t*>(ws), inject);
  a.status = static_cast<unsigned*>(ws);
  a.dq = attn_out;
  a.lse_out = softmax_lse;
  a.sinks = p->sinks;
  MainMaps maps;
  const int D = pad_dim((int)p->D), Dv = pad_dim((int)p->Dv);
  if (!make_maps(&f, &maps, 128, D > 128 ? 64 : 128)) return FABWD_ERR_CUDA;
  // attn_out is written through the dq map's slot: rows of Dv elements, q's row count and box
  {
    const bool tnd = p->layout == FABWD_TND;
    if (!make_map(&maps.dq, attn_out, p->dtype == FABWD_FP16, p->layout, p->Dv, p->N1, tnd ? p->T1 : p->S1,
                  tnd ? 1 : p->B, 128))
      return FABWD_ERR_CUDA;
  }
  cudaError_t e = p->dtype == FABWD_FP16 ? launch_fwd<true>(a, maps, D, Dv, st) : launch_fwd<false>(a, maps, D, Dv, st);
  if (e == cudaSuccess) e = unused_rows(p, attn_out, softmax_lse, true, st);
  return e == cudaSuccess ? FABWD_OK : FABWD_ERR_CUDA;
}

fabwd_status fabwd_read_device_status(const void* ws, size_t ws_bytes, void* stream, uint32_t* device_status) {
  if (!ws || !device_status) return FABWD_ERR_NULLPTR;
  if (ws_bytes < 256) return FABWD_ERR_WORKSPACE;
  uint32_t v = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return FABWD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FABWD_ERR_CUDA;
  *device_status = v;
  if (v & FABWD_DEV_TIMEOUT) return FABWD_ERR_TIMEOUT;
  if (v) return FABWD_ERR_DEVICE;
  return FABWD_OK;
}

uint64_t fabwd_set_wait_limit_ns(uint64_t ns) {
  const uint64_t old = g_wait_ns;
  g_wait_ns = ns ? ns : 2000000000ull;
  return old;
}

int fabwd_debug_inject_timeout(int on) {
  const int old = g_inject_timeout;
  g_inject_timeout = on ? 1 : 0;
  return old;
}

const char* fabwd_status_string(fabwd_status s) {
  switch (s) {
    case FABWD_OK: return "ok";
    case FABWD_ERR_NULLPTR: return "a required pointer is NULL";
    case FABWD_ERR_INVALID: return "invalid argument (dtype, shape, layout, mask, window or alignment)";
    case FABWD_ERR_UNSUPPORTED: return "valid but unsupported (head dims not multiples of 8, atomic dQ with D and Dv > 128, or too many CTAs)";
    case FABWD_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case FABWD_ERR_CUDA: return "CUDA call or kernel launch failed";
    case FABWD_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up (device status)";
    case FABWD_ERR_DEVICE: return "the kernels found inconsistent cu_seqlens (device status)";
  }
  return "unknown status";
}

int fabwd_version(void) { return 101; }

fabwd_status fabwd_kernel_binary_version(int32_t* version) {
  if (!version) return FABWD_ERR_NULLPTR;
  int v = 0;
  if (kernel_binary_version(&v) != cudaSuccess) return FABWD_ERR_CUDA;
  *version = v;
  return FABWD_OK;
}

}  // extern "C"
