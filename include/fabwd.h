/*
 * libfabwd — FlashAttention backward pass for NVIDIA GB300 (sm_103a). C ABI.
 *
 * [FAG] below is the page "CANN ops-transformer FlashAttnGrad 算子详解" (discosf.com/news/4863418).
 * The operation is the one [FAG] defines in §一 (equations), §二 (inputs/outputs/attributes), §4.2 (argument
 * list) and §4.6 (constraints).  Per head, with q-head n1 reading kv-head n2 = n1 / (N1/N2):
 *
 *   S = scale · Q Kᵀ,  P = exp(S − softmax_lse) on visible pairs (0 elsewhere)
 *   dV = Pᵀ dY,  dP = dY Vᵀ,  sfmg = rowsum(dY ⊙ Y),  dS = P ⊙ (dP − sfmg)
 *   dQ = scale · dS K,  dK = scale · dSᵀ Q          (dK, dV summed over the G q-heads of n2)
 *
 * where Y = attn_out and dY = dout, and scale = softmax_scale, or 1/sqrt(D) when it is 0.
 *
 * Use is two-phase, after the aclnn two-step workspace convention on the page
 * "CANN Floyd注意力梯度算子" (jsqmd.com/news/783980), §函数原型:
 *   1. fabwd_workspace_size(&p, &bytes)     host only, no CUDA call
 *   2. caller allocates `bytes` of device memory (the workspace) and the outputs dq, dk, dv
 *   3. fabwd_preprocess(&p, ws, bytes, stream)   sfmg + padded lse + dq accumulator zeroing
 *   4. fabwd_run(&p, ws, bytes, stream)          the backward kernel(s): dq, dk, dv
 * Steps 3 and 4 must see the same params and workspace and run on the same stream, in order.
 *
 * Ownership: the caller owns every buffer.  The library allocates nothing, never synchronises
 * (except fabwd_read_device_status, which exists to read a result back), and only enqueues work
 * on the stream it is given.  No entry point is thread-unsafe except that concurrent calls on
 * different streams must not share a workspace.
 *
 * Errors: every argument problem the host can see is reported before anything is enqueued.
 * Problems only the device can see (cu_seqlens that disagree with T1/T2 or the max sequence
 * lengths; a bounded wait inside a kernel that gave up) set bits in a status word inside the
 * workspace, which fabwd_read_device_status returns.  No kernel traps or spins without limit.
 */
#ifndef FABWD_H
#define FABWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (host side).  The numbering follows the null-pointer / invalid-argument /
 * unsupported split of the error table on the page "CANN Floyd注意力梯度算子", §返回值. */
typedef enum {
  FABWD_OK = 0,
  FABWD_ERR_NULLPTR = 1,     /* a required pointer is NULL */
  FABWD_ERR_INVALID = 2,     /* a dtype / shape / layout / mask argument breaks a stated rule */
  FABWD_ERR_UNSUPPORTED = 3, /* valid per the statement, but no kernel is built for it */
  FABWD_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than fabwd_workspace_size */
  FABWD_ERR_CUDA = 5,        /* a CUDA runtime/driver call or kernel launch failed */
  FABWD_ERR_TIMEOUT = 6,     /* device status: a bounded wait inside a kernel gave up */
  FABWD_ERR_DEVICE = 7       /* device status: the kernels found bad cu_seqlens */
} fabwd_status;

/* io dtype of q, k, v, dout, attn_out, dq, dk, dv ([FAG] §4.4: float16 and bfloat16, all one). */
typedef enum { FABWD_BF16 = 0, FABWD_FP16 = 1 } fabwd_dtype;

/* One layout for q/kv/out ([FAG] §4.6).  Shapes (row-major, innermost last):
 *   BSND: q [B,S1,N1,D]  k [B,S2,N2,D]  v [B,S2,N2,Dv]  dout/attn_out [B,S1,N1,Dv]
 *   BNSD: q [B,N1,S1,D]  k [B,N2,S2,D]  v [B,N2,S2,Dv]  dout/attn_out [B,N1,S1,Dv]
 *   TND:  q [T1,N1,D]    k [T2,N2,D]    v [T2,N2,Dv]    dout/attn_out [T1,N1,Dv]
 * softmax_lse (fp32): [B,N1,S1] for BSND/BNSD, [N1,T1] for TND ([FAG] §4.6). */
typedef enum { FABWD_BSND = 0, FABWD_TND = 1, FABWD_BNSD = 2 } fabwd_layout;

/* mask_mode (the enum table of [FAG] §4.3 did not survive; this library's reading):
 *   0 none (the dense preset: windows must both be -1, [FAG] §4.6),
 *   1 causal, bottom-right aligned: key j is visible to query i iff j <= i + (S2 - S1),
 *   2 band.
 * In modes 1 and 2, win_left >= 0 also requires j >= i + (S2 - S1) - win_left and
 * win_right >= 0 requires j <= i + (S2 - S1) + win_right; -1 means unbounded.  The rules
 * intersect.  S1/S2 here are the lengths of the sequence the pair belongs to. */
typedef enum { FABWD_MASK_NONE = 0, FABWD_MASK_CAUSAL = 1, FABWD_MASK_BAND = 2 } fabwd_mask;

/* How dQ is produced.
 *   FABWD_DQ_ATOMIC:   the kv-stationary kernel reduce-adds fp32 dQ partials into the workspace
 *                      and a convert pass casts scale · accumulator (the fp32-workspace dQ of
 *                      [FAG] §5.2's bn2gs1s2 template); summation order varies between runs.
 *   FABWD_DQ_SEPARATE: the kv-stationary kernel produces dK and dV only; a q-stationary kernel
 *                      recomputes S and dP per query block and accumulates dQ in tensor memory,
 *                      without atomics: bitwise reproducible, no fp32 accumulator in the
 *                      workspace, about 1.4x the tensor-core work.
 *   FABWD_DQ_AUTO:     the library's choice (currently SEPARATE, the faster mode on the measured
 *                      workloads). */
typedef enum { FABWD_DQ_AUTO = 0, FABWD_DQ_ATOMIC = 1, FABWD_DQ_SEPARATE = 2 } fabwd_dq_mode;

/* Device status bits (fabwd_read_device_status). */
#define FABWD_DEV_TIMEOUT 0x1u     /* a bounded mbarrier wait gave up; outputs are not valid */
#define FABWD_DEV_BAD_SEQLENS 0x2u /* cu_seqlens not non-decreasing from 0, or beyond T / max, or a
                                      seqused entry outside [0, the sequence's length] */
#define FABWD_DEV_INTERNAL 0x4u    /* a kernel found its shared memory misaligned; nothing computed */

typedef struct {
  int32_t dtype;   /* fabwd_dtype */
  int32_t layout;  /* fabwd_layout */
  /* Sizes ([FAG] §一 notation).  BSND/BNSD: S1, S2 are the sequence lengths.  TND: B is the
   * number of sequences, S1/S2 are max_seqlen_q/max_seqlen_kv (upper bounds of every
   * sequence's length) and T1/T2 the total token counts.  S1 = 0 or S2 = 0 (and empty TND
   * sequences) are accepted: no pair is visible, so dq = dk = dv = 0.
   * Head dims: 0 < Dv <= D <= 192 ([FAG] §4.6, else INVALID), and D, Dv multiples of 8 (rows of
   * a multiple of 16 bytes for the TMA tensor maps and the 16-byte row stores; else
   * UNSUPPORTED).  Kernels are built for 64, 128 and 192 ([FAG] §5.1's d_align / dv_align
   * classes); another D or Dv runs in the next larger kernel, which reads zeros past the row's
   * end and writes the row's own elements only.  FABWD_DQ_ATOMIC with both D > 128 and
   * Dv > 128 is UNSUPPORTED (its fused kernel's accumulators leave no tensor memory for the
   * step's products); the separate mode takes every pair. */
  int64_t B, S1, S2, N1, N2, D, Dv;
  int64_t T1, T2;
  /* Inputs: device pointers, io dtype, contiguous in the layout above, 16-byte aligned. */
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  const void* attn_out;
  const float* softmax_lse;      /* device, fp32, natural-log lse of the scaled scores (read by
                                    fabwd_preprocess only; unused by fabwd_preprocess_stats and
                                    the run entry points) */
  const int32_t* cu_seqlens_q;   /* device, B+1 entries, TND only (NULL otherwise) */
  const int32_t* cu_seqlens_kv;  /* device, B+1 entries, TND only (NULL otherwise) */
  double softmax_scale;          /* 0 -> 1/sqrt(D) ([FAG] §一 scale rule) */
  int32_t mask_mode;             /* fabwd_mask */
  int32_t dq_mode;               /* fabwd_dq_mode (0 = auto) */
  int64_t win_left, win_right;   /* -1 = unbounded */
  /* Outputs: device pointers, caller-allocated, shapes of q/k/v, io dtype ([FAG] §2.2). */
  void* dq;
  void* dk;
  void* dv;
  /* Optional inputs of [FAG] §2.1 and §4.2; NULL when not given.  The page states no semantics
   * for them; this library's readings:
   *   seqused_q, seqused_kv: device int32, B entries, 4-byte aligned.  Sequence (TND) or batch
   *     row (BSND/BNSD) b takes part with only its first seqused_q[b] query rows and first
   *     seqused_kv[b] key rows, 0 <= seqused <= its length (else FABWD_DEV_BAD_SEQLENS); the
   *     masks align to the used lengths.  The other rows see nothing and are seen by nothing:
   *     their dq / dk / dv rows are written as 0 (fabwd_forward: attn_out 0, softmax_lse +inf).
   *     They are read as parts of 128-row tiles and multiplied by zero, so they must hold finite
   *     values.  Either pointer may be given alone.
   *   sinks: device fp32, N1 entries, 4-byte aligned: one logit per q-head that joins every
   *     row's softmax normaliser with no value vector, lse_i = ln(exp(sinks[n1]) + Σ_j exp(S_ij)).
   *     fabwd_forward includes it in attn_out and softmax_lse.  The backward entry points do not
   *     read it: given that softmax_lse, dq, dk and dv follow §一's formulas unchanged
   *     (rowsum(dY ⊙ Y) still equals Σ_j P_ij dP_ij over the real keys), and the operator has no
   *     sink gradient among its outputs ([FAG] §2.2). */
  const int32_t* seqused_q;
  const int32_t* seqused_kv;
  const float* sinks;
} fabwd_params;

/* Host only.  Validates p (the same checks as fabwd_run, pointers excepted) and returns in
 * *bytes the workspace size fabwd_preprocess/fabwd_run need.  The workspace holds a status
 * word, the fp32 sfmg and log2-scaled lse rows padded per (sequence, q-head) to a multiple of
 * 128, and, in FABWD_DQ_ATOMIC mode only, the fp32 dq accumulator (q's shape with D).  Errors:
 * NULLPTR (p or bytes NULL), INVALID (also when B·N1·roundup(S1, 128) exceeds 2^40 rows, so
 * that no size computation can wrap), UNSUPPORTED (also when ceil(S1/128)·N1 + ceil(S2/128)·N2,
 * the CTAs of one batch's grid row, exceeds 2^31 − 1). */
fabwd_status fabwd_workspace_size(const fabwd_params* p, size_t* bytes);

/* Enqueue on `stream` (a cudaStream_t; NULL = the legacy default stream) the preprocess kernel
 * ([FAG] §5.2 V1 softmaxGradFront): sfmg = rowsum(dout ⊙ attn_out) and lse·log2(e) into the
 * workspace, the dq accumulator set to 0, the device status word cleared and the cu_seqlens
 * checked.  Errors: NULLPTR, INVALID, UNSUPPORTED, WORKSPACE, CUDA (launch failure). */
fabwd_status fabwd_preprocess(const fabwd_params* p, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Enqueue on `stream` the backward proper.  Separate dq mode (the default): ONE grid holding
 * both the kv-stationary CTAs (dK, dV written to dk/dv) and the q-stationary CTAs (dQ written to
 * dq), no atomics, bitwise reproducible.  Atomic dq mode: the kv-stationary kernel (dK, dV, and
 * the dQ partial sums reduce-added into the workspace accumulator) then the convert kernel,
 * dq = cast(scale · accumulator).  Must follow fabwd_preprocess (or fabwd_preprocess_stats) with
 * the same p and workspace on the same stream.  Errors: as fabwd_preprocess.  A TIMEOUT or
 * bad-seqlens condition found on the device shows up in fabwd_read_device_status, not here. */
fabwd_status fabwd_run(const fabwd_params* p, void* workspace, size_t workspace_bytes,
                       void* stream);

/* The two halves of fabwd_run, for callers that schedule or time them separately:
 * fabwd_run_main enqueues the kv-stationary kernel (dk, dv; atomic mode: dQ partials into the
 * workspace accumulator); fabwd_run_dq enqueues the dQ stage (atomic mode: the convert kernel;
 * separate mode: the q-stationary dQ kernel, which needs only the preprocess outputs and may run
 * before, after or beside fabwd_run_main).  The results equal fabwd_run's bit for bit; in
 * separate mode fabwd_run launches the two as one grid instead.
 * Errors: as fabwd_run. */
fabwd_status fabwd_run_main(const fabwd_params* p, void* workspace, size_t workspace_bytes, void* stream);
fabwd_status fabwd_run_dq(const fabwd_params* p, void* workspace, size_t workspace_bytes, void* stream);

/* Synchronising read of the device status word: enqueues a 4-byte device-to-host copy on
 * `stream`, waits for the stream, and stores the FABWD_DEV_* bits in *device_status.  Returns
 * OK when the bits are 0, TIMEOUT when FABWD_DEV_TIMEOUT is set, DEVICE for any other bit,
 * CUDA when the copy or the wait fails, NULLPTR/WORKSPACE for bad arguments. */
fabwd_status fabwd_read_device_status(const void* workspace, size_t workspace_bytes, void* stream,
                                      uint32_t* device_status);

/* Bounded-wait limit in nanoseconds used by the kernels' mbarrier waits (default 2e9).  A value
 * of 0 restores the default.  Returns the previous value.  Process-wide, not thread-safe. */
uint64_t fabwd_set_wait_limit_ns(uint64_t ns);

/* Fault-injection switch for tests of the failure path: when non-zero, the next fabwd_run
 * launches its main kernel so that every CTA first waits on an mbarrier that nothing signals.
 * The wait gives up after the wait limit, the CTA records FABWD_DEV_TIMEOUT, frees its tensor
 * memory and returns.  The switch resets itself after one fabwd_run.  Returns the old value. */
int fabwd_debug_inject_timeout(int on);

/* Host only.  Byte offsets inside the workspace of the fp32 sfmg rows, the fp32 lse·log2(e)
 * rows (both [B][N1][row_stride], row_stride = S1 rounded up to 128; for TND, B counts sequences,
 * rows are sequence-local, and rows past a sequence's length rounded up to 128 are left unwritten)
 * and the fp32 dq accumulator (q's layout with D).  Lets callers inspect the intermediate sfmg
 * (the V1 output of [FAG] §5.2).  Errors as fabwd_workspace_size. */
fabwd_status fabwd_workspace_layout(const fabwd_params* p, size_t* off_sfmg, size_t* off_lse2,
                                    size_t* off_dq_accum, int64_t* row_stride);

/* Forward of [FAG] §一 on the GPU: attn_out Y = P·V and softmax_lse, the two inputs the backward
 * takes from a forward call, with P = exp(S − lse), S = scale·Q·Kᵀ and lse_i = ln Σ_j exp(S_ij)
 * over the keys visible to row i (same masks, GQA map, layouts and scale rule as the backward).
 * p: shapes, q, k, v, cu_seqlens, softmax_scale, mask_mode, win_left, win_right as for the
 * backward; its dout, attn_out, softmax_lse, dq, dk, dv and dq_mode fields are ignored.
 * attn_out: device, io dtype, q's layout with Dv (16-byte aligned); softmax_lse: device fp32,
 * [B][N1][S1] (BSND/BNSD) or [N1][T1] (TND).  Rows with no visible key get Y = 0, lse = +inf.
 * workspace: caller-owned, >= 256 bytes, 256-byte aligned; only its status word is used
 * (fabwd_read_device_status reads it after the call).  Enqueued on `stream`, no allocation, no
 * synchronisation.  Errors as fabwd_run. */
fabwd_status fabwd_forward(const fabwd_params* p, void* attn_out, float* softmax_lse, void* workspace,
                           size_t workspace_bytes, void* stream);

/* fabwd_preprocess for callers that saved the forward's softmax statistics as a per-row maximum
 * and a per-row sum of exp(S - max) (the (softmaxMax, softmaxSum) pair of the pages
 * "LaserAttentionGrad" and "aclnnFusedFloydAttentionGrad", their forward-statistics inputs)
 * instead of softmax_lse: it uses lse = max + ln(sum) per row and is otherwise the same call.
 * softmax_max and softmax_sum: device fp32 in softmax_lse's row layout ([B][N1][S1], or [N1][T1]
 * for TND), each row's value stored stat_stride times in a row (1 for a plain layout; those pages'
 * layout repeats it 8 times), 4-byte aligned; p->softmax_lse is ignored.  A row whose sum is
 * <= 0 (it saw no key) gets lse = +inf, so its P is 0.  Errors: NULLPTR for a missing statistic
 * when there are query rows, INVALID for stat_stride outside [1, 1024] or a misaligned pointer,
 * otherwise as fabwd_preprocess. */
fabwd_status fabwd_preprocess_stats(const fabwd_params* p, const float* softmax_max, const float* softmax_sum,
                                    int64_t stat_stride, void* workspace, size_t workspace_bytes, void* stream);

/* Host only.  Stores in *mode the dQ mode that fabwd_run uses for these parameters: the
 * requested one, or the library's choice (FABWD_DQ_ATOMIC or FABWD_DQ_SEPARATE) for
 * FABWD_DQ_AUTO.  Errors as fabwd_workspace_size. */
fabwd_status fabwd_resolve_dq_mode(const fabwd_params* p, int32_t* mode);

/* Size of the scratch array behind fabwd_run_static_workspace: 64 MiB on every GPU that loads the
 * library.  A problem fits when its fabwd_workspace_size is at most this. */
#define FABWD_STATIC_WORKSPACE_BYTES ((size_t)64 << 20)

/* Allocation-free form of fabwd_preprocess + fabwd_run (the pages have no counterpart; it is a
 * convenience of this library).  For callers that cannot call cudaMalloc when they run the
 * backward: code under a host framework that owns all device memory through its own pool (a
 * foreign allocation can fail or fragment it), or a loop whose rules forbid allocation after
 * start-up.  The caller still allocates and passes the inputs and the outputs dq, dk, dv; the
 * scratch lives in a fixed FABWD_STATIC_WORKSPACE_BYTES array inside the library (held on every
 * GPU that loads the library until the process exits).  A problem whose fabwd_workspace_size
 * exceeds it is refused with FABWD_ERR_WORKSPACE before anything is enqueued; other argument
 * errors as fabwd_run.  Nothing is allocated: no cudaMalloc or cudaFree is called.  The first
 * call on each device looks up the array's device address (cudaGetSymbolAddress, which may load
 * the module) and caches it; make that first call before any stream capture.  Every call on a
 * device shares the one array, which keeps the last call's contents (the kernels clear what must
 * start at zero): calls whose work overlaps on the GPU (other streams, other threads) race and
 * must be serialised by the caller.  The device-side status (FABWD_DEV_*) of the last call is
 * read with fabwd_static_workspace_status. */
fabwd_status fabwd_run_static_workspace(const fabwd_params* p, void* stream);

/* Host only: FABWD_STATIC_WORKSPACE_BYTES, the capacity of fabwd_run_static_workspace's array. */
size_t fabwd_static_workspace_capacity(void);

/* fabwd_read_device_status for fabwd_run_static_workspace: a synchronising read, on `stream`, of
 * the status word the last such call on the current device left in the library's array (bad
 * cu_seqlens, a bounded wait that gave up).  Returns as fabwd_read_device_status; CUDA when the
 * array's address cannot be looked up. */
fabwd_status fabwd_static_workspace_status(void* stream, uint32_t* device_status);

/* Static description of a status code. */
const char* fabwd_status_string(fabwd_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int fabwd_version(void);

/* Diagnostic: the binary architecture of the library's kernels as the CUDA runtime loaded them on
 * the current device (cudaFuncGetAttributes' binaryVersion, major * 10 + minor: 103 for the
 * sm_103a build).  Errors: NULLPTR, CUDA (no device, or no kernel image for it). */
fabwd_status fabwd_kernel_binary_version(int32_t* version);

#ifdef __cplusplus
}
#endif

#endif /* FABWD_H */
