"""fp64 CPU oracle of the FlashAttention backward pass.

TEST INFRASTRUCTURE.  Only the tests, the smoke check of the package entry point and the
bench's CPU-baseline leg may import or run this module.  It shares no code with the CUDA path
(no kernels, headers, helpers or constants) and imports nothing from the package.

What it computes is written out from the definitions on the page
[FAG] = "CANN ops-transformer FlashAttnGrad 算子详解：Flash Attention 反向梯度计算的原理、构建与
Torch 接口实战" (discosf.com/news/4863418):

* §一, forward equations:   S = scale·QKᵀ,  P_ij = exp(S_ij − lse_i),  Y = PV
* §一, scale rule:          softmax_scale ≠ 0 is used as is; 0 means 1/√D
* §一, backward equations:  dV = PᵀdY, dP = dY·Vᵀ, sfmg = rowsum(dY⊙Y), dS = P⊙(dP − sfmg),
                            dQ = scale·dS·K, dK = scale·dSᵀ·Q
* §一, notation:            B, S1, S2, N1, N2, D, Dv, T1, T2; N1 a multiple of N2 (GQA)
* §4.6, layouts:            BSND, BNSD, TND; TND needs cu_seqlens; softmax_lse is fp32 of
                            shape (B, N1, S1) (BSND/BNSD) or (N1, T1) (TND)

Readings where the page is silent (each is listed with its reasoning in the design notes):
* mask_mode 0 = none, 1 = causal, 2 = band; causal is bottom-right aligned (key j is visible
  to query i iff j <= i + S2 − S1); win_left / win_right bound j − i − (S2 − S1) from below
  by −win_left and from above by win_right (−1 = unbounded); the masks intersect.
* a row with no visible key has lse = +inf, P = 0, Y = 0 and dQ = 0; a key seen by no row
  gets dK = dV = 0.
* the GQA head map is q-head n1 -> kv-head n1 // (N1 / N2).
* seqused_q / seqused_kv (the optional int32 inputs of §2.1 and §4.2): sequence b takes part
  with only its first seqused_q[b] query rows and first seqused_kv[b] key rows; the masks are
  aligned to those used lengths; the remaining rows see nothing and are seen by nothing, so
  their lse is +inf, Y = 0 and their gradient rows are 0.
* sinks (the optional fp32 input of §2.1 and §4.2): one logit per q-head that joins every row's
  softmax normaliser and carries no value, lse_i = ln(exp(sink) + Σ_j exp(S_ij)).  It enters
  the forward only; the backward from that lse is §一's unchanged, because sfmg = rowsum(dY⊙Y)
  still equals Σ_j P_ij dP_ij over the real keys.

The backward consumes exactly what the GPU path consumes: Y (attn_out) as given, lse as given
(fp32 values promoted to fp64).  Everything is fp64 numpy; matrix products use numpy matmul as
the library primitive.  There is no tiling, fusion or reordering beyond the definitions.
Each function's parity is pinned by tests that do not re-type its formulas: central finite
differences, a torch fp64 autograd cross-check, closed forms, invariants, GQA == repeated-KV
MHA, TND == per-sequence BSND, and an exact (sympy) golden fixture.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

# ----------------------------------------------------------------------------------------------
# per-head definitions
# ----------------------------------------------------------------------------------------------


def resolve_scale(softmax_scale: float, D: int) -> float:
    """[FAG §一, scale rule] softmax_scale if non-zero, else 1/sqrt(D) with D the q/k head dim."""
    return float(softmax_scale) if softmax_scale != 0 else 1.0 / math.sqrt(D)


def visible(S1: int, S2: int, mask_mode: int, win_left: int, win_right: int) -> np.ndarray:
    """Boolean [S1, S2]: True where key j takes part in query i's softmax.

    mask_mode 0 = none (windows must be -1: [FAG §4.6, dense-attention combination]),
    1 = causal, 2 = band; d = j - i - (S2 - S1) must satisfy d <= 0 (causal),
    d >= -win_left (win_left >= 0), d <= win_right (win_right >= 0).
    """
    if mask_mode not in (0, 1, 2):
        raise ValueError(f"mask_mode must be 0, 1 or 2, got {mask_mode}")
    if mask_mode == 0 and (win_left >= 0 or win_right >= 0):
        raise ValueError("mask_mode 0 (dense) takes no window")
    i = np.arange(S1)[:, None]
    j = np.arange(S2)[None, :]
    d = j - i - (S2 - S1)
    ok = np.ones((S1, S2), dtype=bool)
    if mask_mode == 1:
        ok &= d <= 0
    if win_left >= 0:
        ok &= d >= -win_left
    if win_right >= 0:
        ok &= d <= win_right
    return ok


def _scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """[FAG §一] S = scale · Q Kᵀ."""
    return scale * (q @ k.T)


def _probs(s: np.ndarray, lse: np.ndarray, ok: np.ndarray) -> np.ndarray:
    """[FAG §一] P_ij = exp(S_ij - lse_i) on visible pairs, 0 elsewhere (P rebuilt from lse)."""
    with np.errstate(invalid="ignore", over="ignore"):
        e = np.exp(s - lse[:, None])
    return np.where(ok, e, 0.0)


def _sfmg(dy: np.ndarray, y: np.ndarray) -> np.ndarray:
    """[FAG §一] sfmg = rowsum(dY ⊙ Y)."""
    return (dy * y).sum(axis=1)


def _dp(dy: np.ndarray, v: np.ndarray) -> np.ndarray:
    """[FAG §一] dP = dY · Vᵀ."""
    return dy @ v.T


def _ds(p: np.ndarray, dp: np.ndarray, sfmg: np.ndarray) -> np.ndarray:
    """[FAG §一] dS = P ⊙ (dP - sfmg) with sfmg broadcast along each row."""
    return p * (dp - sfmg[:, None])


def _dv(p: np.ndarray, dy: np.ndarray) -> np.ndarray:
    """[FAG §一] dV = Pᵀ dY."""
    return p.T @ dy


def _dq(ds: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """[FAG §一] dQ = scale · dS · K."""
    return scale * (ds @ k)


def _dk(ds: np.ndarray, q: np.ndarray, scale: float) -> np.ndarray:
    """[FAG §一] dK = scale · dSᵀ · Q."""
    return scale * (ds.T @ q)


def forward_head(q, k, v, scale: float, ok, sink: Optional[float] = None) -> Tuple[np.ndarray, np.ndarray]:
    """[FAG §一] one head's forward: returns (Y [S1, Dv], lse [S1]).

    lse_i = log Σ_{visible j} exp(S_ij) (natural log), evaluated with the row maximum taken out;
    rows with no visible key get lse = +inf and Y = 0.  With a sink logit (reading of the
    optional `sinks` input, see the module notes) the normaliser gains exp(sink): lse_i =
    log(exp(sink) + Σ_{visible j} exp(S_ij)), so a row with no visible key gets lse = sink.
    """
    s = _scores(q, k, scale)
    s = np.where(ok, s, -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    if sink is not None:
        m = np.maximum(m, float(sink))
    has = np.isfinite(m)
    m0 = np.where(has, m, 0.0)
    with np.errstate(invalid="ignore"):
        total = np.exp(s - m0[:, None]).sum(axis=1)
    if sink is not None:
        total = total + np.exp(float(sink) - m0)
    lse = np.where(has, m0 + np.log(np.where(has, total, 1.0)), np.inf)
    p = _probs(np.where(ok, s, 0.0), lse, ok)
    return p @ v, lse


def forward_stats_head(q, k, v, scale: float, ok) -> Tuple[np.ndarray, np.ndarray]:
    """One head's forward statistics in the (softmaxMax, softmaxSum) form that the pages
    "LaserAttentionGrad" (ascend-transformer-boost, its backward inputs) and
    "aclnnFusedFloydAttentionGrad" (its softmaxMax/softmaxSum parameters) take in place of an
    lse: the row maximum m_i of the visible S_ij and the row sum l_i = Σ_{visible j} exp(S_ij − m_i).
    Rows with no visible key get m = −inf, l = 0."""
    s = np.where(ok, _scores(q, k, scale), -np.inf)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    has = np.isfinite(m)
    with np.errstate(invalid="ignore"):
        l = np.where(has, np.exp(s - np.where(has, m, 0.0)[:, None]).sum(axis=1), 0.0)
    return m, l


def lse_from_stats(m, l) -> np.ndarray:
    """lse = m + ln(l) for a (maximum, sum of exp(S − maximum)) pair, so that exp(S − lse) is the
    softmax; a row with l <= 0 saw no key and gets lse = +inf (P = 0), as forward_head gives."""
    m = np.asarray(m, np.float64)
    l = np.asarray(l, np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), np.inf)


def backward_head(q, k, v, dy, y, lse, scale: float, ok):
    """[FAG §一] one head's backward from saved Y and lse: returns (dQ, dK, dV, sfmg)."""
    p = _probs(_scores(q, k, scale), lse, ok)
    sfmg = _sfmg(dy, y)
    ds = _ds(p, _dp(dy, v), sfmg)
    return _dq(ds, k, scale), _dk(ds, q, scale), _dv(p, dy), sfmg


# ----------------------------------------------------------------------------------------------
# layouts: BSND [B,S,N,D], BNSD [B,N,S,D], TND [T,N,D] with cu_seqlens  ([FAG §4.6])
# ----------------------------------------------------------------------------------------------


def _tnd_sequences(cu_q, cu_kv):
    """[FAG §4.6] TND: sequence s covers q rows [cu_q[s], cu_q[s+1]) and kv rows likewise."""
    if cu_q is None or cu_kv is None:
        raise ValueError("TND needs cu_seqlens_q and cu_seqlens_kv")
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_kv = np.asarray(cu_kv, dtype=np.int64)
    if len(cu_q) != len(cu_kv):
        raise ValueError("cu_seqlens_q and cu_seqlens_kv differ in length")
    return [(None, slice(int(cu_q[s]), int(cu_q[s + 1])), slice(int(cu_kv[s]), int(cu_kv[s + 1])))
            for s in range(len(cu_q) - 1)]


class _View:
    """Per-(sequence, head) [rows, dim] views of a tensor in one of the three layouts."""

    def __init__(self, layout: str, x: np.ndarray):
        self.layout, self.x = layout, x

    def get(self, b, rows: slice, n: int) -> np.ndarray:
        if self.layout == "BSND":
            return self.x[b, rows, n, :]
        if self.layout == "BNSD":
            return self.x[b, n, rows, :]
        return self.x[rows, n, :]

    def add(self, b, rows: slice, n: int, val: np.ndarray) -> None:
        if self.layout == "BSND":
            self.x[b, rows, n, :] += val
        elif self.layout == "BNSD":
            self.x[b, n, rows, :] += val
        else:
            self.x[rows, n, :] += val

    @property
    def heads(self) -> int:
        return self.x.shape[2] if self.layout == "BSND" else self.x.shape[1]


def _seq_list(layout, q, k, cu_q, cu_kv, seqused_q=None, seqused_kv=None):
    """(batch or None, q rows, kv rows) of every sequence; with seqused_q / seqused_kv only the
    first seqused[b] rows of sequence b take part (reading of the optional inputs of [FAG §2.1])."""
    if layout == "TND":
        seqs = _tnd_sequences(cu_q, cu_kv)
    elif cu_q is not None or cu_kv is not None:
        raise ValueError("cu_seqlens are only taken with the TND layout")
    elif layout == "BSND":
        seqs = [(b, slice(0, q.shape[1]), slice(0, k.shape[1])) for b in range(q.shape[0])]
    elif layout == "BNSD":
        seqs = [(b, slice(0, q.shape[2]), slice(0, k.shape[2])) for b in range(q.shape[0])]
    else:
        raise ValueError(f"unknown layout {layout!r}")

    def used(rows: slice, u, s) -> slice:
        if u is None:
            return rows
        n = int(np.asarray(u)[s])
        if not 0 <= n <= rows.stop - rows.start:
            raise ValueError(f"seqused[{s}] = {n} is outside [0, {rows.stop - rows.start}]")
        return slice(rows.start, rows.start + n)

    for u in (seqused_q, seqused_kv):
        if u is not None and len(np.asarray(u)) != len(seqs):
            raise ValueError("seqused needs one entry per sequence")
    return [(b, used(rq, seqused_q, s), used(rk, seqused_kv, s)) for s, (b, rq, rk) in enumerate(seqs)]


def _lse_get(layout, lse, b, rows, n):
    return lse[n, rows] if layout == "TND" else lse[b, n, rows]


def _lse_set(layout, lse, b, rows, n, val):
    if layout == "TND":
        lse[n, rows] = val
    else:
        lse[b, n, rows] = val


def _lse_shape(layout, q, N1):
    if layout == "TND":
        return (N1, q.shape[0])
    if layout == "BSND":
        return (q.shape[0], N1, q.shape[1])
    return (q.shape[0], N1, q.shape[2])


def _kv_head(n1: int, N1: int, N2: int) -> int:
    """GQA head map (reading of [FAG §一 notation]): q-heads form contiguous groups of G = N1/N2,
    q-head n1 reads kv-head n1 // G."""
    return n1 // (N1 // N2)


def _group(N1: int, N2: int) -> int:
    """[FAG §一 notation / §4.6] N1 must be a multiple of N2; G = N1 / N2 q-heads per kv-head."""
    if N2 <= 0 or N1 % N2 != 0:
        raise ValueError(f"N1={N1} must be a positive multiple of N2={N2}")
    return N1 // N2


def forward(q, k, v, *, layout="BSND", cu_seqlens_q=None, cu_seqlens_kv=None, softmax_scale=0.0,
            mask_mode=0, win_left=-1, win_right=-1, seqused_q=None, seqused_kv=None, sinks=None):
    """Forward over all sequences and heads: returns (Y in q's layout with Dv, lse fp64).

    lse has shape (B, N1, S1) for BSND/BNSD and (N1, T1) for TND [FAG §4.6]; rows outside every
    sequence's used rows keep lse = +inf and Y = 0.  sinks: None or one logit per q-head.
    """
    Q, K, V = _View(layout, q), _View(layout, k), _View(layout, v)
    N1, N2 = Q.heads, K.heads
    G = _group(N1, N2)
    D, Dv = q.shape[-1], v.shape[-1]
    scale = resolve_scale(softmax_scale, D)
    if sinks is not None and len(np.asarray(sinks)) != N1:
        raise ValueError("sinks needs one logit per q-head")
    y = np.zeros(q.shape[:-1] + (Dv,), dtype=np.float64)
    Y = _View(layout, y)
    lse = np.full(_lse_shape(layout, q, N1), np.inf, dtype=np.float64)
    for b, rq, rk in _seq_list(layout, q, k, cu_seqlens_q, cu_seqlens_kv, seqused_q, seqused_kv):
        S1, S2 = rq.stop - rq.start, rk.stop - rk.start
        ok = visible(S1, S2, mask_mode, win_left, win_right)
        for n1 in range(N1):
            n2 = _kv_head(n1, N1, N2)
            sink = None if sinks is None else float(np.asarray(sinks)[n1])
            yh, lh = forward_head(Q.get(b, rq, n1), K.get(b, rk, n2), V.get(b, rk, n2), scale, ok, sink)
            Y.add(b, rq, n1, yh)
            _lse_set(layout, lse, b, rq, n1, lh)
    return y, lse


def backward(q, k, v, dout, attn_out, softmax_lse, *, layout="BSND", cu_seqlens_q=None,
             cu_seqlens_kv=None, softmax_scale=0.0, mask_mode=0, win_left=-1, win_right=-1, seqused_q=None,
             seqused_kv=None):
    """Backward over all sequences and heads: returns (dq, dk, dv, sfmg), fp64.

    dk/dv of kv-head n2 sum the contributions of its G q-heads; sfmg has lse's shape.  Rows
    outside every sequence's used rows get zero gradients (and sfmg 0).  There is no sinks
    argument: under the reading in the module notes the sink is already inside softmax_lse.
    """
    Q, K, V = _View(layout, q), _View(layout, k), _View(layout, v)
    dY, Yv = _View(layout, dout), _View(layout, attn_out)
    N1, N2 = Q.heads, K.heads
    G = _group(N1, N2)
    scale = resolve_scale(softmax_scale, q.shape[-1])
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    dQ, dK, dV = _View(layout, dq), _View(layout, dk), _View(layout, dv)
    sfmg = np.zeros(_lse_shape(layout, q, N1))
    for b, rq, rk in _seq_list(layout, q, k, cu_seqlens_q, cu_seqlens_kv, seqused_q, seqused_kv):
        S1, S2 = rq.stop - rq.start, rk.stop - rk.start
        ok = visible(S1, S2, mask_mode, win_left, win_right)
        for n1 in range(N1):
            n2 = _kv_head(n1, N1, N2)
            gq, gk, gv, sf = backward_head(
                Q.get(b, rq, n1), K.get(b, rk, n2), V.get(b, rk, n2), dY.get(b, rq, n1),
                Yv.get(b, rq, n1), np.asarray(_lse_get(layout, softmax_lse, b, rq, n1), np.float64),
                scale, ok)
            dQ.add(b, rq, n1, gq)
            dK.add(b, rk, n2, gk)
            dV.add(b, rk, n2, gv)
            _lse_set(layout, sfmg, b, rq, n1, sf)
    return dq, dk, dv, sfmg


# ----------------------------------------------------------------------------------------------
# sampled outputs: the same definitions evaluated for a few output rows (full-size checks)
# ----------------------------------------------------------------------------------------------


def backward_sampled(q, k, v, dout, attn_out, softmax_lse, *, q_rows: Sequence[Tuple[int, int, int]],
                     kv_rows: Sequence[Tuple[int, int, int]], layout="BSND", cu_seqlens_q=None,
                     cu_seqlens_kv=None, softmax_scale=0.0, mask_mode=0, win_left=-1, win_right=-1,
                     seqused_q=None, seqused_kv=None):
    """dQ rows and dK/dV rows for chosen outputs, one at a time.

    q_rows: (sequence or batch s, q-head n1, row i within the sequence) -> dq row [D]
    kv_rows: (sequence or batch s, kv-head n2, row j within the sequence) -> (dk row, dv row)
    Same definitions as `backward` ([FAG §一]); only the requested rows/columns of P and dS are
    formed.  Returns (list of dq rows, list of dk rows, list of dv rows).
    """
    Q, K, V = _View(layout, q), _View(layout, k), _View(layout, v)
    dY, Yv = _View(layout, dout), _View(layout, attn_out)
    N1, N2 = Q.heads, K.heads
    G = _group(N1, N2)
    scale = resolve_scale(softmax_scale, q.shape[-1])
    seqs = _seq_list(layout, q, k, cu_seqlens_q, cu_seqlens_kv, seqused_q, seqused_kv)
    out_q: List[np.ndarray] = []
    for s, n1, i in q_rows:
        b, rq, rk = seqs[s]
        S1, S2 = rq.stop - rq.start, rk.stop - rk.start
        n2 = _kv_head(n1, N1, N2)
        ok = visible(S1, S2, mask_mode, win_left, win_right)[i:i + 1]
        qi = Q.get(b, rq, n1)[i:i + 1]
        kk, vv = K.get(b, rk, n2), V.get(b, rk, n2)
        lse_i = np.asarray(_lse_get(layout, softmax_lse, b, rq, n1), np.float64)[i:i + 1]
        p = _probs(_scores(qi, kk, scale), lse_i, ok)
        dyi, yi = dY.get(b, rq, n1)[i:i + 1], Yv.get(b, rq, n1)[i:i + 1]
        ds = _ds(p, _dp(dyi, vv), _sfmg(dyi, yi))
        out_q.append(_dq(ds, kk, scale)[0])
    out_k: List[np.ndarray] = []
    out_v: List[np.ndarray] = []
    for s, n2, j in kv_rows:
        b, rq, rk = seqs[s]
        S1, S2 = rq.stop - rq.start, rk.stop - rk.start
        ok = visible(S1, S2, mask_mode, win_left, win_right)[:, j:j + 1]
        kj, vj = K.get(b, rk, n2)[j:j + 1], V.get(b, rk, n2)[j:j + 1]
        gk = np.zeros(k.shape[-1])
        gv = np.zeros(v.shape[-1])
        for n1 in [h for h in range(N1) if _kv_head(h, N1, N2) == n2]:
            qq, dyy, yy = Q.get(b, rq, n1), dY.get(b, rq, n1), Yv.get(b, rq, n1)
            lse_h = np.asarray(_lse_get(layout, softmax_lse, b, rq, n1), np.float64)
            p = _probs(_scores(qq, kj, scale), lse_h, ok)          # column j of P: [S1, 1]
            ds = _ds(p, _dp(dyy, vj), _sfmg(dyy, yy))
            gk += _dk(ds, qq, scale)[0]
            gv += _dv(p, dyy)[0]
        out_k.append(gk)
        out_v.append(gv)
    return out_q, out_k, out_v
