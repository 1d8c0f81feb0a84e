"""torch-facing call with the argument list of the page "CANN ops-transformer FlashAttnGrad 算子详解"
(discosf.com/news/4863418), §4.2 function prototype, over the libfabwd C ABI.

torch provides device memory and the stream only; every step of the backward runs in libfabwd's
CUDA kernels.  The outputs and the workspace are allocated here (caller-owned in the C ABI).
"""
from __future__ import annotations

import enum
from typing import Optional, Tuple, Union

import torch

from . import fabwd as F


class MaskMode(enum.IntEnum):
    """mask_mode values ([FAG] §4.3 lists an IntEnum whose table was lost; this is the reading
    the library implements): 0 none, 1 causal (bottom-right aligned), 2 band (windows)."""

    NONE = 0
    CAUSAL = 1
    BAND = 2


_DTYPES = {torch.bfloat16: F.FABWD_BF16, torch.float16: F.FABWD_FP16}
_DQ_MODES = {"auto": F.FABWD_DQ_AUTO, "atomic": F.FABWD_DQ_ATOMIC, "separate": F.FABWD_DQ_SEPARATE}


def dq_mode_value(dq_mode: Union[int, str]) -> int:
    """'auto' (0), 'atomic' (1: fp32 workspace + convert) or 'separate' (2: deterministic pass)."""
    if isinstance(dq_mode, str):
        try:
            return _DQ_MODES[dq_mode.strip().lower()]
        except KeyError:
            raise ValueError(f"unknown dq_mode {dq_mode!r}") from None
    return int(dq_mode)


_LAYOUTS = {"BSND": F.FABWD_BSND, "TND": F.FABWD_TND, "BNSD": F.FABWD_BNSD}


def mask_mode_value(mask_mode: Union[int, str, MaskMode]) -> int:
    """Accept an IntEnum, an int or the enum name as a case-insensitive string ([FAG] §4.3)."""
    if isinstance(mask_mode, str):
        try:
            return int(MaskMode[mask_mode.strip().upper()])
        except KeyError:
            raise ValueError(f"unknown mask_mode name {mask_mode!r}") from None
    return int(mask_mode)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def make_params(q, k, v, dout, attn_out, softmax_lse, dq, dk, dv, *, cu_seqlens_q=None, cu_seqlens_kv=None,
                softmax_scale=0.0, mask_mode=0, win_left=-1, win_right=-1, max_seqlen_q=-1, max_seqlen_kv=-1,
                layout="BSND", dq_mode="auto", seqused_q=None, seqused_kv=None, sinks=None) -> F.fabwd_params:
    """Fill fabwd_params from tensors (shapes give B, S1, S2, N1, N2, D, Dv, T1, T2)."""
    if layout not in _LAYOUTS:
        raise ValueError(f"layout must be one of {sorted(_LAYOUTS)}, got {layout!r}")
    if q.dtype not in _DTYPES:
        raise TypeError(f"q must be bfloat16 or float16, got {q.dtype}")
    p = F.fabwd_params()
    p.dtype = _DTYPES[q.dtype]
    p.layout = _LAYOUTS[layout]
    if layout == "TND":
        if cu_seqlens_q is None or cu_seqlens_kv is None:
            raise ValueError("the TND layout needs cu_seqlens_q and cu_seqlens_kv")
        p.B = cu_seqlens_q.numel() - 1
        p.T1, p.N1, p.D = q.shape
        p.T2, p.N2, _ = k.shape
        p.Dv = v.shape[-1]
        if max_seqlen_q < 0 or max_seqlen_kv < 0:
            cq, ck = cu_seqlens_q.to("cpu", torch.int64), cu_seqlens_kv.to("cpu", torch.int64)   # synchronises
            if max_seqlen_q < 0:
                max_seqlen_q = int((cq[1:] - cq[:-1]).max()) if p.B > 0 else 0
            if max_seqlen_kv < 0:
                max_seqlen_kv = int((ck[1:] - ck[:-1]).max()) if p.B > 0 else 0
        p.S1, p.S2 = max_seqlen_q, max_seqlen_kv
    elif layout == "BSND":
        p.B, p.S1, p.N1, p.D = q.shape
        _, p.S2, p.N2, _ = k.shape
        p.Dv = v.shape[-1]
    else:
        p.B, p.N1, p.S1, p.D = q.shape
        _, p.N2, p.S2, _ = k.shape
        p.Dv = v.shape[-1]
    p.q, p.k, p.v, p.dout, p.attn_out = (_ptr(t) for t in (q, k, v, dout, attn_out))
    p.softmax_lse = _ptr(softmax_lse)
    p.cu_seqlens_q, p.cu_seqlens_kv = _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv)
    p.softmax_scale = float(softmax_scale)
    p.mask_mode = mask_mode_value(mask_mode)
    p.win_left, p.win_right = int(win_left), int(win_right)
    p.dq_mode = dq_mode_value(dq_mode)
    p.dq, p.dk, p.dv = _ptr(dq), _ptr(dk), _ptr(dv)
    p.seqused_q, p.seqused_kv, p.sinks = _ptr(seqused_q), _ptr(seqused_kv), _ptr(sinks)
    return p


def _check_tensors(q, k, v, dout, attn_out, stats, cu_q, cu_kv, seqused=(), sinks=None, B=None, N1=None):
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("libfabwd runs on CUDA tensors only")
    for name, t in (("k", k), ("v", v), ("dout", dout), ("attn_out", attn_out)):
        if t.dtype != q.dtype:
            raise TypeError(f"{name} must have q's dtype {q.dtype} ([FAG] §4.6), got {t.dtype}")
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, q on {dev}")
    for name, t in stats:
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32 ([FAG] §4.6)")
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, q on {dev}")
    for name, t in (("cu_seqlens_q", cu_q), ("cu_seqlens_kv", cu_kv)):
        if t is not None and t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    for name, t in seqused:
        if t is None:
            continue
        if t.dtype != torch.int32 or t.device != dev:
            raise TypeError(f"{name} must be an int32 tensor on {dev} ([FAG] §2.1)")
        if B is not None and t.numel() != B:
            raise ValueError(f"{name} needs one entry per sequence ({B}), got {t.numel()}")
    if sinks is not None:
        if sinks.dtype != torch.float32 or sinks.device != dev:
            raise TypeError(f"sinks must be a float32 tensor on {dev} ([FAG] §2.1)")
        if N1 is not None and sinks.numel() != N1:
            raise ValueError(f"sinks needs one logit per q-head ({N1}), got {sinks.numel()}")


def _batch_and_heads(q, layout, cu_q):
    if layout == "TND":
        return (cu_q.numel() - 1 if cu_q is not None else None), q.shape[1]
    return q.shape[0], (q.shape[2] if layout == "BSND" else q.shape[1])


def flash_attn_grad(q, k, v, dout, attn_out, softmax_lse, cu_seqlens_q=None, cu_seqlens_kv=None, seqused_q=None,
                    seqused_kv=None, sinks=None, attn_mask=None, metadata=None, softmax_scale=0.0, mask_mode=0,
                    win_left=-1, win_right=-1, max_seqlen_q=-1, max_seqlen_kv=-1, layout_q="BSND",
                    layout_kv="BSND", layout_out="BSND", *, softmax_max=None, softmax_sum=None, dq_mode="auto",
                    check_status=False, return_workspace=False) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Gradients (dq, dk, dv) of attention from the saved attn_out and softmax_lse.

    Arguments follow [FAG] §4.2.  The page states no semantics for seqused_q/kv and sinks; the
    readings taken (include/fabwd.h, fabwd_params): seqused_q[b] / seqused_kv[b] (int32, one per
    sequence) are the used query / key rows of sequence b, the rest are padding (zero gradient,
    finite values required); sinks (fp32, one logit per q-head) are already inside softmax_lse,
    so dq, dk and dv do not depend on them and they are only checked.  attn_mask (its layout is not
    stated) raises; `metadata` (an Ascend core-split plan) is accepted and ignored, the GPU
    schedule is derived from the shapes.  The three layouts must
    agree ([FAG] §4.6).  Non-contiguous inputs are made contiguous.  With TND and
    max_seqlen_* = -1 the lengths are read from cu_seqlens on the host (a synchronisation).
    dq_mode selects how dQ is formed: 'atomic' (fp32 reduce-adds into a workspace accumulator, then
    a convert pass), 'separate' (a q-stationary pass, bitwise reproducible) or 'auto'.
    softmax_max / softmax_sum: the forward statistics as a row maximum and a row sum of
    exp(S − max), in place of softmax_lse (which may then be None): lse = max + ln(sum).  They
    have softmax_lse's shape, optionally with a trailing axis that repeats each row's value (the
    (..., 8) layout of the LaserAttentionGrad and FusedFloydAttentionGrad pages).
    check_status=True synchronises and raises if the kernels reported a device-side problem.
    """
    if attn_mask is not None:
        raise NotImplementedError("attn_mask is not supported (its layout and meaning are not stated)")
    if not (layout_q == layout_kv == layout_out):
        raise ValueError("layout_q, layout_kv and layout_out must be the same ([FAG] §4.6)")
    use_stats = softmax_max is not None or softmax_sum is not None
    if use_stats and (softmax_max is None or softmax_sum is None):
        raise ValueError("softmax_max and softmax_sum go together")
    if not use_stats and softmax_lse is None:
        raise ValueError("softmax_lse (or softmax_max with softmax_sum) is required")
    q, k, v, dout, attn_out = (t.contiguous() for t in (q, k, v, dout, attn_out))
    if use_stats:
        softmax_max, softmax_sum = softmax_max.contiguous(), softmax_sum.contiguous()
        if softmax_max.shape != softmax_sum.shape:
            raise ValueError("softmax_max and softmax_sum must have the same shape")
        lse_dims = 2 if layout_q == "TND" else 3
        stat_stride = softmax_max.shape[-1] if softmax_max.dim() == lse_dims + 1 else 1
        softmax_lse = None
    else:
        softmax_lse = softmax_lse.contiguous()
    if cu_seqlens_q is not None:
        cu_seqlens_q = cu_seqlens_q.contiguous()
    if cu_seqlens_kv is not None:
        cu_seqlens_kv = cu_seqlens_kv.contiguous()
    stats = [("softmax_max", softmax_max), ("softmax_sum", softmax_sum)] if use_stats else [("softmax_lse", softmax_lse)]
    seqused_q, seqused_kv, sinks = (None if t is None else t.contiguous() for t in (seqused_q, seqused_kv, sinks))
    B, N1 = _batch_and_heads(q, layout_q, cu_seqlens_q)
    _check_tensors(q, k, v, dout, attn_out, stats, cu_seqlens_q, cu_seqlens_kv,
                   (("seqused_q", seqused_q), ("seqused_kv", seqused_kv)), sinks, B, N1)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    p = make_params(q, k, v, dout, attn_out, softmax_lse, dq, dk, dv, cu_seqlens_q=cu_seqlens_q,
                    cu_seqlens_kv=cu_seqlens_kv, softmax_scale=softmax_scale, mask_mode=mask_mode,
                    win_left=win_left, win_right=win_right, max_seqlen_q=max_seqlen_q,
                    max_seqlen_kv=max_seqlen_kv, layout=layout_q, dq_mode=dq_mode, seqused_q=seqused_q,
                    seqused_kv=seqused_kv, sinks=sinks)
    nbytes = F.fabwd_workspace_size(p)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    if use_stats:
        F.fabwd_preprocess_stats(p, softmax_max.data_ptr(), softmax_sum.data_ptr(), stat_stride, ws.data_ptr(),
                                 ws.numel(), stream)
    else:
        F.fabwd_preprocess(p, ws.data_ptr(), ws.numel(), stream)
    F.fabwd_run(p, ws.data_ptr(), ws.numel(), stream)
    if check_status:
        s, bits = F.fabwd_read_device_status(ws.data_ptr(), ws.numel(), stream)
        if s != F.FABWD_OK:
            raise F.FabwdError(s, f"device status 0x{bits:x}")
    if return_workspace:
        return dq, dk, dv, (p, ws)
    return dq, dk, dv


def flash_attn_forward(q, k, v, cu_seqlens_q=None, cu_seqlens_kv=None, softmax_scale=0.0, mask_mode=0,
                       win_left=-1, win_right=-1, max_seqlen_q=-1, max_seqlen_kv=-1, layout="BSND",
                       check_status=False, seqused_q=None, seqused_kv=None,
                       sinks=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """(attn_out, softmax_lse) of the attention whose gradients flash_attn_grad computes, on the GPU.

    The forward of [FAG] §一 with the same masks, GQA map, layouts and scale rule as the backward:
    attn_out has q's layout with Dv, softmax_lse is fp32 [B][N1][S1] (BSND/BNSD) or [N1][T1] (TND),
    natural-log; a row with no visible key gets attn_out = 0 and softmax_lse = +inf.  The pair is
    what flash_attn_grad takes as attn_out and softmax_lse.  seqused_q / seqused_kv and sinks as
    for flash_attn_grad: rows past seqused get attn_out = 0 and softmax_lse = +inf, and a sink
    logit joins every row's normaliser (softmax_lse = ln(exp(sink) + Σ exp(S))).
    """
    q, k, v = (t.contiguous() for t in (q, k, v))
    if cu_seqlens_q is not None:
        cu_seqlens_q = cu_seqlens_q.contiguous()
    if cu_seqlens_kv is not None:
        cu_seqlens_kv = cu_seqlens_kv.contiguous()
    seqused_q, seqused_kv, sinks = (None if t is None else t.contiguous() for t in (seqused_q, seqused_kv, sinks))
    B, N1 = _batch_and_heads(q, layout, cu_seqlens_q)
    _check_tensors(q, k, v, q, q, [], cu_seqlens_q, cu_seqlens_kv, (("seqused_q", seqused_q), ("seqused_kv", seqused_kv)),
                   sinks, B, N1)
    out = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    # make_params reads the shapes from q, k, v; dout/attn_out/lse/dq/dk/dv are unused by the forward.
    p = make_params(q, k, v, None, out, None, None, None, None, cu_seqlens_q=cu_seqlens_q,
                    cu_seqlens_kv=cu_seqlens_kv, softmax_scale=softmax_scale, mask_mode=mask_mode,
                    win_left=win_left, win_right=win_right, max_seqlen_q=max_seqlen_q,
                    max_seqlen_kv=max_seqlen_kv, layout=layout, seqused_q=seqused_q, seqused_kv=seqused_kv,
                    sinks=sinks)
    if layout == "TND":
        lse = torch.empty((p.N1, p.T1), dtype=torch.float32, device=q.device)
    else:
        lse = torch.empty((p.B, p.N1, p.S1), dtype=torch.float32, device=q.device)
    ws = torch.empty(256, dtype=torch.uint8, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    F.fabwd_forward(p, out.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    if check_status:
        s, bits = F.fabwd_read_device_status(ws.data_ptr(), ws.numel(), stream)
        if s != F.FABWD_OK:
            raise F.FabwdError(s, f"device status 0x{bits:x}")
    return out, lse
