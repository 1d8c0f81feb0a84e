"""Test helpers: oracle references for drawn problems and the parity metrics.

The reference side calls only the fp64 oracle; the GPU side calls only the libfabwd C ABI
(through the package's binding).  They share the seeded input generator and nothing else.
"""
from __future__ import annotations

import dataclasses
import multiprocessing
import os
from typing import Optional

import numpy as np
import torch

from attention_backward_fabwd_gb300 import inputs
from oracle import fabwd_oracle as orc

# Tolerances for bf16/fp16 outputs and the fp32 sfmg, as the measurement statement gives them:
# relative L2 error per output tensor <= 1e-2, max-abs error <= 2e-2 * max|ref|, sfmg rel <= 1e-5.
REL_L2 = 1e-2
MAX_ABS_FRAC = 2e-2
SFMG_REL = 1e-5


def mask_kwargs(w: inputs.Workload) -> dict:
    return dict(softmax_scale=w.softmax_scale, mask_mode=w.mask_mode, win_left=w.win_left, win_right=w.win_right)


def oracle_kwargs(pb: inputs.Problem) -> dict:
    kw = dict(layout=pb.w.layout, **mask_kwargs(pb.w))
    if pb.w.layout == "TND":
        kw.update(cu_seqlens_q=pb.cu_seqlens_q, cu_seqlens_kv=pb.cu_seqlens_kv)
    return kw


@dataclasses.dataclass
class Reference:
    attn_out: torch.Tensor        # io dtype, CPU
    lse: torch.Tensor             # fp32, CPU
    dq: Optional[np.ndarray] = None
    dk: Optional[np.ndarray] = None
    dv: Optional[np.ndarray] = None
    sfmg: Optional[np.ndarray] = None


def forward_inputs(pb: inputs.Problem) -> Reference:
    """attn_out (rounded to the io dtype) and fp32 lse from the fp64 oracle forward."""
    q, k, v = (inputs.to_f64(t) for t in (pb.q, pb.k, pb.v))
    y, lse = orc.forward(q, k, v, **oracle_kwargs(pb))
    return Reference(attn_out=inputs.round_io(y, pb.w.dtype), lse=torch.from_numpy(lse.astype(np.float32)))


def full_reference(pb: inputs.Problem) -> Reference:
    """Forward inputs plus the oracle backward computed from exactly those inputs."""
    ref = forward_inputs(pb)
    q, k, v, dy = (inputs.to_f64(t) for t in (pb.q, pb.k, pb.v, pb.dout))
    dq, dk, dv, sf = orc.backward(q, k, v, dy, inputs.to_f64(ref.attn_out), ref.lse.numpy().astype(np.float64),
                                  **oracle_kwargs(pb))
    ref.dq, ref.dk, ref.dv, ref.sfmg = dq, dk, dv, sf
    return ref


def run_gpu(pb: inputs.Problem, ref: Reference, device="cuda", check_status=True, dq_mode="auto"):
    """Run the libfabwd path on the GPU; returns (dq, dk, dv, sfmg fp32 in lse's layout)."""
    from attention_backward_fabwd_gb300 import api, fabwd

    dev = torch.device(device)
    t = lambda x: x.to(dev)
    cu_q = cu_kv = None
    extra = {}
    if pb.w.layout == "TND":
        cu_q = torch.from_numpy(pb.cu_seqlens_q).to(dev)
        cu_kv = torch.from_numpy(pb.cu_seqlens_kv).to(dev)
        extra = dict(max_seqlen_q=pb.S1, max_seqlen_kv=pb.S2)
    dq, dk, dv, (p, ws) = api.flash_attn_grad(
        t(pb.q), t(pb.k), t(pb.v), t(pb.dout), t(ref.attn_out), t(ref.lse), cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv,
        layout_q=pb.w.layout, layout_kv=pb.w.layout, layout_out=pb.w.layout, check_status=check_status,
        return_workspace=True, dq_mode=dq_mode, **mask_kwargs(pb.w), **extra)
    torch.cuda.synchronize()
    lay = fabwd.fabwd_workspace_layout(p)
    B, N1, R = p.B, p.N1, lay["row_stride"]
    sf_pad = ws[lay["sfmg"]:lay["sfmg"] + B * N1 * R * 4].view(torch.float32).view(B, N1, R).cpu().numpy()
    if pb.w.layout == "TND":
        sf = np.zeros((N1, pb.T1), np.float32)
        cu = pb.cu_seqlens_q
        for s in range(B):
            L = cu[s + 1] - cu[s]
            sf[:, cu[s]:cu[s + 1]] = sf_pad[s, :, :L]
    else:
        sf = sf_pad[:, :, :pb.S1]
    return dq.cpu(), dk.cpu(), dv.cpu(), sf


def errors(got, ref) -> dict:
    """Relative L2 error (over all elements, zeros included) and max-abs error / max|ref|."""
    g = inputs.to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    nref = np.linalg.norm(r)
    diff = g - r
    rel = np.linalg.norm(diff) / nref if nref > 0 else np.linalg.norm(diff)
    mref = np.abs(r).max() if r.size else 0.0
    mabs = np.abs(diff).max() / mref if r.size and mref > 0 else (np.abs(diff).max() if r.size else 0.0)
    return {"rel_l2": float(rel), "max_abs_frac": float(mabs), "finite": bool(np.isfinite(g).all())}


def assert_close(name, got, ref, rel=REL_L2, mabs=MAX_ABS_FRAC):
    e = errors(got, ref)
    assert e["finite"], f"{name}: non-finite values"
    assert e["rel_l2"] <= rel, f"{name}: relative L2 {e['rel_l2']:.3g} > {rel}"
    assert e["max_abs_frac"] <= mabs, f"{name}: max-abs/max|ref| {e['max_abs_frac']:.3g} > {mabs}"
    return e


# ---------------------------------------------------------------------------------------------
# full-size references: the oracle per (batch, kv-head group) in a pool of spawned processes
# ---------------------------------------------------------------------------------------------


def _group_slices(pb: inputs.Problem):
    """Independent pieces of a problem: (batch or all sequences, kv-head n2 with its G q-heads).
    Each piece is a whole problem of its own (N1 = G, N2 = 1), so the oracle's result on it is
    exactly the matching slice of its result on the whole problem."""
    w = pb.w
    G = w.N1 // w.N2
    out = []
    for n2 in range(w.N2):
        hq, hk = slice(n2 * G, (n2 + 1) * G), slice(n2, n2 + 1)
        if w.layout == "TND":
            out.append(((slice(None), hq), (slice(None), hk), (hq, slice(None))))
        elif w.layout == "BSND":
            for b in range(w.B):
                bb = slice(b, b + 1)
                out.append(((bb, slice(None), hq), (bb, slice(None), hk), (bb, hq, slice(None))))
        else:
            for b in range(w.B):
                bb = slice(b, b + 1)
                out.append(((bb, hq), (bb, hk), (bb, hq, slice(None))))
    return out


def _piece(args):
    """Worker: oracle forward (Y rounded to the io dtype, lse to fp32) then oracle backward."""
    q, k, v, dy, dtype, kw = args
    y, lse = orc.forward(q, k, v, **kw)
    y_io = inputs.to_f64(inputs.round_io(y, dtype))
    lse32 = lse.astype(np.float32)
    dq, dk, dv, sf = orc.backward(q, k, v, dy, y_io, lse32.astype(np.float64), **kw)
    return y_io, lse32, dq, dk, dv, sf


def _pool_size(bytes_per_worker: int) -> int:
    n = min(os.cpu_count() or 1, 16)
    try:
        with open("/proc/meminfo") as f:
            avail = next(int(line.split()[1]) * 1024 for line in f if line.startswith("MemAvailable"))
        n = min(n, max(1, int(0.6 * avail // max(bytes_per_worker, 1))))
    except (OSError, StopIteration, ValueError):
        n = min(n, 4)
    return max(1, n)


def full_reference_parallel(pb: inputs.Problem) -> Reference:
    """full_reference of a large problem: the same oracle calls, one per independent piece
    (_group_slices), in a pool of spawned processes with single-threaded BLAS each."""
    w = pb.w
    q, k, v, dy = (inputs.to_f64(t) for t in (pb.q, pb.k, pb.v, pb.dout))
    kw = oracle_kwargs(pb)
    pieces = _group_slices(pb)
    jobs = [(q[sq], k[sk], v[sk], dy[sq], w.dtype, kw) for sq, sk, _ in pieces]
    # per worker: a handful of S1 x S2 fp64 matrices of the longest sequence
    per = 6 * 8 * max(pb.S1, 1) * max(pb.S2, 1) + (1 << 28)
    threads = {k_: os.environ.get(k_) for k_ in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    os.environ.update({k_: "1" for k_ in threads})
    try:
        with multiprocessing.get_context("spawn").Pool(_pool_size(per)) as pool:
            res = pool.map(_piece, jobs, chunksize=1)
    finally:
        for k_, v_ in threads.items():
            if v_ is None:
                os.environ.pop(k_, None)
            else:
                os.environ[k_] = v_
    y = np.zeros(dy.shape)
    lse = np.zeros((w.N1, pb.T1) if w.layout == "TND" else (w.B, w.N1, pb.S1), np.float32)
    dq, dk, dv, sf = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape), np.zeros(lse.shape)
    for (sq, sk, sl), (y_, l_, dq_, dk_, dv_, sf_) in zip(pieces, res):
        y[sq], lse[sl], dq[sq], dk[sk], dv[sk], sf[sl] = y_, l_, dq_, dk_, dv_, sf_
    ref = Reference(attn_out=inputs.round_io(y, w.dtype), lse=torch.from_numpy(lse))
    ref.dq, ref.dk, ref.dv, ref.sfmg = dq, dk, dv, sf
    return ref
