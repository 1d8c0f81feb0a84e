"""Seeded synthetic inputs for the FlashAttention backward pass.

This module is the one piece shared by the CUDA path's callers (tests, bench, smoke check) and
the fp64 oracle's callers.  It holds none of the attention arithmetic: it draws iid normal
values from a seeded numpy PCG64 stream, rounds them to the io dtype (round-to-nearest-even via
torch's dtype conversion), and draws varlen sequence lengths.  attn_out and softmax_lse are NOT
made here: they come from a forward pass run by whoever needs them.

Workloads follow the shapes of the flash_attn_grad statement on the page
"CANN ops-transformer FlashAttnGrad 算子详解" (discosf.com/news/4863418), §一 notation
(B, S1, S2, N1, N2, D, Dv, T1, T2) and §4.6 constraints (0 < Dv <= D <= 192, N1 % N2 == 0).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

IO_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention-backward problem: shapes, layout, mask and how its inputs are drawn."""

    name: str
    layout: str            # "BSND", "TND" or "BNSD"
    dtype: str             # "bf16" or "fp16"
    B: int                 # batch (BSND/BNSD) or number of sequences (TND)
    N1: int
    N2: int
    D: int
    Dv: int
    S1: int = 0            # BSND/BNSD sequence lengths; TND: max_seqlen (derived from lengths)
    S2: int = 0
    mask_mode: int = 0     # 0 none, 1 causal, 2 band
    win_left: int = -1
    win_right: int = -1
    softmax_scale: float = 0.0   # 0 -> 1/sqrt(D)
    dout_std: float = 1.0
    varlen_lo: int = 0     # TND lengths drawn uniformly from [varlen_lo, varlen_hi]
    varlen_hi: int = 0
    seed: int = 0


# The five workloads of the attention-backward measurement, named by what they are.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("mha_s128_d64", "BSND", "bf16", B=1, N1=2, N2=2, D=64, Dv=64, S1=128, S2=128,
                 softmax_scale=1.0 / 8.0, seed=1000),
        Workload("causal_b2_s2048_d128", "BSND", "bf16", B=2, N1=16, N2=16, D=128, Dv=128,
                 S1=2048, S2=2048, mask_mode=1, softmax_scale=1.0 / math.sqrt(128), seed=1001),
        Workload("gqa_causal_s4096_d128", "BSND", "bf16", B=1, N1=32, N2=8, D=128, Dv=128,
                 S1=4096, S2=4096, mask_mode=1, dout_std=0.1, seed=1002),
        Workload("varlen_window_fp16_d128", "TND", "fp16", B=8, N1=16, N2=16, D=128, Dv=128,
                 mask_mode=1, win_left=1024, win_right=0, varlen_lo=256, varlen_hi=4096,
                 seed=1003),
        Workload("causal_s8192_d192_dv128", "BSND", "bf16", B=1, N1=16, N2=16, D=192, Dv=128,
                 S1=8192, S2=8192, mask_mode=1, softmax_scale=1.0 / math.sqrt(192), seed=1004),
    ]
}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal(gen: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """iid N(0, std^2) draws in fp64."""
    return gen.standard_normal(size=shape, dtype=np.float64) * std


def round_io(x: np.ndarray, dtype: str) -> torch.Tensor:
    """Round fp64 values to the io dtype (RNE); returns a contiguous CPU tensor."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(IO_DTYPES[dtype]).contiguous()


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def varlen_lengths(gen: np.random.Generator, n: int, lo: int, hi: int) -> np.ndarray:
    """n integer lengths drawn uniformly from [lo, hi], both ends included."""
    return gen.integers(lo, hi + 1, size=n, dtype=np.int64)


def cu_seqlens(lengths) -> np.ndarray:
    """int32 prefix sums with a leading 0: sequence s covers rows [cu[s], cu[s+1])."""
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    return cu.astype(np.int32)


@dataclasses.dataclass
class Problem:
    """Drawn inputs of one workload (CPU tensors in the io dtype) and its resolved sizes."""

    w: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dout: torch.Tensor
    S1: int
    S2: int
    T1: int
    T2: int
    cu_seqlens_q: Optional[np.ndarray]
    cu_seqlens_kv: Optional[np.ndarray]


def _shape(layout: str, B: int, S: int, N: int, D: int, T: int):
    if layout == "BSND":
        return (B, S, N, D)
    if layout == "BNSD":
        return (B, N, S, D)
    if layout == "TND":
        return (T, N, D)
    raise ValueError(f"unknown layout {layout!r}")


def make_problem(w: Workload, lengths_q=None, lengths_kv=None) -> Problem:
    """Draw q, k, v, dout for workload w (seeded by w.seed).

    TND lengths are drawn from [varlen_lo, varlen_hi] unless given; kv lengths equal q lengths
    unless given.
    """
    g = rng(w.seed)
    cu_q = cu_kv = None
    S1, S2, T1, T2 = w.S1, w.S2, w.B * w.S1, w.B * w.S2
    if w.layout == "TND":
        if lengths_q is None:
            lengths_q = varlen_lengths(g, w.B, w.varlen_lo, w.varlen_hi)
        lengths_q = np.asarray(lengths_q, dtype=np.int64)
        lengths_kv = lengths_q if lengths_kv is None else np.asarray(lengths_kv, dtype=np.int64)
        cu_q, cu_kv = cu_seqlens(lengths_q), cu_seqlens(lengths_kv)
        T1, T2 = int(cu_q[-1]), int(cu_kv[-1])
        S1 = int(lengths_q.max()) if len(lengths_q) else 0
        S2 = int(lengths_kv.max()) if len(lengths_kv) else 0
    q = round_io(normal(g, _shape(w.layout, w.B, S1, w.N1, w.D, T1)), w.dtype)
    k = round_io(normal(g, _shape(w.layout, w.B, S2, w.N2, w.D, T2)), w.dtype)
    v = round_io(normal(g, _shape(w.layout, w.B, S2, w.N2, w.Dv, T2)), w.dtype)
    dout = round_io(normal(g, _shape(w.layout, w.B, S1, w.N1, w.Dv, T1), w.dout_std), w.dtype)
    return Problem(w, q, k, v, dout, S1, S2, T1, T2, cu_q, cu_kv)


def sized(w: Workload, **changes) -> Workload:
    """A copy of w with some fields changed (smaller parity cases of the same structure)."""
    return dataclasses.replace(w, **changes)
