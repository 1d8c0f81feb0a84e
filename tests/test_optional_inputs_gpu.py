"""GPU parity of the optional inputs seqused_q / seqused_kv and sinks ([FAG] §2.1 and §4.2) against
the fp64 oracle, with the readings the oracle states (used rows per sequence; a per-q-head sink
logit inside the softmax normaliser).

The rows past seqused are filled with large finite values that would show in every output if a
kernel let them in; their output rows must come back exactly zero.
"""
import numpy as np
import pytest
import torch

from attention_backward_fabwd_gb300 import api, build, fabwd as F, inputs
from oracle import fabwd_oracle as orc

import fabwd_testlib as tl

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    F.lib()


def _rows_past(pb, used, side):
    """Boolean masks of the padding rows (True) along the token/sequence axis of q or kv."""
    w = pb.w
    if w.layout == "TND":
        cu = pb.cu_seqlens_q if side == "q" else pb.cu_seqlens_kv
        T = pb.T1 if side == "q" else pb.T2
        pad = np.zeros(T, bool)
        for s in range(w.B):
            pad[cu[s] + used[s]:cu[s + 1]] = True
        return pad
    S = pb.S1 if side == "q" else pb.S2
    pad = np.zeros((w.B, S), bool)
    for b in range(w.B):
        pad[b, used[b]:] = True
    return pad


def _fill_padding(x, pad, layout, value):
    x = x.clone()
    m = torch.from_numpy(pad)
    if layout == "TND":
        x[m] = value
    elif layout == "BSND":
        x[m] = value
    else:  # BNSD: [B, N, S, D]
        x.permute(0, 2, 1, 3)[m] = value
    return x


CASES = [
    # name, workload, lengths (TND), seqused_q, seqused_kv
    ("tnd_window_both", inputs.sized(W["varlen_window_fp16_d128"], B=3, N1=4, N2=2, win_left=100),
     ([300, 140, 260], None), [211, 0, 260], [300, 77, 129]),
    ("tnd_causal_q_only", inputs.sized(W["varlen_window_fp16_d128"], dtype="bf16", B=2, N1=2, N2=2, win_left=-1),
     ([257, 190], None), [100, 190], None),
    ("bsnd_gqa_causal_both", inputs.sized(W["gqa_causal_s4096_d128"], B=2, N1=4, N2=2, S1=320, S2=320, dout_std=1.0),
     None, [320, 131], [200, 250]),
    ("bsnd_dense_kv_only_d64", inputs.sized(W["mha_s128_d64"], B=2, S1=200, S2=300), None, None, [1, 300]),
    ("bnsd_band_both", inputs.sized(W["mha_s128_d64"], layout="BNSD", B=2, S1=190, S2=190, mask_mode=2, win_left=20,
                                    win_right=7), None, [150, 190], [190, 64]),
    ("d192_bsnd_causal_both", inputs.sized(W["causal_s8192_d192_dv128"], B=2, N1=2, N2=2, S1=300, S2=300),
     None, [300, 170], [299, 170]),
]


def _problem(case):
    name, w, lens, uq, ukv = case
    pb = inputs.make_problem(w, *(lens or ()))
    uq_ = np.asarray(uq, np.int32) if uq is not None else None
    ukv_ = np.asarray(ukv, np.int32) if ukv is not None else None
    kw = tl.oracle_kwargs(pb)
    kw.update(seqused_q=uq_, seqused_kv=ukv_)
    q, k, v, dy = (inputs.to_f64(t) for t in (pb.q, pb.k, pb.v, pb.dout))
    y, lse = orc.forward(q, k, v, **kw)
    y_io = inputs.round_io(y, w.dtype)
    lse32 = lse.astype(np.float32)
    ref = orc.backward(q, k, v, dy, inputs.to_f64(y_io), lse32.astype(np.float64), **kw)
    return pb, uq_, ukv_, y_io, lse32, ref


def _spans(pb):
    w = pb.w
    if w.layout == "TND":
        return np.diff(pb.cu_seqlens_q), np.diff(pb.cu_seqlens_kv)
    return np.full(w.B, pb.S1), np.full(w.B, pb.S2)


@pytest.mark.parametrize("dq_mode", ["separate", "atomic"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_seqused_against_oracle(case, dq_mode):
    pb, uq, ukv, y_io, lse32, (rdq, rdk, rdv, _) = _problem(case)
    w = pb.w
    span_q, span_k = _spans(pb)
    pad_q = _rows_past(pb, uq if uq is not None else span_q, "q")
    pad_k = _rows_past(pb, ukv if ukv is not None else span_k, "kv")
    # padding rows hold large finite values: q, dout, attn_out and lse there are never used
    big = 300.0
    q, dout, y = (_fill_padding(t, pad_q, w.layout, big) for t in (pb.q, pb.dout, y_io))
    k, v = (_fill_padding(t, pad_k, w.layout, -big) for t in (pb.k, pb.v))
    lse = torch.from_numpy(lse32)
    dev = torch.device("cuda")
    d = lambda x: None if x is None else x.to(dev)
    kw = dict(layout_q=w.layout, layout_kv=w.layout, layout_out=w.layout, check_status=True, dq_mode=dq_mode,
              **tl.mask_kwargs(w))
    if w.layout == "TND":
        kw.update(cu_seqlens_q=d(torch.from_numpy(pb.cu_seqlens_q)), cu_seqlens_kv=d(torch.from_numpy(pb.cu_seqlens_kv)),
                  max_seqlen_q=pb.S1, max_seqlen_kv=pb.S2)
    dq, dk, dv = api.flash_attn_grad(d(q), d(k), d(v), d(dout), d(y), d(lse),
                                     seqused_q=d(torch.from_numpy(uq)) if uq is not None else None,
                                     seqused_kv=d(torch.from_numpy(ukv)) if ukv is not None else None, **kw)
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    tl.assert_close("dq", dq, rdq)
    tl.assert_close("dk", dk, rdk)
    tl.assert_close("dv", dv, rdv)
    # padding rows come back exactly zero
    for t, pad in ((dq, pad_q), (dk, pad_k), (dv, pad_k)):
        x = t.permute(0, 2, 1, 3) if w.layout == "BNSD" else t
        assert x[torch.from_numpy(pad)].abs().max().item() == 0 if pad.any() else True


def test_bad_seqused_is_reported_not_faulted():
    case = CASES[2]
    pb, uq, ukv, y_io, lse32, _ = _problem(case)
    dev = torch.device("cuda")
    args = [t.to(dev) for t in (pb.q, pb.k, pb.v, pb.dout, y_io, torch.from_numpy(lse32))]
    bad = torch.tensor([321, 5], dtype=torch.int32, device=dev)   # 321 > S1 = 320
    with pytest.raises(F.FabwdError) as ei:
        api.flash_attn_grad(*args, mask_mode=1, seqused_q=bad, check_status=True)
    assert ei.value.status == F.FABWD_ERR_DEVICE
    with pytest.raises(ValueError):   # one entry per sequence, checked on the host
        api.flash_attn_grad(*args, mask_mode=1, seqused_kv=bad[:1], check_status=True)
    api.flash_attn_grad(*args, mask_mode=1, check_status=True)   # the context stays usable


@pytest.mark.parametrize("case", [CASES[0], CASES[2], CASES[5]], ids=["tnd", "bsnd", "d192"])
def test_forward_with_seqused_and_sinks(case):
    # fabwd_forward: attn_out and softmax_lse of the used rows (the sink inside the normaliser);
    # padding rows give attn_out = 0, softmax_lse = +inf
    name, w, lens, uq, ukv = case
    pb = inputs.make_problem(w, *(lens or ()))
    sinks = np.random.default_rng(3).standard_normal(w.N1).astype(np.float32) * 2
    kw = tl.oracle_kwargs(pb)
    kw.update(seqused_q=np.asarray(uq, np.int32) if uq is not None else None,
              seqused_kv=np.asarray(ukv, np.int32) if ukv is not None else None)
    q, k, v = (inputs.to_f64(t) for t in (pb.q, pb.k, pb.v))
    y, lse = orc.forward(q, k, v, sinks=sinks.astype(np.float64), **kw)
    dev = torch.device("cuda")
    d = lambda x: None if x is None else torch.from_numpy(np.asarray(x)).to(dev)
    fkw = dict(layout=w.layout, check_status=True, **tl.mask_kwargs(w))
    if w.layout == "TND":
        fkw.update(cu_seqlens_q=d(pb.cu_seqlens_q), cu_seqlens_kv=d(pb.cu_seqlens_kv), max_seqlen_q=pb.S1,
                   max_seqlen_kv=pb.S2)
    yg, lg = api.flash_attn_forward(pb.q.to(dev), pb.k.to(dev), pb.v.to(dev), seqused_q=d(kw["seqused_q"]),
                                    seqused_kv=d(kw["seqused_kv"]), sinks=d(sinks), **fkw)
    tl.assert_close("attn_out", yg.cpu(), y)
    lg = lg.cpu().numpy()
    # as the forward tests: within 1e-4 + 1e-5·|lse| where finite, +inf exactly where the oracle's is
    assert np.array_equal(np.isinf(lg), np.isinf(lse)) and (lg[np.isinf(lse)] > 0).all()
    fin = np.isfinite(lse)
    assert (np.abs(lg[fin] - lse[fin]) <= 1e-4 + 1e-5 * np.abs(lse[fin])).all()


def test_backward_with_sinks_equals_oracle():
    # the lse of a forward with sinks; the backward given the same sinks (which it does not read)
    w = inputs.sized(W["gqa_causal_s4096_d128"], N1=4, N2=2, S1=300, S2=300, dout_std=1.0)
    pb = inputs.make_problem(w)
    sinks = np.array([0.5, -1.0, 3.0, 1.5])
    q, k, v, dy = (inputs.to_f64(t) for t in (pb.q, pb.k, pb.v, pb.dout))
    kw = tl.oracle_kwargs(pb)
    y, lse = orc.forward(q, k, v, sinks=sinks, **kw)
    y_io = inputs.round_io(y, w.dtype)
    lse32 = lse.astype(np.float32)
    rdq, rdk, rdv, _ = orc.backward(q, k, v, dy, inputs.to_f64(y_io), lse32.astype(np.float64), **kw)
    dev = torch.device("cuda")
    args = [t.to(dev) for t in (pb.q, pb.k, pb.v, pb.dout, y_io, torch.from_numpy(lse32))]
    dq, dk, dv = api.flash_attn_grad(*args, mask_mode=1, sinks=torch.tensor(sinks, dtype=torch.float32, device=dev),
                                     check_status=True)
    tl.assert_close("dq", dq.cpu(), rdq)
    tl.assert_close("dk", dk.cpu(), rdk)
    tl.assert_close("dv", dv.cpu(), rdv)
    with pytest.raises(ValueError):   # one logit per q-head
        api.flash_attn_grad(*args, mask_mode=1, sinks=torch.zeros(3, device=dev))
