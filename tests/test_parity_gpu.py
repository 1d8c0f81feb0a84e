"""GPU parity: the libfabwd CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (the measurement statement's): per output tensor relative L2 <= 1e-2 and
max-abs <= 2e-2 · max|ref|; the fp32 sfmg within 1e-5 relative.  Small cases compare every
element and span several 128-row tiles with ragged tails; the five full-size workloads compare
every element too, with the oracle run per kv-head group in a pool of processes.
"""
import math

import numpy as np
import pytest
import torch

from attention_backward_fabwd_gb300 import api, fabwd as F, inputs
from oracle import fabwd_oracle as orc

import fabwd_testlib as tl

pytestmark = pytest.mark.gpu

W = inputs.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_backward_fabwd_gb300 import build

    build.build()
    F.lib()


def check_all(pb, ref, dq, dk, dv, sf):
    out = {}
    out["dq"] = tl.assert_close("dq", dq, ref.dq)
    out["dk"] = tl.assert_close("dk", dk, ref.dk)
    out["dv"] = tl.assert_close("dv", dv, ref.dv)
    e = tl.errors(sf, ref.sfmg)
    assert e["rel_l2"] <= tl.SFMG_REL, f"sfmg rel {e['rel_l2']}"
    return out


SMALL = [
    ("mha_s128_d64", W["mha_s128_d64"], None),
    ("causal_b2_s384", inputs.sized(W["causal_b2_s2048_d128"], N1=2, N2=2, S1=384, S2=384), None),
    ("gqa_causal_ragged", inputs.sized(W["gqa_causal_s4096_d128"], N1=4, N2=2, S1=300, S2=300, dout_std=1.0), None),
    ("gqa8", inputs.sized(W["gqa_causal_s4096_d128"], N1=8, N2=1, S1=200, S2=200, dout_std=1.0), None),
    ("dense_s1_lt_s2", inputs.sized(W["mha_s128_d64"], S1=200, S2=333, D=128, Dv=128), None),
    ("causal_s1_gt_s2", inputs.sized(W["causal_b2_s2048_d128"], B=1, N1=2, N2=2, S1=300, S2=150), None),
    ("causal_s1_lt_s2", inputs.sized(W["causal_b2_s2048_d128"], B=1, N1=2, N2=2, S1=150, S2=420), None),
    ("band_bnsd_d64", inputs.sized(W["mha_s128_d64"], layout="BNSD", S1=190, S2=190, mask_mode=2, win_left=20,
                                    win_right=7), None),
    ("band_wide", inputs.sized(W["causal_b2_s2048_d128"], B=1, N1=2, N2=2, S1=520, S2=520, mask_mode=2,
                               win_left=200, win_right=150), None),
    ("window_left_only", inputs.sized(W["causal_b2_s2048_d128"], B=1, N1=2, N2=1, S1=400, S2=400, mask_mode=2,
                                      win_left=64), None),
    ("fp16_dense_d64", inputs.sized(W["mha_s128_d64"], dtype="fp16", S1=257, S2=129), None),
    ("scale_0_3", inputs.sized(W["mha_s128_d64"], softmax_scale=0.3, S1=130, S2=260), None),
    ("bsnd_bf16_causal_window", inputs.sized(W["causal_b2_s2048_d128"], B=1, N1=2, N2=2, S1=700, S2=700,
                                             win_left=150, win_right=0), None),
    ("tnd_fp16_window", inputs.sized(W["varlen_window_fp16_d128"], B=5, N1=2, N2=2, win_left=64),
     ([130, 1, 0, 257, 64], None)),
    ("tnd_bf16_gqa_dense", inputs.sized(W["varlen_window_fp16_d128"], dtype="bf16", B=3, N1=4, N2=2, mask_mode=0,
                                        win_left=-1, win_right=-1), ([200, 33, 129], [90, 300, 129])),
    ("tnd_causal_unequal", inputs.sized(W["varlen_window_fp16_d128"], B=3, N1=2, N2=1, win_left=-1),
     ([200, 33, 300], [150, 60, 300])),
    # more sequences than a warp has lanes (the varlen grid's unit scan runs over groups of 32),
    # empty ones among them, q and kv lengths unequal
    ("tnd_many_sequences", inputs.sized(W["varlen_window_fp16_d128"], B=37, N1=2, N2=1, win_left=64),
     ([(i * 53) % 190 for i in range(37)], [(i * 71 + 5) % 160 for i in range(37)])),
    # exactly one warp's worth of sequences (every lane of the varlen scans holds one)
    ("tnd_32_sequences", inputs.sized(W["varlen_window_fp16_d128"], dtype="bf16", B=32, N1=4, N2=2, win_left=40),
     ([(i * 29) % 140 for i in range(32)], [(i * 43 + 7) % 150 for i in range(32)])),
    # more sequences than the flat varlen grid takes: the (units, B) grid, empty CTAs included
    ("tnd_70_sequences", inputs.sized(W["varlen_window_fp16_d128"], B=70, N1=2, N2=2, win_left=-1),
     ([(i * 37) % 150 for i in range(70)], None)),
    ("d192_dv128_causal", inputs.sized(W["causal_s8192_d192_dv128"], N1=2, N2=2, S1=300, S2=300), None),
    ("d192_dv128_gqa_fp16_band", inputs.sized(W["causal_s8192_d192_dv128"], dtype="fp16", N1=4, N2=2, S1=260,
                                              S2=390, mask_mode=2, win_left=100, win_right=30), None),
    ("d192_tnd", inputs.sized(W["varlen_window_fp16_d128"], D=192, Dv=128, B=3, N1=2, N2=2, win_left=64),
     ([70, 1, 200], None)),
    # the other head-dim classes of [FAG] §5.1 (d_align 64/128/192, Dv <= D), and dims between
    # them, which run in the next larger kernel
    ("d128_dv64_causal", inputs.sized(W["causal_b2_s2048_d128"], B=1, N1=2, N2=2, S1=300, S2=300, Dv=64), None),
    ("d192_dv64_gqa_fp16_band", inputs.sized(W["causal_s8192_d192_dv128"], dtype="fp16", Dv=64, N1=4, N2=2, S1=260,
                                             S2=390, mask_mode=2, win_left=100, win_right=30), None),
    ("d192_dv192_causal", inputs.sized(W["causal_s8192_d192_dv128"], Dv=192, N1=2, N2=2, S1=300, S2=300), None),
    ("d192_dv192_tnd_gqa", inputs.sized(W["varlen_window_fp16_d128"], D=192, Dv=192, B=3, N1=4, N2=2, win_left=64),
     ([70, 1, 200], None)),
    ("d96_causal", inputs.sized(W["causal_b2_s2048_d128"], B=1, N1=2, N2=2, S1=300, S2=300, D=96, Dv=96), None),
    ("d80_dv48_bnsd_band", inputs.sized(W["mha_s128_d64"], layout="BNSD", S1=190, S2=250, D=80, Dv=48,
                                        mask_mode=2, win_left=20, win_right=7), None),
    ("d40_dv8_dense", inputs.sized(W["mha_s128_d64"], S1=150, S2=200, D=40, Dv=8), None),
    ("d160_dv136_tnd_fp16", inputs.sized(W["varlen_window_fp16_d128"], D=160, Dv=136, B=3, N1=4, N2=2, win_left=64),
     ([200, 33, 129], None)),
    ("d136_dv72_gqa_causal", inputs.sized(W["gqa_causal_s4096_d128"], D=136, Dv=72, N1=4, N2=2, S1=260, S2=260,
                                          dout_std=1.0), None),
]


def _pad(d):
    return 64 if d <= 64 else 128 if d <= 128 else 192


def atomic_unsupported(w):
    """The atomic mode's fused kernel has no room in tensor memory for D and Dv both above 128."""
    return _pad(w.D) == 192 and _pad(w.Dv) == 192


@pytest.mark.parametrize("dq_mode", ["separate", "atomic"])
@pytest.mark.parametrize("name,w,lens", SMALL, ids=[c[0] for c in SMALL])
def test_small_elementwise(name, w, lens, dq_mode):
    pb = inputs.make_problem(w, *(lens or ()))
    ref = tl.full_reference(pb)
    if dq_mode == "atomic" and atomic_unsupported(w):
        with pytest.raises(F.FabwdError) as ei:
            tl.run_gpu(pb, ref, dq_mode=dq_mode)
        assert ei.value.status == F.FABWD_ERR_UNSUPPORTED
        return
    dq, dk, dv, sf = tl.run_gpu(pb, ref, dq_mode=dq_mode)
    check_all(pb, ref, dq, dk, dv, sf)


def test_page_example_shapes_gqa_fp16():
    # The BSND GQA call of [FAG] §4.8: B=2, S1=S2=128, N1=8, N2=2, D=Dv=128, fp16, dense.
    w = inputs.Workload("page_example", "BSND", "fp16", B=2, N1=8, N2=2, D=128, Dv=128, S1=128, S2=128,
                        softmax_scale=1.0 / math.sqrt(128), seed=7)
    pb = inputs.make_problem(w)
    ref = tl.full_reference(pb)
    dq, dk, dv, sf = tl.run_gpu(pb, ref)
    assert dq.shape == pb.q.shape and dk.shape == pb.k.shape and dv.shape == pb.v.shape
    assert dq.dtype == pb.q.dtype == dk.dtype == dv.dtype
    check_all(pb, ref, dq, dk, dv, sf)


@pytest.mark.parametrize("dq_mode", ["separate", "atomic"])
def test_determinism_and_workspace_reuse(dq_mode):
    w = inputs.sized(W["gqa_causal_s4096_d128"], N1=4, N2=2, S1=700, S2=700, dout_std=1.0)
    pb = inputs.make_problem(w)
    ref = tl.forward_inputs(pb)
    dev = torch.device("cuda")
    args = [t.to(dev) for t in (pb.q, pb.k, pb.v, pb.dout, ref.attn_out, ref.lse)]
    dq1, dk1, dv1 = api.flash_attn_grad(*args, mask_mode=1, dq_mode=dq_mode, check_status=True)
    dq2, dk2, dv2 = api.flash_attn_grad(*args, mask_mode=1, dq_mode=dq_mode, check_status=True)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)   # no atomics on dK/dV in either mode
    if dq_mode == "separate":
        assert torch.equal(dq1, dq2)                          # one CTA sums each dQ element in order
    else:
        assert (dq1.float() - dq2.float()).abs().max().item() <= 1e-2 * dq1.float().abs().max().item()


def test_modes_agree():
    w = inputs.sized(W["varlen_window_fp16_d128"], B=3, N1=4, N2=2, win_left=100)
    pb = inputs.make_problem(w, [300, 17, 260])
    ref = tl.full_reference(pb)
    outs = {m: tl.run_gpu(pb, ref, dq_mode=m) for m in ("atomic", "separate")}
    for i, name in enumerate(("dq", "dk", "dv")):
        tl.assert_close(f"{name} atomic vs separate", outs["atomic"][i], inputs.to_f64(outs["separate"][i]))


@pytest.mark.parametrize("case", ["gqa_causal_ragged", "band_bnsd_d64", "tnd_bf16_gqa_dense", "d192_dv128_gqa_fp16_band"])
def test_one_grid_equals_separate_launches(case):
    # fabwd_run launches the dK/dV and dQ CTAs of the separate mode as one grid; launched on
    # their own (fabwd_run_main, then fabwd_run_dq) the same CTA code must give identical bits
    name, w, lens = next(c for c in SMALL if c[0] == case)
    pb = inputs.make_problem(w, *(lens or ()))
    ref = tl.forward_inputs(pb)
    dev = torch.device("cuda")
    d = lambda x: x.to(dev)
    cu_q = cu_kv = None
    extra = {}
    if w.layout == "TND":
        cu_q, cu_kv = d(torch.from_numpy(pb.cu_seqlens_q)), d(torch.from_numpy(pb.cu_seqlens_kv))
        extra = dict(max_seqlen_q=pb.S1, max_seqlen_kv=pb.S2)
    ins = [d(t) for t in (pb.q, pb.k, pb.v, pb.dout, ref.attn_out, ref.lse)]
    outs = []
    for one_grid in (True, False):
        dq, dk, dv = (torch.full_like(ins[i], 3.0) for i in (0, 1, 2))
        p = api.make_params(*ins, dq, dk, dv, cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv, layout=w.layout,
                            dq_mode="separate", **tl.mask_kwargs(w), **extra)
        n = F.fabwd_workspace_size(p)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
        st = torch.cuda.current_stream().cuda_stream
        F.fabwd_preprocess(p, ws.data_ptr(), ws.numel(), st)
        if one_grid:
            F.fabwd_run(p, ws.data_ptr(), ws.numel(), st)
        else:
            F.fabwd_run_main(p, ws.data_ptr(), ws.numel(), st)
            F.fabwd_run_dq(p, ws.data_ptr(), ws.numel(), st)
        s_, bits = F.fabwd_read_device_status(ws.data_ptr(), ws.numel(), st)
        assert s_ == F.FABWD_OK, hex(bits)
        outs.append((dq, dk, dv))
    for name, a, b in zip(("dq", "dk", "dv"), outs[0], outs[1]):
        assert torch.equal(a, b), name


def _oracle_stats(pb):
    """(row maximum, row sum) of the fp64 forward per head, in softmax_lse's layout."""
    w = pb.w
    q, k, v = (inputs.to_f64(t) for t in (pb.q, pb.k, pb.v))
    scale = orc.resolve_scale(w.softmax_scale, w.D)
    G = w.N1 // w.N2
    if w.layout == "TND":
        m, l = np.zeros((w.N1, pb.T1)), np.zeros((w.N1, pb.T1))
        cu_q, cu_k = pb.cu_seqlens_q, pb.cu_seqlens_kv
        for s_ in range(w.B):
            rq, rk = slice(int(cu_q[s_]), int(cu_q[s_ + 1])), slice(int(cu_k[s_]), int(cu_k[s_ + 1]))
            ok = orc.visible(rq.stop - rq.start, rk.stop - rk.start, w.mask_mode, w.win_left, w.win_right)
            for n1 in range(w.N1):
                m[n1, rq], l[n1, rq] = orc.forward_stats_head(q[rq, n1], k[rk, n1 // G], v[rk, n1 // G], scale, ok)
    else:
        m, l = np.zeros((w.B, w.N1, pb.S1)), np.zeros((w.B, w.N1, pb.S1))
        ok = orc.visible(pb.S1, pb.S2, w.mask_mode, w.win_left, w.win_right)
        for b in range(w.B):
            for n1 in range(w.N1):
                m[b, n1], l[b, n1] = orc.forward_stats_head(q[b, :, n1], k[b, :, n1 // G], v[b, :, n1 // G], scale, ok)
    return m.astype(np.float32), l.astype(np.float32)


@pytest.mark.parametrize("stride", [1, 8])
@pytest.mark.parametrize("case", ["gqa_causal_ragged", "tnd_fp16_window"])
def test_max_sum_statistics_in_place_of_lse(case, stride):
    # the forward's (row maximum, row sum) pair instead of softmax_lse, optionally with each row's
    # value repeated `stride` times (the (..., 8) layout of the LaserAttentionGrad and
    # FusedFloydAttentionGrad pages); rows without a visible key carry (-inf, 0)
    name, w, lens = next(c for c in SMALL if c[0] == case)
    pb = inputs.make_problem(w, *(lens or ()))
    ref = tl.full_reference(pb)
    m, l = _oracle_stats(pb)
    if stride > 1:
        m, l = np.repeat(m[..., None], stride, axis=-1), np.repeat(l[..., None], stride, axis=-1)
    dev = torch.device("cuda")
    d = lambda x: x.to(dev)
    kw = dict(layout_q=w.layout, layout_kv=w.layout, layout_out=w.layout, check_status=True, **tl.mask_kwargs(w))
    if w.layout == "TND":
        kw.update(cu_seqlens_q=d(torch.from_numpy(pb.cu_seqlens_q)), cu_seqlens_kv=d(torch.from_numpy(pb.cu_seqlens_kv)),
                  max_seqlen_q=pb.S1, max_seqlen_kv=pb.S2)
    ins = [d(t) for t in (pb.q, pb.k, pb.v, pb.dout, ref.attn_out)]
    dq, dk, dv = api.flash_attn_grad(*ins, None, softmax_max=d(torch.from_numpy(m)), softmax_sum=d(torch.from_numpy(l)),
                                     **kw)
    tl.assert_close("dq", dq.cpu(), ref.dq)
    tl.assert_close("dk", dk.cpu(), ref.dk)
    tl.assert_close("dv", dv.cpu(), ref.dv)


# ---------------------------------------------------------------------------------------------
# degenerate and edge cases
# ---------------------------------------------------------------------------------------------


def _gpu_call(q, k, v, do, y, lse, **kw):
    dev = torch.device("cuda")
    return api.flash_attn_grad(*(t.to(dev) if t is not None else None for t in (q, k, v, do, y, lse)),
                               check_status=True, **kw)


def test_single_key_closed_form_on_gpu():
    # one key: P == 1 and dS = P (dY·v − dY·Y) vanishes up to the bf16 rounding of Y (attn_out),
    # so dQ and dK are tiny next to dV = Σ_i dY_i
    w = inputs.sized(W["mha_s128_d64"], S1=300, S2=1, N1=2, N2=2)
    pb = inputs.make_problem(w)
    ref = tl.full_reference(pb)
    dq, dk, dv, sf = tl.run_gpu(pb, ref)
    scale = dv.float().abs().max().item()
    assert dq.float().abs().max().item() <= 1e-4 * scale and dk.float().abs().max().item() <= 1e-4 * scale
    tl.assert_close("dv", dv, ref.dv)
    want = inputs.to_f64(pb.dout).sum(axis=1)[0]          # [N, Dv]: Σ_i dY_i per head
    tl.assert_close("dv closed form", inputs.to_f64(dv)[0, 0], want)


def test_s2_zero_gives_zero_dq():
    w = inputs.sized(W["mha_s128_d64"], S1=130, S2=0)
    pb = inputs.make_problem(w)
    lse = torch.full((1, 2, 130), float("inf"))
    dq, dk, dv = _gpu_call(pb.q, pb.k, pb.v, pb.dout, torch.zeros_like(pb.dout), lse)
    torch.cuda.synchronize()
    assert dk.numel() == 0 and dv.numel() == 0 and dq.abs().max().item() == 0


def test_s1_zero_gives_zero_dk_dv():
    w = inputs.sized(W["mha_s128_d64"], S1=0, S2=200)
    pb = inputs.make_problem(w)
    dq, dk, dv = _gpu_call(pb.q, pb.k, pb.v, pb.dout, pb.dout.clone(), torch.zeros(1, 2, 0), mask_mode=1)
    torch.cuda.synchronize()
    assert dq.numel() == 0 and dk.abs().max().item() == 0 and dv.abs().max().item() == 0


def test_tnd_all_sequences_empty_but_one():
    w = inputs.sized(W["varlen_window_fp16_d128"], B=4, N1=2, N2=2)
    pb = inputs.make_problem(w, [0, 0, 5, 0], [0, 3, 7, 0])
    ref = tl.full_reference(pb)
    dq, dk, dv, sf = tl.run_gpu(pb, ref)
    check_all(pb, ref, dq, dk, dv, sf)


def test_rows_without_keys_get_zero_dq():
    # causal with S1 > S2: the first S1 - S2 rows see no key (lse = +inf)
    w = inputs.sized(W["causal_b2_s2048_d128"], B=1, N1=2, N2=2, S1=260, S2=100)
    pb = inputs.make_problem(w)
    ref = tl.full_reference(pb)
    assert np.isinf(ref.lse.numpy()[0, :, :160]).all()
    dq, dk, dv, sf = tl.run_gpu(pb, ref)
    assert dq[0, :160].abs().max().item() == 0
    check_all(pb, ref, dq, dk, dv, sf)


def test_bad_cu_seqlens_reported_not_faulted():
    w = inputs.sized(W["varlen_window_fp16_d128"], B=2, N1=2, N2=2)
    pb = inputs.make_problem(w, [100, 60])
    ref = tl.forward_inputs(pb)
    dev = torch.device("cuda")
    bad = torch.tensor([0, 100, 170], dtype=torch.int32, device=dev)   # ends beyond T = 160
    args = [t.to(dev) for t in (pb.q, pb.k, pb.v, pb.dout, ref.attn_out, ref.lse)]
    with pytest.raises(F.FabwdError) as ei:
        api.flash_attn_grad(*args, cu_seqlens_q=bad, cu_seqlens_kv=bad, max_seqlen_q=128, max_seqlen_kv=128,
                            layout_q="TND", layout_kv="TND", layout_out="TND", check_status=True)
    assert ei.value.status == F.FABWD_ERR_DEVICE
    # the context stays usable: a correct call right after succeeds
    cu = torch.from_numpy(pb.cu_seqlens_q).to(dev)
    api.flash_attn_grad(*args, cu_seqlens_q=cu, cu_seqlens_kv=cu, layout_q="TND", layout_kv="TND",
                        layout_out="TND", mask_mode=1, win_left=1024, win_right=0, check_status=True)


def test_decreasing_cu_seqlens_reported_not_faulted():
    # a sequence with a negative span owns no unit of the varlen grids: the backward's preprocess
    # and the forward's first CTA still report it; the rows the other sequences cover stay in range
    w = inputs.sized(W["varlen_window_fp16_d128"], B=3, N1=2, N2=2)
    pb = inputs.make_problem(w, [100, 0, 60])
    ref = tl.forward_inputs(pb)
    dev = torch.device("cuda")
    bad = torch.tensor([0, 100, 40, 160], dtype=torch.int32, device=dev)
    args = [t.to(dev) for t in (pb.q, pb.k, pb.v, pb.dout, ref.attn_out, ref.lse)]
    kw = dict(cu_seqlens_q=bad, cu_seqlens_kv=bad, max_seqlen_q=128, max_seqlen_kv=128)
    with pytest.raises(F.FabwdError) as ei:
        api.flash_attn_grad(*args, layout_q="TND", layout_kv="TND", layout_out="TND", check_status=True, **kw)
    assert ei.value.status == F.FABWD_ERR_DEVICE
    with pytest.raises(F.FabwdError) as ei:
        api.flash_attn_forward(*args[:3], layout="TND", check_status=True, **kw)
    assert ei.value.status == F.FABWD_ERR_DEVICE
    # the context stays usable
    cu = torch.from_numpy(pb.cu_seqlens_q).to(dev)
    api.flash_attn_forward(*args[:3], cu_seqlens_q=cu, cu_seqlens_kv=cu, layout="TND", check_status=True)


def test_timeout_injection_returns_status_and_context_survives():
    w = inputs.sized(W["gqa_causal_s4096_d128"], N1=4, N2=2, S1=256, S2=256, dout_std=1.0)
    pb = inputs.make_problem(w)
    ref = tl.full_reference(pb)
    old = F.fabwd_set_wait_limit_ns(20_000_000)  # 20 ms
    try:
        F.fabwd_debug_inject_timeout(True)
        with pytest.raises(F.FabwdError) as ei:
            _gpu_call(pb.q, pb.k, pb.v, pb.dout, ref.attn_out, ref.lse, mask_mode=1)
        assert ei.value.status == F.FABWD_ERR_TIMEOUT
    finally:
        F.fabwd_debug_inject_timeout(False)
        F.fabwd_set_wait_limit_ns(old)
    dq, dk, dv, sf = tl.run_gpu(pb, ref)   # same process, same context: still correct
    check_all(pb, ref, dq, dk, dv, sf)


# ---------------------------------------------------------------------------------------------
# full-size workloads, every element
# ---------------------------------------------------------------------------------------------


FULL = [(name, "auto") for name in ("mha_s128_d64", "causal_b2_s2048_d128", "gqa_causal_s4096_d128",
                                    "varlen_window_fp16_d128", "causal_s8192_d192_dv128")]
FULL.append(("causal_b2_s2048_d128", "atomic"))


@pytest.mark.parametrize("name,dq_mode", FULL, ids=[f"{n}-{m}" for n, m in FULL])
def test_full_size_elementwise(name, dq_mode, parity_report):
    # The workload at its measured size, in the launch configuration the bench times (the
    # library's default dQ mode, plus the atomic mode once): every element of dq, dk, dv and every
    # sfmg row against the fp64 oracle, computed per kv-head group in a pool of processes.
    w = W[name]
    pb = inputs.make_problem(w)
    ref = tl.full_reference_parallel(pb)
    dq, dk, dv, sf = tl.run_gpu(pb, ref, dq_mode=dq_mode)
    errs = check_all(pb, ref, dq, dk, dv, sf)
    errs["sfmg"] = tl.errors(sf, ref.sfmg)
    parity_report(f"{name} [{dq_mode}]", errs)


def test_long_sequence_elementwise(parity_report):
    # twice the longest measured sequence (128 key and query blocks per head, GQA G = 2, causal):
    # every element against the oracle
    w = inputs.sized(W["causal_b2_s2048_d128"], B=1, N1=2, N2=1, S1=16384, S2=16384, D=64, Dv=64)
    pb = inputs.make_problem(w)
    ref = tl.full_reference_parallel(pb)
    dq, dk, dv, sf = tl.run_gpu(pb, ref)
    errs = check_all(pb, ref, dq, dk, dv, sf)
    errs["sfmg"] = tl.errors(sf, ref.sfmg)
    parity_report("causal S=16384 D=64 G=2 [auto]", errs)


def test_head_dim_not_multiple_of_8_is_unsupported():
    q = torch.zeros(1, 256, 2, 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(F.FabwdError) as ei:
        api.flash_attn_grad(q, q, q, q, q, torch.zeros(1, 2, 256, device="cuda"), mask_mode=1)
    assert ei.value.status == F.FABWD_ERR_UNSUPPORTED
