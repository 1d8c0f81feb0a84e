"""GPU forward (fabwd_forward): attn_out and softmax_lse against the fp64 oracle forward, and
the forward feeding the backward.

attn_out within the output tolerance of the backward's outputs (relative L2 <= 1e-2, max-abs
<= 2e-2 · max|ref|); lse within 1e-4 + 1e-5·|lse| wherever it is finite, +inf exactly where the
row sees no key.
"""
import math

import numpy as np
import pytest
import torch

from attention_backward_fabwd_gb300 import api, fabwd as F, inputs
from oracle import fabwd_oracle as orc

import fabwd_testlib as tl
from test_parity_gpu import SMALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_backward_fabwd_gb300 import build

    build.build()
    F.lib()


def gpu_forward(pb):
    w = pb.w
    dev = torch.device("cuda")
    d = lambda x: x.to(dev)
    q, k, v = d(pb.q), d(pb.k), d(pb.v)
    cu_q = cu_kv = None
    extra = {}
    if w.layout == "TND":
        cu_q, cu_kv = d(torch.from_numpy(pb.cu_seqlens_q)), d(torch.from_numpy(pb.cu_seqlens_kv))
        extra = dict(max_seqlen_q=pb.S1, max_seqlen_kv=pb.S2)
        lse_shape = (w.N1, pb.T1)
    else:
        lse_shape = (w.B, w.N1, pb.S1)
    y = torch.full(pb.dout.shape, 7.0, dtype=q.dtype, device=dev)
    lse = torch.full(lse_shape, 7.0, dtype=torch.float32, device=dev)
    p = api.make_params(q, k, v, q, y, lse, q, k, v, cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv, layout=w.layout,
                        **tl.mask_kwargs(w), **extra)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream().cuda_stream
    F.fabwd_forward(p, y.data_ptr(), lse.data_ptr(), ws.data_ptr(), 256, st)
    s, bits = F.fabwd_read_device_status(ws.data_ptr(), 256, st)
    assert s == F.FABWD_OK, hex(bits)
    return y.cpu(), lse.cpu()


def check_lse(got, want):
    got = got.numpy().astype(np.float64)
    want = np.asarray(want, np.float64)
    inf_w = np.isinf(want)
    assert np.array_equal(np.isinf(got), inf_w), "rows without a visible key must get +inf, and only they"
    assert (got[inf_w] > 0).all()
    fin = ~inf_w
    err = np.abs(got[fin] - want[fin])
    assert (err <= 1e-4 + 1e-5 * np.abs(want[fin])).all(), f"max lse error {err.max()}"


@pytest.mark.parametrize("name,w,lens", SMALL, ids=[c[0] for c in SMALL])
def test_forward_matches_oracle(name, w, lens):
    pb = inputs.make_problem(w, *(lens or ()))
    y_ref, lse_ref = orc.forward(*(inputs.to_f64(t) for t in (pb.q, pb.k, pb.v)), **tl.oracle_kwargs(pb))
    y, lse = gpu_forward(pb)
    tl.assert_close("attn_out", y, y_ref)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("case", ["gqa_causal_ragged", "tnd_fp16_window", "d192_dv128_causal"])
def test_forward_then_backward(case):
    # the library's own forward feeding its backward: gradients within tolerance of the oracle's
    name, w, lens = next(c for c in SMALL if c[0] == case)
    pb = inputs.make_problem(w, *(lens or ()))
    ref = tl.full_reference(pb)
    y, lse = gpu_forward(pb)
    dev = torch.device("cuda")
    d = lambda x: x.to(dev)
    kw = dict(layout_q=w.layout, layout_kv=w.layout, layout_out=w.layout, check_status=True, **tl.mask_kwargs(w))
    if w.layout == "TND":
        kw.update(cu_seqlens_q=d(torch.from_numpy(pb.cu_seqlens_q)), cu_seqlens_kv=d(torch.from_numpy(pb.cu_seqlens_kv)),
                  max_seqlen_q=pb.S1, max_seqlen_kv=pb.S2)
    dq, dk, dv = api.flash_attn_grad(d(pb.q), d(pb.k), d(pb.v), d(pb.dout), d(y), d(lse), **kw)
    tl.assert_close("dq", dq.cpu(), ref.dq)
    tl.assert_close("dk", dk.cpu(), ref.dk)
    tl.assert_close("dv", dv.cpu(), ref.dv)


def test_forward_without_keys():
    w = inputs.sized(inputs.WORKLOADS["mha_s128_d64"], S1=70, S2=0)
    pb = inputs.make_problem(w)
    y, lse = gpu_forward(pb)
    assert (y.float() == 0).all() and torch.isinf(lse).all() and (lse > 0).all()


@pytest.mark.parametrize("case", ["gqa_causal_ragged", "tnd_fp16_window"])
def test_api_forward_equals_c_forward(case):
    # api.flash_attn_forward is argument marshalling over fabwd_forward: bit-identical results
    name, w, lens = next(c for c in SMALL if c[0] == case)
    pb = inputs.make_problem(w, *(lens or ()))
    y0, lse0 = gpu_forward(pb)
    dev = torch.device("cuda")
    d = lambda x: x.to(dev)
    kw = dict(layout=w.layout, check_status=True, **tl.mask_kwargs(w))
    if w.layout == "TND":
        kw.update(cu_seqlens_q=d(torch.from_numpy(pb.cu_seqlens_q)), cu_seqlens_kv=d(torch.from_numpy(pb.cu_seqlens_kv)),
                  max_seqlen_q=pb.S1, max_seqlen_kv=pb.S2)
    y, lse = api.flash_attn_forward(d(pb.q), d(pb.k), d(pb.v), **kw)
    assert torch.equal(y.cpu(), y0)
    assert torch.equal(lse.cpu(), lse0)


@pytest.mark.parametrize("case", ["dense_s1_lt_s2", "causal_b2_s384", "fp16_dense_d64", "band_wide"])
def test_forward_growing_maximum(case):
    # Keys scaled up along the sequence (x1 at the first key to x6 at the last), so a row's
    # maximum score keeps rising from key block to key block by more than 8 in log2 units: the
    # running reference moves after the first tile, O and the row sum are rescaled and P is formed
    # again from the kept scores.
    name, w, lens = next(c for c in SMALL if c[0] == case)
    pb = inputs.make_problem(w, *(lens or ()))
    k = pb.k.double()
    seq_axis = 2 if w.layout == "BNSD" else 1
    ramp = 1.0 + 5.0 * torch.arange(k.shape[seq_axis], dtype=torch.float64) / max(k.shape[seq_axis] - 1, 1)
    shape = [1] * k.dim()
    shape[seq_axis] = -1
    pb.k = (k * ramp.view(shape)).to(pb.k.dtype).contiguous()
    y_ref, lse_ref = orc.forward(*(inputs.to_f64(t) for t in (pb.q, pb.k, pb.v)), **tl.oracle_kwargs(pb))
    y, lse = gpu_forward(pb)
    tl.assert_close("attn_out", y, y_ref)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("case", ["causal_b2_s384", "band_bnsd_d64", "tnd_fp16_window", "d192_dv128_causal"])
def test_forward_negative_scale(case):
    # a negative softmax_scale: the row maximum of scale·S is scale times the row minimum of S,
    # hidden keys included in neither
    name, w, lens = next(c for c in SMALL if c[0] == case)
    w = inputs.sized(w, softmax_scale=-0.7 / math.sqrt(w.D))
    pb = inputs.make_problem(w, *(lens or ()))
    y_ref, lse_ref = orc.forward(*(inputs.to_f64(t) for t in (pb.q, pb.k, pb.v)), **tl.oracle_kwargs(pb))
    y, lse = gpu_forward(pb)
    tl.assert_close("attn_out", y, y_ref)
    check_lse(lse, lse_ref)
