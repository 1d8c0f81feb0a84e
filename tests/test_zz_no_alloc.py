"""The allocation-free entry point, checked against the caller-workspace path.

fabwd_run_static_workspace serves callers that cannot call cudaMalloc when they run the
backward: code under a host framework that owns all device memory through its own pool, or a
loop whose rules forbid allocation after start-up.  They pass inputs and outputs only; the
scratch is a fixed 64 MiB array inside the library.  This file is collected last so that a run
stopping at the first failure has already run every other test; it also passes on its own in a
fresh process.
"""
import ctypes

import pytest
import torch

from attention_backward_fabwd_gb300 import api, build, fabwd as F, inputs

import fabwd_testlib as tl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return F.lib()


def test_static_workspace_matches_caller_workspace_twice(lib):
    w = inputs.sized(inputs.WORKLOADS["gqa_causal_s4096_d128"], N1=4, N2=2, S1=300, S2=300, dout_std=1.0)
    pb = inputs.make_problem(w)
    ref = tl.forward_inputs(pb)
    dev = torch.device("cuda")
    q, k, v, do, y, lse = (t.to(dev) for t in (pb.q, pb.k, pb.v, pb.dout, ref.attn_out, ref.lse))
    # the existing entry points, with a workspace allocated by the caller
    dq0, dk0, dv0 = api.flash_attn_grad(q, k, v, do, y, lse, mask_mode=1, check_status=True)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # the second call runs on the array the first one left behind
        dq, dk, dv = torch.full_like(q, 7.0), torch.full_like(k, 7.0), torch.full_like(v, 7.0)
        p = api.make_params(q, k, v, do, y, lse, dq, dk, dv, mask_mode=1)
        status = lib.fabwd_run_static_workspace(ctypes.byref(p), ctypes.c_void_p(stream))
        assert status == F.FABWD_OK, F.status_string(status)
        torch.cuda.synchronize()
        for name, got, want in (("dq", dq, dq0), ("dk", dk, dk0), ("dv", dv, dv0)):
            tl.assert_close(f"{name} (call {call + 1})", got.cpu(), inputs.to_f64(want.cpu()))


def test_static_workspace_refuses_oversized_problems(lib):
    # The pointers below are placeholders that must never reach a kernel, so the problem is
    # chosen to need far more than the 64 MiB array in every dQ mode (the lse/sfmg rows alone are
    # 2 x 4 x 64 x 65536 x 4 B = 128 MiB), and the size is checked on the host before the call.
    p = F.fabwd_params()
    p.dtype, p.layout = F.FABWD_BF16, F.FABWD_BSND
    p.B, p.S1, p.S2, p.N1, p.N2, p.D, p.Dv = 4, 65536, 65536, 64, 8, 128, 128
    p.mask_mode, p.win_left, p.win_right = 1, -1, -1
    for name in ("q", "k", "v", "dout", "attn_out", "softmax_lse", "dq", "dk", "dv"):
        setattr(p, name, 0x10000)
    for mode in (F.FABWD_DQ_AUTO, F.FABWD_DQ_ATOMIC, F.FABWD_DQ_SEPARATE):
        p.dq_mode = mode
        need = F.fabwd_workspace_size(p)
        assert need >= 96 << 20, "the placeholder pointers would reach a kernel"
        assert lib.fabwd_run_static_workspace(ctypes.byref(p), None) == F.FABWD_ERR_WORKSPACE
