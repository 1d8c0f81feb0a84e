"""The allocation-free entry point, checked against the caller-workspace path.

fabwd_run_static_workspace serves callers that cannot call cudaMalloc when they run the
backward: code under a host framework that owns all device memory through its own pool, or a
loop whose rules forbid allocation after start-up.  They pass inputs and outputs only; the
scratch is a fixed array inside the library (fabwd_static_workspace_capacity bytes).  This file
is collected last so that a run stopping at the first failure has already run every other test;
it also passes on its own in a fresh process.
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


def _static_call(lib, ins, mode):
    q, k, v = ins[:3]
    dq, dk, dv = torch.full_like(q, 7.0), torch.full_like(k, 7.0), torch.full_like(v, 7.0)
    p = api.make_params(*ins, dq, dk, dv, mask_mode=1, dq_mode=mode)
    stream = torch.cuda.current_stream().cuda_stream
    status = lib.fabwd_run_static_workspace(ctypes.byref(p), ctypes.c_void_p(stream))
    assert status == F.FABWD_OK, F.status_string(status)
    s_, bits = F.fabwd_static_workspace_status(stream)
    assert s_ == F.FABWD_OK, hex(bits)
    return dq, dk, dv


def _inputs(S):
    w = inputs.sized(inputs.WORKLOADS["gqa_causal_s4096_d128"], N1=4, N2=2, S1=S, S2=S, dout_std=1.0)
    pb = inputs.make_problem(w)
    ref = tl.forward_inputs(pb)
    dev = torch.device("cuda")
    return [t.to(dev) for t in (pb.q, pb.k, pb.v, pb.dout, ref.attn_out, ref.lse)]


@pytest.mark.parametrize("mode", ["separate", "atomic"])
def test_static_workspace_matches_caller_workspace_twice(lib, mode):
    ins = _inputs(300)
    # the existing entry points, with a workspace allocated by the caller
    dq0, dk0, dv0 = api.flash_attn_grad(*ins, mask_mode=1, dq_mode=mode, check_status=True)
    # a larger problem first leaves the shared array dirty where the next call keeps its scratch
    # (in atomic mode its fp32 dq accumulator, which the kernels must clear before summing)
    _static_call(lib, _inputs(700), mode)
    for call in range(2):  # the second call also runs on what the first one left behind
        dq, dk, dv = _static_call(lib, ins, mode)
        torch.cuda.synchronize()
        for name, got, want in (("dq", dq, dq0), ("dk", dk, dk0), ("dv", dv, dv0)):
            tl.assert_close(f"{name} (call {call + 1})", got.cpu(), inputs.to_f64(want.cpu()))


def test_static_workspace_refuses_oversized_problems(lib):
    # Every device pointer is left NULL: a problem that needs more than the array is refused by
    # the size check, and were that check ever skipped, the host's pointer check would refuse the
    # call (FABWD_ERR_NULLPTR) before any kernel could run.
    cap = F.fabwd_static_workspace_capacity()
    assert cap == 64 << 20
    p = F.fabwd_params()
    p.dtype, p.layout = F.FABWD_BF16, F.FABWD_BSND
    p.B, p.S1, p.S2, p.N1, p.N2, p.D, p.Dv = 4, 65536, 65536, 64, 8, 128, 128
    p.mask_mode, p.win_left, p.win_right = 1, -1, -1
    for mode in (F.FABWD_DQ_AUTO, F.FABWD_DQ_ATOMIC, F.FABWD_DQ_SEPARATE):
        p.dq_mode = mode
        assert F.fabwd_workspace_size(p) > cap
        assert lib.fabwd_run_static_workspace(ctypes.byref(p), None) == F.FABWD_ERR_WORKSPACE
    # a problem that fits but has no buffers: refused on the host as well
    p.B, p.S1, p.S2, p.N1, p.N2 = 1, 256, 256, 2, 2
    assert F.fabwd_workspace_size(p) <= cap
    assert lib.fabwd_run_static_workspace(ctypes.byref(p), None) == F.FABWD_ERR_NULLPTR
