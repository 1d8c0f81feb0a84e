"""CPU-only checks of the C ABI boundary and the host logic (no CUDA compute call is made).

* libfabwd builds for sm_103a and exports every function include/fabwd.h declares;
* the host validation returns the documented status for each broken rule of the page
  "CANN ops-transformer FlashAttnGrad 算子详解" (discosf.com/news/4863418), §4.6 constraints,
  before anything is enqueued;
* workspace sizing, the torch-facing argument handling and the bench's work counts.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest
import torch

from attention_backward_fabwd_gb300 import api, build, fabwd as F, inputs
from oracle import fabwd_oracle as orc


@pytest.fixture(scope="module")
def lib():
    build.build()
    return F.lib()


def base_params(**kw):
    p = F.fabwd_params()
    p.dtype, p.layout = F.FABWD_BF16, F.FABWD_BSND
    p.B, p.S1, p.S2, p.N1, p.N2, p.D, p.Dv = 2, 300, 300, 4, 2, 128, 128
    p.T1, p.T2 = 0, 0
    p.softmax_scale, p.mask_mode, p.win_left, p.win_right = 0.0, 1, -1, -1
    fake = 0x10000  # aligned dummy addresses: never dereferenced by the host checks
    for name in ("q", "k", "v", "dout", "attn_out", "softmax_lse", "dq", "dk", "dv"):
        setattr(p, name, fake)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def ws_size(p):
    n = ctypes.c_size_t(0)
    s = F.lib().fabwd_workspace_size(ctypes.byref(p), ctypes.byref(n))
    return s, n.value


def test_library_exports_every_declared_symbol(lib):
    declared = F.declared_functions()
    assert len(declared) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [f for f in declared if f not in exported]
    assert not missing, f"declared but not exported: {missing}"
    for f in declared:
        assert hasattr(lib, f)


def test_version_and_status_strings(lib):
    assert F.fabwd_version() >= 100
    for code in range(8):
        assert F.status_string(code) and F.status_string(code) != "unknown status"
    assert F.status_string(99) == "unknown status"


def test_workspace_size_formula(lib):
    p = base_params(dq_mode=F.FABWD_DQ_ATOMIC)
    s, n = ws_size(p)
    assert s == F.FABWD_OK
    S1p = 384
    rows = 2 * 4 * S1p * 4
    r256 = lambda x: (x + 255) // 256 * 256
    assert n == 256 + 2 * r256(rows) + r256(2 * 300 * 4 * 128 * 4)
    lay = F.fabwd_workspace_layout(p)
    assert lay["row_stride"] == S1p and lay["lse2"] == 256 and lay["sfmg"] == 256 + r256(rows)
    assert lay["dq_accum"] == lay["sfmg"] + r256(rows)
    # separate dQ mode (auto's choice) keeps no fp32 accumulator
    assert ws_size(base_params(dq_mode=F.FABWD_DQ_SEPARATE)) == (F.FABWD_OK, 256 + 2 * r256(rows))
    assert ws_size(base_params(dq_mode=F.FABWD_DQ_AUTO)) == (F.FABWD_OK, 256 + 2 * r256(rows))


def test_resolve_dq_mode(lib):
    for asked, got in ((F.FABWD_DQ_ATOMIC, F.FABWD_DQ_ATOMIC), (F.FABWD_DQ_SEPARATE, F.FABWD_DQ_SEPARATE),
                       (F.FABWD_DQ_AUTO, F.FABWD_DQ_SEPARATE)):
        assert F.fabwd_resolve_dq_mode(base_params(dq_mode=asked)) == got
        assert F.fabwd_resolve_dq_mode(base_params(dq_mode=asked, D=192)) == got
    with pytest.raises(F.FabwdError):
        F.fabwd_resolve_dq_mode(base_params(dq_mode=3))


@pytest.mark.parametrize("change,code", [
    (dict(dtype=2), F.FABWD_ERR_INVALID),
    (dict(layout=3), F.FABWD_ERR_INVALID),
    (dict(B=0), F.FABWD_ERR_INVALID),
    (dict(B=65536), F.FABWD_ERR_INVALID),            # B in (0, 65536)
    (dict(N1=3), F.FABWD_ERR_INVALID),               # N1 % N2 != 0
    (dict(N2=0), F.FABWD_ERR_INVALID),
    (dict(Dv=192, D=128), F.FABWD_ERR_INVALID),      # Dv > D
    (dict(D=256, Dv=128), F.FABWD_ERR_INVALID),      # D > 192
    (dict(D=0), F.FABWD_ERR_INVALID),
    (dict(S1=-1), F.FABWD_ERR_INVALID),
    (dict(mask_mode=3), F.FABWD_ERR_INVALID),
    (dict(mask_mode=0, win_left=10), F.FABWD_ERR_INVALID),   # dense preset takes no window
    (dict(mask_mode=1, win_left=-2), F.FABWD_ERR_INVALID),
    (dict(softmax_scale=float("nan")), F.FABWD_ERR_INVALID),
    (dict(cu_seqlens_q=0x20000, cu_seqlens_kv=0x20000), F.FABWD_ERR_INVALID),  # non-TND with cu_seqlens
    (dict(layout=F.FABWD_TND), F.FABWD_ERR_INVALID),                            # TND without cu_seqlens
    (dict(D=100, Dv=96), F.FABWD_ERR_UNSUPPORTED),   # valid per the statement; rows not 16-byte multiples
    (dict(D=128, Dv=60), F.FABWD_ERR_UNSUPPORTED),
    (dict(D=192, Dv=192, dq_mode=F.FABWD_DQ_ATOMIC), F.FABWD_ERR_UNSUPPORTED),   # no fused kernel for it
    (dict(D=136, Dv=136, dq_mode=F.FABWD_DQ_ATOMIC), F.FABWD_ERR_UNSUPPORTED),
    (dict(dq_mode=3), F.FABWD_ERR_INVALID),
])
def test_validation_codes(lib, change, code):
    p = base_params(**change)
    assert ws_size(p)[0] == code
    for fn in ("fabwd_preprocess", "fabwd_run", "fabwd_run_main", "fabwd_run_dq"):
        assert F.call_status(fn, p, 0x100000, 1 << 30, None) == code


@pytest.mark.parametrize("D,Dv", [(64, 64), (128, 64), (128, 128), (192, 64), (192, 128), (192, 192), (8, 8),
                                  (40, 8), (96, 96), (80, 48), (136, 72), (160, 136), (184, 176)])
def test_head_dims_accepted(lib, D, Dv):
    # every D, Dv <= D that is a multiple of 8 has a kernel (its own class or the next larger one);
    # the atomic mode too unless both exceed 128
    for mode in (F.FABWD_DQ_AUTO, F.FABWD_DQ_SEPARATE, F.FABWD_DQ_ATOMIC):
        want = F.FABWD_ERR_UNSUPPORTED if mode == F.FABWD_DQ_ATOMIC and D > 128 and Dv > 128 else F.FABWD_OK
        assert ws_size(base_params(D=D, Dv=Dv, dq_mode=mode))[0] == want, (D, Dv, mode)


def test_null_and_workspace_codes(lib):
    assert F.lib().fabwd_workspace_size(None, ctypes.byref(ctypes.c_size_t())) == F.FABWD_ERR_NULLPTR
    p = base_params()
    assert F.lib().fabwd_workspace_size(ctypes.byref(p), None) == F.FABWD_ERR_NULLPTR
    for name in ("q", "k", "dout", "attn_out", "dq", "dv"):
        pp = base_params(**{name: None})
        assert F.call_status("fabwd_run", pp, 0x100000, 1 << 30, None) == F.FABWD_ERR_NULLPTR, name
    # softmax_lse is read by the preprocess only
    assert F.call_status("fabwd_preprocess", base_params(softmax_lse=None), 0x100000, 1 << 30, None) == F.FABWD_ERR_NULLPTR
    _, need = ws_size(p)
    assert F.call_status("fabwd_preprocess", p, None, need, None) == F.FABWD_ERR_WORKSPACE
    assert F.call_status("fabwd_run", p, 0x100000, need - 1, None) == F.FABWD_ERR_WORKSPACE
    assert F.call_status("fabwd_run", p, 0x100010, need, None) == F.FABWD_ERR_WORKSPACE  # not 256-aligned
    misaligned = base_params(q=0x10008)
    assert F.call_status("fabwd_run", misaligned, 0x100000, need, None) == F.FABWD_ERR_INVALID
    v = ctypes.c_uint32(0)
    assert F.lib().fabwd_read_device_status(None, 256, None, ctypes.byref(v)) == F.FABWD_ERR_NULLPTR


def test_optional_inputs_validation(lib):
    # seqused_q / seqused_kv (int32) and sinks (fp32) must be 4-byte aligned; refused on the host
    _, need = ws_size(base_params())
    for name in ("seqused_q", "seqused_kv", "sinks"):
        p = base_params(**{name: 0x20002})
        assert ws_size(p)[0] == F.FABWD_ERR_INVALID, name
        for fn in ("fabwd_preprocess", "fabwd_run"):
            assert F.call_status(fn, p, 0x100000, need, None) == F.FABWD_ERR_INVALID, (fn, name)
        assert ws_size(base_params(**{name: 0x20004}))[0] == F.FABWD_OK
    # the sizes do not change with them
    assert ws_size(base_params(seqused_q=0x20000, seqused_kv=0x20000, sinks=0x20000)) == ws_size(base_params())


def test_params_struct_matches_the_header():
    # the ctypes mirror ends with the optional inputs, in the header's order
    import re
    with open(F.HEADER) as f:
        text = f.read()
    body = text[text.index("typedef struct {"):text.index("} fabwd_params;")]
    fields = []
    for line in body.splitlines():
        line = line.split("/*")[0].strip()
        m = re.match(r"^(?:const\s+)?\w+\*?\s+\*?(.+);$", line)
        if m:
            fields += [x.strip().lstrip("*") for x in m.group(1).split(",")]
    assert fields == [f[0] for f in F.fabwd_params._fields_], fields


def test_statistics_preprocess_validation(lib):
    # every case below is refused on the host, before anything is enqueued
    p = base_params(softmax_lse=None)   # softmax_lse is not used by this entry point
    _, need = ws_size(base_params())
    st = lambda mx, sm, stride, ws=0x100000, n=need, pp=p: F.call_status("fabwd_preprocess_stats", pp, mx, sm,
                                                                        stride, ws, n, None)
    assert st(None, 0x20000, 1) == F.FABWD_ERR_NULLPTR
    assert st(0x20000, None, 1) == F.FABWD_ERR_NULLPTR
    assert st(0x20000, 0x20000, 0) == F.FABWD_ERR_INVALID
    assert st(0x20000, 0x20000, 1025) == F.FABWD_ERR_INVALID
    assert st(0x20000, 0x20002, 8) == F.FABWD_ERR_INVALID          # misaligned sum
    assert st(0x20002, 0x20000, 8) == F.FABWD_ERR_INVALID          # misaligned max (checked as softmax_lse)
    assert st(0x20000, 0x20000, 8, n=need - 1) == F.FABWD_ERR_WORKSPACE
    assert st(0x20000, 0x20000, 8, pp=base_params(N1=3)) == F.FABWD_ERR_INVALID
    assert F.call_status("fabwd_preprocess_stats", None, 0x20000, 0x20000, 1, 0x100000, need, None) == F.FABWD_ERR_NULLPTR


def test_forward_validation(lib):
    # refused on the host before anything is enqueued
    p = base_params(dout=None, attn_out=None, softmax_lse=None, dq=None, dk=None, dv=None)
    fw = lambda y, lse, ws, n, pp=p: F.call_status("fabwd_forward", pp, y, lse, ws, n, None)
    assert fw(None, 0x30000, 0x100000, 256) == F.FABWD_ERR_NULLPTR
    assert fw(0x30000, None, 0x100000, 256) == F.FABWD_ERR_NULLPTR
    assert fw(0x30000, 0x30000, None, 256) == F.FABWD_ERR_NULLPTR
    assert fw(0x30000, 0x30000, 0x100000, 255) == F.FABWD_ERR_WORKSPACE
    assert fw(0x30000, 0x30000, 0x100010, 256) == F.FABWD_ERR_WORKSPACE
    assert fw(0x30008, 0x30000, 0x100000, 256) == F.FABWD_ERR_INVALID       # attn_out not 16-byte aligned
    assert fw(0x30000, 0x30000, 0x100000, 256, pp=base_params(N1=3)) == F.FABWD_ERR_INVALID
    assert fw(0x30000, 0x30000, 0x100000, 256, pp=base_params(D=100, Dv=100)) == F.FABWD_ERR_UNSUPPORTED
    assert F.call_status("fabwd_forward", None, 0x30000, 0x30000, 0x100000, 256, None) == F.FABWD_ERR_NULLPTR


def test_tnd_validation(lib):
    p = base_params(layout=F.FABWD_TND, cu_seqlens_q=0x20000, cu_seqlens_kv=0x20000, B=3, T1=700, T2=650,
                    S1=300, S2=300)
    assert ws_size(p)[0] == F.FABWD_OK
    assert ws_size(base_params(layout=F.FABWD_TND, cu_seqlens_q=0x20000, cu_seqlens_kv=0x20000, T1=-1))[0] == \
        F.FABWD_ERR_INVALID
    # tokens but no max length
    assert ws_size(base_params(layout=F.FABWD_TND, cu_seqlens_q=0x20000, cu_seqlens_kv=0x20000, T1=5, S1=0))[0] == \
        F.FABWD_ERR_INVALID


def test_workspace_size_cannot_wrap(lib):
    # TND bounds B, N1 and max_seqlen_q one by one; their product sizes the workspace rows and
    # would wrap 64 bits at the extremes: refused on the host instead of a short workspace
    tnd = dict(layout=F.FABWD_TND, cu_seqlens_q=0x20000, cu_seqlens_kv=0x20000, T1=1 << 20, T2=1 << 20)
    assert ws_size(base_params(B=65535, N1=65535, N2=65535, S1=(1 << 30) - 1, S2=4096, **tnd))[0] == \
        F.FABWD_ERR_INVALID
    # a large but representable plan still sizes: 2^40 rows exactly
    s, nbytes = ws_size(base_params(B=1 << 12, N1=1 << 8, N2=1 << 8, S1=1 << 20, S2=4096, **tnd))
    assert s == F.FABWD_OK and nbytes >= 2 * 4 * (1 << 40)


def test_grid_size_limit(lib):
    # 2^27 queries over 4096 heads: 2^32 query-block CTAs in one grid row, more than a launch's x
    # dimension holds (the workspace, 2^39 rows, would still be sizable)
    p = base_params(B=1, N1=4096, N2=4096, S1=1 << 27, S2=128)
    assert ws_size(p)[0] == F.FABWD_ERR_UNSUPPORTED
    assert ws_size(base_params(B=1, N1=4096, N2=4096, S1=1 << 20, S2=128))[0] == F.FABWD_OK


def test_empty_sizes_are_valid(lib):
    assert ws_size(base_params(S1=0))[0] == F.FABWD_OK
    assert ws_size(base_params(S2=0))[0] == F.FABWD_OK


def test_wait_limit_and_injection_switches(lib):
    old = F.fabwd_set_wait_limit_ns(12345)
    assert F.fabwd_set_wait_limit_ns(0) == 12345
    assert F.fabwd_set_wait_limit_ns(old) == 2_000_000_000
    assert F.fabwd_debug_inject_timeout(True) == 0
    assert F.fabwd_debug_inject_timeout(False) == 1


def test_mask_mode_values():
    assert api.mask_mode_value("Causal") == 1 and api.mask_mode_value("none") == 0
    assert api.mask_mode_value(api.MaskMode.BAND) == 2 and api.mask_mode_value(1) == 1
    with pytest.raises(ValueError):
        api.mask_mode_value("diagonal")


def test_make_params_shapes_bsnd_tnd_bnsd():
    q = torch.zeros(2, 5, 4, 64, dtype=torch.bfloat16)
    k = torch.zeros(2, 7, 2, 64, dtype=torch.bfloat16)
    v = torch.zeros(2, 7, 2, 64, dtype=torch.bfloat16)
    o = torch.zeros(2, 5, 4, 64, dtype=torch.bfloat16)
    lse = torch.zeros(2, 4, 5)
    p = api.make_params(q, k, v, o, o, lse, q, k, v, mask_mode="causal")
    assert (p.B, p.S1, p.S2, p.N1, p.N2, p.D, p.Dv, p.mask_mode) == (2, 5, 7, 4, 2, 64, 64, 1)
    p = api.make_params(q.transpose(1, 2).contiguous(), k.transpose(1, 2).contiguous(), v.transpose(1, 2).contiguous(),
                        o, o, lse, q, k, v, layout="BNSD")
    assert (p.B, p.S1, p.S2, p.N1, p.N2) == (2, 5, 7, 4, 2)
    cu = torch.tensor([0, 3, 10], dtype=torch.int32)
    qt = torch.zeros(10, 4, 64, dtype=torch.float16)
    kt = torch.zeros(10, 2, 64, dtype=torch.float16)
    p = api.make_params(qt, kt, kt, qt, qt, torch.zeros(4, 10), qt, kt, kt, cu_seqlens_q=cu, cu_seqlens_kv=cu,
                        layout="TND")
    assert (p.B, p.T1, p.T2, p.S1, p.S2, p.dtype) == (2, 10, 10, 7, 7, F.FABWD_FP16)


def test_api_rejects_unsupported_inputs():
    t = torch.zeros(1, 4, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(NotImplementedError):
        api.flash_attn_grad(t, t, t, t, t, torch.zeros(1, 1, 4), attn_mask=torch.zeros(1, dtype=torch.int8))
    with pytest.raises(ValueError):
        api.flash_attn_grad(t, t, t, t, t, torch.zeros(1, 1, 4), layout_kv="TND")
    with pytest.raises(ValueError):   # CPU tensors: the library runs on CUDA only, no fallback
        api.flash_attn_grad(t, t, t, t, t, torch.zeros(1, 1, 4))
    with pytest.raises(ValueError):   # the forward too
        api.flash_attn_forward(t, t, t)


def test_lib_missing_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(F, "_lib", None)
    monkeypatch.setattr(build, "LIB", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="not built"):
        F.lib()


# ---------------------------------------------------------------------------------------------
# bench host logic
# ---------------------------------------------------------------------------------------------


def test_bench_flop_counts_match_the_convention():
    import bench

    pb = inputs.make_problem(inputs.WORKLOADS["gqa_causal_s4096_d128"])
    conv, alg = bench.flop_counts(pb)
    assert conv == 32 * 2 * 4096 * 4096 * (3 * 128 + 2 * 128) / 2
    assert alg == 32 * 2 * (3 * 128 + 2 * 128) * 4096 * 4097 // 2


@pytest.mark.parametrize("L1,L2,mode,wl,wr", [(7, 9, 1, -1, -1), (9, 7, 1, 2, -1), (12, 12, 2, 3, 1), (5, 8, 0, -1, -1),
                                              (10, 10, 1, 4, 0), (6, 6, 2, -1, 0)])
def test_bench_visible_pairs_brute_force(L1, L2, mode, wl, wr):
    import bench

    w = inputs.sized(inputs.WORKLOADS["mha_s128_d64"], mask_mode=mode, win_left=wl, win_right=wr)
    assert bench.visible_pairs(L1, L2, w) == int(orc.visible(L1, L2, mode, wl, wr).sum())


def test_inputs_are_seeded_and_shaped():
    w = inputs.WORKLOADS["varlen_window_fp16_d128"]
    a, b = inputs.make_problem(w), inputs.make_problem(w)
    assert torch.equal(a.q, b.q) and np.array_equal(a.cu_seqlens_q, b.cu_seqlens_q)
    lens = np.diff(a.cu_seqlens_q)
    assert len(lens) == 8 and lens.min() >= 256 and lens.max() <= 4096
    assert a.q.shape == (a.T1, 16, 128) and a.q.dtype == torch.float16
    g = inputs.make_problem(inputs.WORKLOADS["gqa_causal_s4096_d128"])
    assert abs(float(g.dout.float().std()) - 0.1) < 0.01
