"""CPU check of the test infrastructure itself: the pooled full-size reference (the oracle run
per kv-head group in spawned processes) equals the oracle run on the whole problem."""
import numpy as np
import pytest

from attention_backward_fabwd_gb300 import inputs

import fabwd_testlib as tl

W = inputs.WORKLOADS


@pytest.mark.parametrize("w,lens", [
    (inputs.sized(W["gqa_causal_s4096_d128"], B=2, N1=4, N2=2, S1=70, S2=90, D=64, Dv=64, dout_std=1.0), None),
    (inputs.sized(W["varlen_window_fp16_d128"], B=3, N1=4, N2=2, D=64, Dv=64, win_left=20), ([30, 0, 41], None)),
    (inputs.sized(W["mha_s128_d64"], layout="BNSD", B=2, N1=2, N2=1, S1=33, S2=47, mask_mode=2, win_left=5,
                  win_right=3), None),
], ids=["bsnd_gqa", "tnd_window", "bnsd_band"])
def test_pooled_reference_equals_whole_problem(w, lens):
    pb = inputs.make_problem(w, *(lens or ()))
    whole = tl.full_reference(pb)
    pooled = tl.full_reference_parallel(pb)
    assert np.array_equal(inputs.to_f64(whole.attn_out), inputs.to_f64(pooled.attn_out))
    assert np.array_equal(whole.lse.numpy(), pooled.lse.numpy())
    for name in ("dq", "dk", "dv", "sfmg"):
        a, b = getattr(whole, name), getattr(pooled, name)
        assert a.shape == b.shape, name
        assert np.allclose(a, b, rtol=1e-12, atol=1e-13 * max(np.abs(a).max(), 1e-300)), name
