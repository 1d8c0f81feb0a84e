"""Host-side pieces of bench.py: the per-stage work counts and the clock-sample summary."""
import os
import tempfile
import time

import pytest

from attention_backward_fabwd_gb300 import inputs


def _r(separate, ms=(0.01, 0.2, 0.1), merged=False):
    return {"separate": separate, "ms_pre": ms[0], "ms_main": ms[1], "ms_conv": ms[2], "dq_elems": 1000,
            "merged": merged}


def test_stage_table_splits_the_five_products():
    import bench
    pb = inputs.make_problem(inputs.sized(inputs.WORKLOADS["mha_s128_d64"], S1=100, S2=100))
    w = pb.w
    conv, alg = bench.flop_counts(pb)
    sep = bench.stage_table(pb, _r(True), 1000.0, 5000.0)
    ato = bench.stage_table(pb, _r(False), 1000.0, 5000.0)
    assert set(sep) == {"preprocess", "dkdv", "dq"} and set(ato) == {"preprocess", "main", "convert"}
    # the fused kernel forms the method's five products once
    assert ato["main"]["flops"] == pytest.approx(alg)
    # dK/dV kernel: S, dP, dV, dK; dQ kernel: S, dP again and dQ, credited with dQ only
    assert sep["dkdv"]["flops_per_pair"] == 2 * (2 * w.D + 2 * w.Dv)
    assert sep["dq"]["flops_per_pair"] == 2 * w.D
    assert sep["dq"]["executed_flops_per_pair"] == 2 * (2 * w.D + w.Dv)
    assert sep["dkdv"]["flops"] + sep["dq"]["flops"] == pytest.approx(alg)
    assert sep["dkdv"]["executed_flops"] + sep["dq"]["executed_flops"] == \
        pytest.approx(alg * (4 * w.D + 3 * w.Dv) / (3 * w.D + 2 * w.Dv))
    assert sep["dkdv"]["TFLOP/s"] == pytest.approx(sep["dkdv"]["flops"] / 0.2e-3 / 1e12)
    # one grid for both separate-mode kernels: the method's work once (frac), every product formed
    # (executed_frac) beside it
    mer = bench.stage_table(pb, _r(True, merged=True), 1000.0, 5000.0)
    assert set(mer) == {"preprocess", "backward"}
    assert mer["backward"]["flops"] == pytest.approx(alg)
    assert mer["backward"]["flops_per_pair"] == 2 * (3 * w.D + 2 * w.Dv)
    assert mer["backward"]["executed_flops"] == pytest.approx(sep["dkdv"]["executed_flops"] + sep["dq"]["executed_flops"])
    assert mer["backward"]["frac_of_peak"] == pytest.approx(alg / 0.2e-3 / 1e12 / 1000.0)
    assert mer["backward"]["executed_frac_of_peak"] > mer["backward"]["frac_of_peak"]
    # the separate mode has no fp32 accumulator to zero
    assert ato["preprocess"]["bytes"] - sep["preprocess"]["bytes"] == 4 * 1000
    assert ato["convert"]["bytes"] == 6 * 1000


def test_clock_summary_keeps_the_timed_window():
    import bench
    fd, path = tempfile.mkstemp(suffix=".csv")
    os.close(fd)
    base = time.time()
    rows = []
    for dt, mhz, reason in [(-1.0, 1000, "Not Active"), (0.1, 1800, "Not Active"), (0.2, 1700, "Active"),
                            (2.0, 900, "Not Active")]:
        t = base + dt
        stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + f".{int((t % 1) * 1000):03d}"
        rows.append(f"{stamp}, 0, 00000000:1B:00.0, {mhz}, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, {reason}")
    with open(path, "w") as f:
        f.write("\n".join(rows) + "\n")
    c = bench.ClockSampler()
    c.proc, c.path, c.t0, c.t1 = object(), path, base, base + 0.5
    s = c.summary()
    assert s["samples"] == 2 and s["samples_in_timed_region"] == 2
    assert s["sm_mhz"] == pytest.approx(1750) and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_nvml_sampler_summary_keeps_the_timed_window():
    import bench
    c = bench.NvmlClocks.__new__(bench.NvmlClocks)
    c.available, c.sm_max, c.period_s = True, 2070, 0.002
    base = time.time()
    c.samples = [(base - 1, 900, 100.0, 0x1), (base + 0.1, 2070, 900.0, 0x0), (base + 0.2, 2000, 1000.0, 0x4),
                 (base + 2, 1000, 50.0, 0x0)]
    c.t0, c.t1 = base, base + 0.5
    s = c.summary()
    assert s["samples_in_timed_region"] == 2 and s["sm_mhz"] == pytest.approx(2035)
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1000.0 and s["source"] == "nvml"


def test_nvml_sampler_without_a_gpu_is_unavailable():
    import bench
    c = bench.NvmlClocks("00000000:00:00.0")
    if not c.available:
        assert c.summary() is None


def test_seq_len_sizes_the_chosen_workload():
    # --seq-len runs a BSND/BNSD workload at S1 = S2 = N under its own name; varlen is refused
    import argparse
    import bench

    args = argparse.Namespace(workload="causal_s8192_d192_dv128", seq_len=512)
    w = bench.chosen_workload(args)
    base = inputs.WORKLOADS["causal_s8192_d192_dv128"]
    assert (w.S1, w.S2, w.name) == (512, 512, "causal_s8192_d192_dv128@S512")
    assert (w.D, w.Dv, w.N1, w.N2, w.mask_mode, w.dtype) == (base.D, base.Dv, base.N1, base.N2, base.mask_mode,
                                                             base.dtype)
    args.seq_len = 0
    assert bench.chosen_workload(args) is base
    with pytest.raises(SystemExit):
        bench.chosen_workload(argparse.Namespace(workload="varlen_window_fp16_d128", seq_len=512))


def test_cpu_model_is_named():
    import bench
    name = bench.cpu_model()
    assert isinstance(name, str) and name
