#!/usr/bin/env python
"""Benchmark: attention-backward TFLOP/s (bf16) on one GB300 and % of dense tensor peak.

One step = one pass of the whole backward path over one batch of synthetic input:
fabwd_preprocess (sfmg, lse rows, dq accumulator zeroing) then fabwd_run (in the default
separate dQ mode one grid of dK/dV and dQ CTAs; in the atomic dQ mode the fused kv-stationary
kernel and the convert pass), all libfabwd kernels on one stream, with CUDA events between the
stages.

`value` follows the measurement convention: per head 2·S1·S2·(3D + 2Dv), halved under a causal
mask, over the whole step.  `roofline` is the tensor kernel with the longest time, credited with
the method's algorithmic work only: 2·(3D + 2Dv) flops per visible (query, key) pair, the five
products of the backward once each.  The separate dQ mode forms S and dP a second time in its
dQ CTAs; that executed work, 2·(4D + 3Dv) per pair, is reported beside it as `executed_frac`
and never counted in `frac`.

The headline workload (--workload, default the causal GQA S=4096 one) carries every extra: the
e2e pass through pinned host buffers, the forward side pass, the per-kind breakdown and the CPU
baseline.  The `workloads` object times the step of every workload of the measurement with the
same --steps/--warmup, L2 flushed between steps.

Inputs: q, k, v, dout are the seeded draws of attention_backward_fabwd_gb300.inputs; attn_out
and softmax_lse come from a plain torch fp32 forward on the GPU (input synthesis, untimed).
The L2 cache (129 MB) is flushed between timed steps by writing a 256 MB buffer (untimed).
SM clocks, power and clock-event reasons are read in-process through NVML's read-only queries
every 2 ms inside the timed region (nvidia-smi at 50 ms when NVML cannot be loaded).

`--impl reference` times the fp64 CPU oracle instead (host cores, bounded sample per step).
Multi-GPU (torchrun): each rank runs an independent replica (no collective on the data path);
the step time is the max over ranks and the value counts all ranks' work (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "gqa_causal_s4096_d128"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["fabwd", "reference"], default="fabwd")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--dq-mode", default="auto", choices=["auto", "atomic", "separate"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-forward", action="store_true", help="skip the untimed pass that times fabwd_forward")
    ap.add_argument("--no-breakdown", action="store_true",
                    help="skip the untimed pass that launches the dK/dV and dQ kernels on their own")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="run the chosen BSND/BNSD workload at S1 = S2 = this length: a smaller case of the same "
                         "kernels for profiler captures; the JSON line names the sized workload")
    ap.add_argument("--workloads", default="all",
                    help="comma-separated workloads whose step is timed beside the headline one, 'all' or 'none'")
    return ap.parse_args()


# ----------------------------------------------------------------------------------------------
# work counts
# ----------------------------------------------------------------------------------------------


def seq_lengths(pb):
    if pb.w.layout == "TND":
        return list(zip(np.diff(pb.cu_seqlens_q).tolist(), np.diff(pb.cu_seqlens_kv).tolist()))
    return [(pb.S1, pb.S2)] * pb.w.B


def visible_pairs(L1, L2, w):
    """Number of (i, j) pairs with lo <= j - i - (L2 - L1) <= hi, 0 <= j < L2 (per head)."""
    if L1 == 0 or L2 == 0:
        return 0
    lo, hi = -(1 << 40), 1 << 40
    if w.mask_mode != 0:
        if w.win_left >= 0:
            lo = -w.win_left
        if w.win_right >= 0:
            hi = w.win_right
        if w.mask_mode == 1:
            hi = min(hi, 0)
    i = np.arange(L1, dtype=np.int64)
    off = L2 - L1
    jlo = np.clip(i + off + lo, 0, L2)
    jhi = np.clip(i + off + hi + 1, 0, L2)
    return int(np.maximum(jhi - jlo, 0).sum())


def flop_counts(pb, per_pair=None):
    """(convention flops, algorithmic flops) of the step: per_pair flops per (query, key) pair,
    2·(3D + 2Dv) for the backward by default; S1·S2 pairs per head (halved when causal) or the
    visible pairs."""
    w = pb.w
    per_pair = 2 * (3 * w.D + 2 * w.Dv) if per_pair is None else per_pair
    conv = alg = 0
    for L1, L2 in seq_lengths(pb):
        f = per_pair * L1 * L2
        conv += f / 2 if w.mask_mode == 1 else f
        alg += per_pair * visible_pairs(L1, L2, w)
    return conv * w.N1, alg * w.N1


def io_bytes(pb):
    e = 2
    w = pb.w
    qn = pb.q.numel()
    kn, vn, on = pb.k.numel(), pb.v.numel(), pb.dout.numel()
    lse = w.N1 * pb.T1 * 4
    h2d = e * (qn + kn + vn + 2 * on) + lse
    d2h = e * (qn + kn + vn)
    return h2d, d2h


# ----------------------------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------------------------


def synth_forward(pb, dev):
    """attn_out (io dtype) and fp32 lse by a plain torch fp32 forward on the GPU (input synthesis)."""
    import torch

    w = pb.w
    scale = w.softmax_scale if w.softmax_scale != 0 else 1.0 / math.sqrt(w.D)
    q, k, v = (t.to(dev) for t in (pb.q, pb.k, pb.v))
    G = w.N1 // w.N2
    y = torch.empty(pb.dout.shape, dtype=q.dtype, device=dev)
    if w.layout == "TND":
        lse = torch.empty(w.N1, pb.T1, dtype=torch.float32, device=dev)
        seqs = [(None, slice(int(pb.cu_seqlens_q[s]), int(pb.cu_seqlens_q[s + 1])),
                 slice(int(pb.cu_seqlens_kv[s]), int(pb.cu_seqlens_kv[s + 1]))) for s in range(w.B)]
    else:
        lse = torch.empty(w.B, w.N1, pb.S1, dtype=torch.float32, device=dev)
        seqs = [(b, slice(0, pb.S1), slice(0, pb.S2)) for b in range(w.B)]

    def head(x, b, rows, n):
        if w.layout == "BSND":
            return x[b, rows, n]
        if w.layout == "BNSD":
            return x[b, n, rows]
        return x[rows, n]

    for b, rq, rk in seqs:
        L1, L2 = rq.stop - rq.start, rk.stop - rk.start
        if L1 == 0:
            continue
        ii = torch.arange(L1, device=dev)[:, None]
        jj = torch.arange(L2, device=dev)[None, :]
        d = jj - ii - (L2 - L1)
        ok = torch.ones(L1, L2, dtype=torch.bool, device=dev)
        if w.mask_mode == 1:
            ok &= d <= 0
        if w.mask_mode != 0 and w.win_left >= 0:
            ok &= d >= -w.win_left
        if w.mask_mode != 0 and w.win_right >= 0:
            ok &= d <= w.win_right
        for n1 in range(w.N1):
            n2 = n1 // G
            qh = head(q, b, rq, n1).float()
            s = (qh @ head(k, b, rk, n2).float().T) * scale
            s = s.masked_fill(~ok, float("-inf"))
            l = torch.logsumexp(s, dim=1)
            l = torch.where(torch.isfinite(l), l, torch.full_like(l, float("inf")))
            p = torch.exp(s - l[:, None]).masked_fill(~ok, 0.0)
            yh = p @ head(v, b, rk, n2).float()
            if w.layout == "BSND":
                y[b, rq, n1] = yh.to(y.dtype)
                lse[b, n1, rq] = l
            elif w.layout == "BNSD":
                y[b, n1, rq] = yh.to(y.dtype)
                lse[b, n1, rq] = l
            else:
                y[rq, n1] = yh.to(y.dtype)
                lse[n1, rq] = l
    return y, lse


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 50 ms; summary() keeps the samples taken
    inside the window marked by mark_start()/mark_end() (wall clock)."""

    FIELDS = ("timestamp,index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.bus_id = bus_id
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.out, stderr=subprocess.DEVNULL)
            deadline = time.time() + 10.0   # nvidia-smi takes a moment to print its first sample
            while time.time() < deadline and os.path.getsize(self.path) == 0:
                time.sleep(0.05)
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    @staticmethod
    def _when(stamp):
        try:
            head, _, frac = stamp.partition(".")
            return time.mktime(time.strptime(head, "%Y/%m/%d %H:%M:%S")) + float("0." + (frac or "0"))
        except ValueError:
            return None

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 11:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        if self.bus_id:
            mine = [r for r in rows if r[2].lower().endswith(self.bus_id.lower()[-12:])]
            rows = mine or rows
        ids = sorted(set(r[1] for r in rows))
        if len(ids) > 1:
            rows = [r for r in rows if r[1] == ids[0]]
        window = rows
        if self.t0 is not None and self.t1 is not None:
            def inside(r):
                t = self._when(r[0])
                return t is not None and self.t0 - 0.025 <= t <= self.t1 + 0.025
            window = [r for r in rows if inside(r)] or rows
        try:
            sm = [float(r[3]) for r in window]
            smax = max(float(r[4]) for r in window)
            power = [float(r[5]) for r in window]
        except ValueError:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in window for k in range(4) if r[7 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons, "samples": len(window),
                "samples_in_timed_region": len(window) if window is not rows else 0,
                "power_w_max": max(power), "period_ms": 50}


class NvmlClocks:
    """SM clock, power and clock-event reasons of one GPU, read in-process through NVML's
    read-only queries every `period_s` by a background thread (no setting is changed).
    summary() keeps the samples taken inside the window marked by mark_start()/mark_end().
    available is False when libnvidia-ml cannot be loaded or the GPU is not found."""

    # nvmlClocksEventReasons bits (NVML API constants)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id=None, period_s=0.002):
        import ctypes
        import threading

        self.period_s = period_s
        self.samples = []
        self.t0 = self.t1 = None
        self.available = False
        self._stop = threading.Event()
        self._thread = None
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            ok = False
            if pci_bus_id:
                ok = self.nv.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h)) == 0
            if not ok:
                n = ctypes.c_uint(0)
                if self.nv.nvmlDeviceGetCount_v2(ctypes.byref(n)) != 0 or n.value != 1:
                    return
                ok = self.nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) == 0
            if not ok:
                return
            self._reasons = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint(0)
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM = 1
            self.sm_max = mx.value
            self.available = self._read() is not None
        except (OSError, AttributeError):
            self.available = False

    def _read(self):
        import ctypes

        clk, mw, rs = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_ulonglong(0)
        if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) != 0:
            return None
        self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw))
        self._reasons(self.h, ctypes.byref(rs))
        return time.time(), clk.value, mw.value / 1000.0, rs.value

    def _loop(self):
        while not self._stop.is_set():
            r = self._read()
            if r is not None:
                self.samples.append(r)
            time.sleep(self.period_s)

    def __enter__(self):
        import threading

        if self.available:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def summary(self):
        if not self.available or not self.samples:
            return None
        win = [r for r in self.samples if self.t0 is not None and self.t1 is not None and self.t0 <= r[0] <= self.t1]
        rows = win or self.samples
        reasons = sorted({name for r in rows for bit, name in self.REASONS.items() if r[3] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": self.sm_max, "reasons": reasons,
                "samples": len(rows), "samples_in_timed_region": len(win),
                "power_w_max": max(r[2] for r in rows), "period_ms": 1e3 * self.period_s, "source": "nvml"}


def pci_bus_id_string(dev):
    """The GPU's PCI address in NVML's form (domain:bus:device.0), or None."""
    import torch

    try:
        pr = torch.cuda.get_device_properties(dev)
        return f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
    except Exception:
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


def profile_traffic(workload, kernel):
    """dram bytes per launch of `kernel` on `workload` from a committed ncu capture, if one matches
    the current kernel revision (profiles/traffic.json)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        v = d.get(workload, {}).get(kernel)
        if v and v.get("kernel_rev") == KERNEL_REV.get(kernel):
            return v.get("dram_bytes_per_launch")
    return None


def stage_table(pb, r, peak_tf, peak_hbm):
    """Per-stage timing with each kernel's algorithmic work.  Tensor stages are credited with the
    method's products they form, 2·(inner dimension) flops per visible (query, key) pair each:
    the one-grid separate-mode kernel and the fused atomic-mode kernel with all five,
    2·(3D + 2Dv); the dK/dV kernel alone with S, dP, dV, dK, 2·(2D + 2Dv); the dQ kernel alone
    with dQ, 2·D (its S and dP are recomputed).  `executed_*` counts every product a kernel
    forms, recomputed ones included.  HBM stages count the bytes they must read and write."""
    w = pb.w
    pairs = w.N1 * sum(visible_pairs(L1, L2, w) for L1, L2 in seq_lengths(pb))
    e = 2
    rows_pad = w.B * w.N1 * ((pb.S1 + 127) // 128 * 128)
    dq_acc = 0 if r["separate"] else 4 * r["dq_elems"]
    pre_bytes = e * 2 * pb.dout.numel() + 4 * w.N1 * pb.T1 + 2 * 4 * rows_pad + dq_acc

    def hbm(kernel, ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
        return {"kernel": kernel, "bound": "hbm", "ms": ms, "bytes": nbytes, "GB/s": gbs, "frac_of_hbm": gbs / peak_hbm}

    def tensor(kernel, ms, method_per_pair, executed_per_pair):
        f, fx = method_per_pair * pairs, executed_per_pair * pairs
        tf = f / (ms * 1e-3) / 1e12 if ms > 0 else 0.0
        tfx = fx / (ms * 1e-3) / 1e12 if ms > 0 else 0.0
        return {"kernel": kernel, "bound": "tensor", "ms": ms, "flops": f, "flops_per_pair": method_per_pair,
                "TFLOP/s": tf, "frac_of_peak": tf / peak_tf, "executed_flops": fx,
                "executed_flops_per_pair": executed_per_pair, "executed_TFLOP/s": tfx,
                "executed_frac_of_peak": tfx / peak_tf}

    full = 2 * (3 * w.D + 2 * w.Dv)
    kv_part, dq_exec = 2 * (2 * w.D + 2 * w.Dv), 2 * (2 * w.D + w.Dv)
    out = {"preprocess": hbm("preprocess_kernel", r["ms_pre"], pre_bytes)}
    if r.get("merged"):
        # one grid of dK/dV CTAs (S, dP, dV, dK) and dQ CTAs (S, dP again, dQ)
        out["backward"] = tensor("fabwd_bwd_kernel" if w.D <= 128 else "fabwd_bwd_wide_kernel", r["ms_main"], full,
                                 kv_part + dq_exec)
        if r.get("alone"):
            out["backward"]["launched_alone_ms"] = r["alone"]
    elif r["separate"]:
        out["dkdv"] = tensor("fabwd_kv_kernel" if w.D <= 128 else "fabwd_main_kernel", r["ms_main"], kv_part, kv_part)
        out["dq"] = tensor("fabwd_dq_kernel", r["ms_conv"], 2 * w.D, dq_exec)
    else:
        out["main"] = tensor("fabwd_main_kernel", r["ms_main"], full, full)
        out["convert"] = hbm("convert_kernel", r["ms_conv"], (4 + e) * r["dq_elems"])
    return out


# revision of each kernel's code that profiles/traffic.json must match
KERNEL_REV = {"fabwd_bwd_kernel": "bwd-v9", "fabwd_bwd_wide_kernel": "wide-v8", "fabwd_kv_kernel": "kv-v11",
              "fabwd_dq_kernel": "dq-v11", "fabwd_main_kernel": "main-v8"}


def max_over_ranks(values, world, device="cpu"):
    """Element-wise max of per-rank timings (every rank gets the result)."""
    import torch

    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist

        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.cpu().tolist()


def job_tflops(flops_per_rank, world, ms):
    """Whole-job throughput: every rank processed flops_per_rank in at most ms milliseconds."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def chosen_workload(args):
    """The workload named by --workload, at S1 = S2 = --seq-len when that is given."""
    from attention_backward_fabwd_gb300 import inputs

    w = inputs.WORKLOADS[args.workload]
    if args.seq_len:
        if w.layout == "TND":
            raise SystemExit("--seq-len applies to BSND/BNSD workloads")
        w = inputs.sized(w, name=f"{w.name}@S{args.seq_len}", S1=args.seq_len, S2=args.seq_len)
    return w


def replica_workload(w, rank):
    """Each rank draws its own batch of the same shape (independent replicas, weak scaling)."""
    from attention_backward_fabwd_gb300 import inputs

    return inputs.sized(w, seed=w.seed + 7919 * rank)


def prepare(w, dev, dq_mode):
    """Device inputs, outputs, params and workspace of one workload (untimed)."""
    import torch
    from attention_backward_fabwd_gb300 import api, fabwd, inputs

    pb = inputs.make_problem(w)
    attn_out, lse = synth_forward(pb, dev)
    q, k, v, dout = (t.to(dev) for t in (pb.q, pb.k, pb.v, pb.dout))
    cu_q = cu_kv = None
    extra = {}
    if w.layout == "TND":
        cu_q = torch.from_numpy(pb.cu_seqlens_q).to(dev)
        cu_kv = torch.from_numpy(pb.cu_seqlens_kv).to(dev)
        extra = dict(max_seqlen_q=pb.S1, max_seqlen_kv=pb.S2)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    mk = dict(cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv, softmax_scale=w.softmax_scale, mask_mode=w.mask_mode,
              win_left=w.win_left, win_right=w.win_right, layout=w.layout, dq_mode=dq_mode, **extra)
    p = api.make_params(q, k, v, dout, attn_out, lse, dq, dk, dv, **mk)
    nbytes = fabwd.fabwd_workspace_size(p)
    resolved = fabwd.fabwd_resolve_dq_mode(p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    # separate dQ mode: fabwd_run launches the dK/dV and dQ CTAs as one grid
    return dict(pb=pb, w=w, ins=[q, k, v, dout, attn_out, lse], outs=[dq, dk, dv], p=p, mk=mk, ws=ws, nbytes=nbytes,
                separate=resolved == fabwd.FABWD_DQ_SEPARATE, merged=resolved == fabwd.FABWD_DQ_SEPARATE,
                cu_q=cu_q, cu_kv=cu_kv)


def run_step(c, st, evs=None, split=True):
    """One step on stream st: preprocess, then the backward.  evs: 4 events, recorded before the
    preprocess, between the stages (split only) and after the backward.  An event between the two
    kernels stops the backward's programmatic dependent launch from overlapping the preprocess,
    so whole-step timings are taken without them (split=False)."""
    from attention_backward_fabwd_gb300 import fabwd

    p, ws, nbytes, sp = c["p"], c["ws"], c["nbytes"], st.cuda_stream
    if evs:
        evs[0].record(st)
    fabwd.fabwd_preprocess(p, ws.data_ptr(), nbytes, sp)
    if evs and split:
        evs[1].record(st)
    if c["merged"]:
        fabwd.fabwd_run(p, ws.data_ptr(), nbytes, sp)
        if evs:
            if split:
                evs[2].record(st)
            evs[3].record(st)
        return
    fabwd.fabwd_run_main(p, ws.data_ptr(), nbytes, sp)
    if evs and split:
        evs[2].record(st)
    fabwd.fabwd_run_dq(p, ws.data_ptr(), nbytes, sp)
    if evs:
        evs[3].record(st)


def check_status(c, st, when):
    from attention_backward_fabwd_gb300 import fabwd

    s_, bits = fabwd.fabwd_read_device_status(c["ws"].data_ptr(), c["nbytes"], st.cuda_stream)
    if s_ != fabwd.FABWD_OK:
        raise RuntimeError(f"device status {bits:#x} {when}")


def time_steps(c, dev, st, steps, warmup, flush, barrier=lambda: None, clk=None):
    """W untimed warm-up steps, then `steps` timed whole steps (events around each step only), then
    `steps` more with events between the stages, each step after an untimed L2 flush.  Returns the
    mean whole-step ms, the per-stage mean ms (preprocess, main, dQ stage) of the split loop, and
    the wall time of the whole-step loop."""
    import torch

    for _ in range(max(warmup, 0)):
        flush.fill_(1)
        run_step(c, st)
    check_status(c, st, "after warm-up")

    def loop(split):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for i in range(steps):
            flush.fill_(i & 0xFF)
            run_step(c, st, evs[i], split)
        return evs

    torch.cuda.synchronize(dev)
    barrier()
    t_wall0 = time.perf_counter()
    if clk is not None:
        clk.mark_start()
    whole = loop(False)
    torch.cuda.synchronize(dev)
    if clk is not None:
        clk.mark_end()
    barrier()
    t_wall = time.perf_counter() - t_wall0
    check_status(c, st, "after the timed steps")
    parts = loop(True)
    torch.cuda.synchronize(dev)
    check_status(c, st, "after the split steps")
    mean = lambda evs, i, j: statistics.mean(e[i].elapsed_time(e[j]) for e in evs)
    return dict(ms_step=mean(whole, 0, 3), ms_pre=mean(parts, 0, 1), ms_main=mean(parts, 1, 2),
                ms_conv=mean(parts, 2, 3), ms_step_split=mean(parts, 0, 3), t_wall=t_wall)


def gpu_arm(args, rank, world, local_rank):
    import torch
    from attention_backward_fabwd_gb300 import api, build, fabwd, inputs

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = replica_workload(chosen_workload(args), rank)
    c = prepare(w, dev, args.dq_mode)
    pb = c["pb"]
    q, k, v, dout, attn_out, lse = c["ins"]
    dq, dk, dv = c["outs"]
    p, ws, nbytes, merged = c["p"], c["ws"], c["nbytes"], c["merged"]
    cu_q, cu_kv = c["cu_q"], c["cu_kv"]
    st = torch.cuda.current_stream(dev)
    sp = st.cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    bus = pci_bus_id_string(dev)
    nv = NvmlClocks(bus)
    with (nv if nv.available else ClockSampler(bus)) as clk:
        t = time_steps(c, dev, st, args.steps, args.warmup, flush, barrier, clk)
    clocks = clk.summary()

    # the library's forward on the same inputs (untimed region, reported beside the step)
    fwd = None
    if not args.no_forward:
        y_f, lse_f = torch.empty_like(attn_out), torch.empty_like(lse)
        ws_f = torch.empty(256, dtype=torch.uint8, device=dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(10)]
        for i in range(13):
            flush.fill_(5)
            if i >= 3:
                ev[i - 3][0].record(st)
            fabwd.fabwd_forward(p, y_f.data_ptr(), lse_f.data_ptr(), ws_f.data_ptr(), 256, sp)
            if i >= 3:
                ev[i - 3][1].record(st)
        s_, bits = fabwd.fabwd_read_device_status(ws_f.data_ptr(), 256, sp)
        if s_ != fabwd.FABWD_OK:
            raise RuntimeError(f"device status {bits:#x} after the forward")
        fwd = {"ms": statistics.mean(e_[0].elapsed_time(e_[1]) for e_ in ev)}

    # breakdown only (untimed region): the dK/dV and dQ kernels launched on their own
    alone = None
    if merged and not args.no_breakdown:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(10)]
        for e_ in ev:
            flush.fill_(3)
            fabwd.fabwd_preprocess(p, ws.data_ptr(), nbytes, sp)
            e_[0].record(st)
            fabwd.fabwd_run_main(p, ws.data_ptr(), nbytes, sp)
            e_[1].record(st)
            fabwd.fabwd_run_dq(p, ws.data_ptr(), nbytes, sp)
            e_[2].record(st)
        torch.cuda.synchronize(dev)
        alone = {"dkdv_ms": statistics.mean(e_[0].elapsed_time(e_[1]) for e_ in ev),
                 "dq_ms": statistics.mean(e_[1].elapsed_time(e_[2]) for e_ in ev)}

    # e2e: pinned host buffers through the C ABI, every step's H2D copies and D2H reads inside the
    # timed region.  Steps are pipelined the way a caller streaming batches would run them: two
    # sets of device buffers, the H2D copies of step i+1 and the D2H reads of step i-1 on their
    # own streams while step i computes.
    e2e = None
    if not args.no_e2e:
        h_in = [t.cpu().pin_memory() for t in (q, k, v, dout, attn_out, lse)]
        h2d, d2h = io_bytes(pb)
        slots = []
        for sl in range(2):
            d_in = [q, k, v, dout, attn_out, lse] if sl == 0 else [torch.empty_like(t) for t in (q, k, v, dout, attn_out, lse)]
            d_out = [dq, dk, dv] if sl == 0 else [torch.empty_like(t) for t in (dq, dk, dv)]
            h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in d_out]
            ps = api.make_params(*d_in, *d_out, **c["mk"])
            wss = ws if sl == 0 else torch.empty(nbytes, dtype=torch.uint8, device=dev)
            slots.append((d_in, d_out, h_out, ps, wss))
        s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        n_e2e = min(50, max(3, args.steps // 2))
        n_all = n_e2e + 2
        ev_h2d = [torch.cuda.Event() for _ in range(n_all)]
        ev_cmp = [torch.cuda.Event() for _ in range(n_all)]
        ev_d2h = [torch.cuda.Event() for _ in range(n_all)]
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        for i in range(n_all):
            d_in, d_out, h_out, ps, wss = slots[i % 2]
            if i == 2:
                t_start.record(s_h2d)
            if i >= 2:
                s_h2d.wait_event(ev_cmp[i - 2])  # step i-2 has finished reading this slot's inputs
            with torch.cuda.stream(s_h2d):
                for d_, h_ in zip(d_in, h_in):
                    d_.copy_(h_, non_blocking=True)
            ev_h2d[i].record(s_h2d)
            st.wait_event(ev_h2d[i])
            if i >= 2:
                st.wait_event(ev_d2h[i - 2])  # this slot's outputs of step i-2 are on the host
            fabwd.fabwd_preprocess(ps, wss.data_ptr(), nbytes, sp)
            fabwd.fabwd_run(ps, wss.data_ptr(), nbytes, sp)
            ev_cmp[i].record(st)
            s_d2h.wait_event(ev_cmp[i])
            with torch.cuda.stream(s_d2h):
                for h_, d_ in zip(h_out, d_out):
                    h_.copy_(d_, non_blocking=True)
            ev_d2h[i].record(s_d2h)
        t_end.record(s_d2h)
        torch.cuda.synchronize(dev)
        e2e_ms = t_start.elapsed_time(t_end) / n_e2e
        e2e = {"ms": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "pipelining": "two device buffer sets; H2D of step i+1 and D2H of step i-1 overlap step i"}

    # every workload of the measurement: its step with the same steps/warm-up (the headline one
    # reuses the numbers above)
    others = {}
    names = list(inputs.WORKLOADS) if args.workloads == "all" else \
        ([] if args.workloads == "none" else [x for x in args.workloads.split(",") if x])
    for name in names:
        if name == args.workload and not args.seq_len:
            continue
        wo = replica_workload(inputs.WORKLOADS[name], rank)
        co = prepare(wo, dev, args.dq_mode)
        to = time_steps(co, dev, st, args.steps, args.warmup, flush, barrier)
        others[name] = dict(co=co, t=to)
        for key in ("ins", "outs", "ws"):
            co.pop(key)
        torch.cuda.empty_cache()

    keys = ("ms_step", "ms_main", "ms_pre", "ms_conv", "ms_step_split")
    vals = [t[k_] for k_ in keys] + [e2e["ms"] if e2e else 0.0, t["t_wall"]]
    for name in others:
        vals += [others[name]["t"][k_] for k_ in keys]
    vals = max_over_ranks(vals, world, dev)
    nk = len(keys)
    t = dict(zip(keys, vals[:nk]))
    e2e_ms, t_wall = vals[nk], vals[nk + 1]
    for i, name in enumerate(others):
        others[name]["t"] = dict(zip(keys, vals[nk + 2 + nk * i:nk + 2 + nk * (i + 1)]))
    return dict(pb=pb, w=w, **t, e2e=e2e, e2e_ms=e2e_ms, t_wall=t_wall, clocks=clocks, dq_elems=dq.numel(),
                nbytes=nbytes, separate=c["separate"], merged=merged, alone=alone, fwd=fwd, others=others)


# ----------------------------------------------------------------------------------------------
# CPU oracle (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------------------------


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def oracle_head_sampler(pb):
    """Yields (seconds, flops_convention) of the fp64 oracle backward of one head at a time."""
    from attention_backward_fabwd_gb300 import inputs
    from oracle import fabwd_oracle as orc

    w = pb.w
    scale = orc.resolve_scale(w.softmax_scale, w.D)
    G = w.N1 // w.N2
    seqs = []
    if w.layout == "TND":
        for s in range(w.B):
            seqs.append((None, slice(int(pb.cu_seqlens_q[s]), int(pb.cu_seqlens_q[s + 1])),
                         slice(int(pb.cu_seqlens_kv[s]), int(pb.cu_seqlens_kv[s + 1]))))
    else:
        seqs = [(b, slice(0, pb.S1), slice(0, pb.S2)) for b in range(w.B)]

    def head(x, b, rows, n):
        if w.layout == "BSND":
            return x[b, rows, n]
        if w.layout == "BNSD":
            return x[b, n, rows]
        return x[rows, n]

    units = [(sq, n1) for sq in seqs for n1 in range(w.N1)]
    per_pair = 2 * (3 * w.D + 2 * w.Dv)
    idx = 0
    while True:
        (b, rq, rk), n1 = units[idx % len(units)]
        idx += 1
        L1, L2 = rq.stop - rq.start, rk.stop - rk.start
        n2 = n1 // G
        qh, kh, vh, dyh = (inputs.to_f64(head(t, b, r, n)) for t, r, n in
                           ((pb.q, rq, n1), (pb.k, rk, n2), (pb.v, rk, n2), (pb.dout, rq, n1)))
        ok = orc.visible(L1, L2, w.mask_mode, w.win_left, w.win_right)
        y, lse = orc.forward_head(qh, kh, vh, scale, ok)
        y = inputs.to_f64(inputs.round_io(y, w.dtype))
        lse = lse.astype(np.float32).astype(np.float64)
        t0 = time.perf_counter()
        orc.backward_head(qh, kh, vh, dyh, y, lse, scale, ok)
        dt = time.perf_counter() - t0
        f = per_pair * L1 * L2
        yield dt, (f / 2 if w.mask_mode == 1 else f), (L1, L2)


def cpu_baseline(pb, budget_s):
    secs = flops = 0.0
    heads = 0
    shape = None
    for dt, f, shp in oracle_head_sampler(pb):
        secs += dt
        flops += f
        heads += 1
        shape = shp
        if secs >= budget_s:
            break
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "cpu_model": cpu_model(),
            "kind": "oracle", "sample": f"fp64 numpy oracle backward of {heads} head(s) of the workload (S1xS2 {shape[0]}x{shape[1]}), "
                      f"{secs:.1f} s of CPU time, same flop convention"}


def reference_arm(args, rank, world):
    from attention_backward_fabwd_gb300 import inputs

    if rank != 0:
        return None
    w = chosen_workload(args)
    pb = inputs.make_problem(w)
    gen = oracle_head_sampler(pb)
    for _ in range(max(args.warmup, 0)):
        next(gen)
    secs = flops = 0.0
    times = []
    shape = None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        dt, f, shape = next(gen)
        secs += dt
        flops += f
        times.append(dt)
    value = flops / secs / 1e12
    cores = blas_threads()
    sample = (f"each step: fp64 numpy oracle backward of one head (S1xS2 {shape[0]}x{shape[1]}) of the workload, "
              f"same flop convention")
    conv, _ = flop_counts(pb)
    return {"metric": "attention-backward TFLOP/s (bf16) at 1 GB300 and % of dense tensor peak", "value": value,
            "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(pb, l2="n/a (CPU)"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "cpu_model": cpu_model(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0, "wall_s": time.perf_counter() - t0}


def workload_config(pb, l2):
    w = pb.w
    cfg = {"workload": w.name, "layout": w.layout, "B": w.B, "S1": pb.S1, "S2": pb.S2, "N1": w.N1, "N2": w.N2,
           "D": w.D, "Dv": w.Dv, "mask_mode": w.mask_mode, "win_left": w.win_left, "win_right": w.win_right,
           "io_dtype": w.dtype, "l2": l2}
    if w.layout == "TND":
        cfg["seq_lengths"] = np.diff(pb.cu_seqlens_q).tolist()
        cfg["T1"] = pb.T1
    return cfg


def workloads_table(r, peak_tf, peak_hbm, world):
    """Per workload: step time, the dominant tensor kernel's time and its fraction of the peak on
    the method's work (2·(3D + 2Dv) flops per visible pair), and the executed-work fraction."""
    rows = {r["w"].name: dict(pb=r["pb"], t={k: r[k] for k in ("ms_step", "ms_main", "ms_pre", "ms_conv", "ms_step_split")},
                              separate=r["separate"], merged=r["merged"], dq_elems=r["dq_elems"])}
    for name, o in r["others"].items():
        co = o["co"]
        rows[name] = dict(pb=co["pb"], t=o["t"], separate=co["separate"], merged=co["merged"],
                          dq_elems=co["pb"].q.numel())
    out = {}
    for name, x in rows.items():
        pb = x["pb"]
        conv, alg = flop_counts(pb)
        rr = dict(x["t"], separate=x["separate"], merged=x["merged"], dq_elems=x["dq_elems"])
        stg = stage_table(pb, rr, peak_tf, peak_hbm)
        dom = max((v for v in stg.values() if v["bound"] == "tensor"), key=lambda v: v["ms"])
        out[name] = {"step_ms": x["t"]["ms_step"], "step_ms_with_stage_events": x["t"]["ms_step_split"],
                     "value": job_tflops(conv, world, x["t"]["ms_step"]),
                     "kernel": dom["kernel"], "kernel_ms": dom["ms"], "method_TFLOP/s": dom["TFLOP/s"],
                     "frac": dom["frac_of_peak"], "executed_frac": dom["executed_frac_of_peak"],
                     "preprocess_ms": x["t"]["ms_pre"], "flops_convention": conv, "flops_algorithmic": alg,
                     "dtype": pb.w.dtype}
        if pb.w.layout == "TND":
            out[name]["seq_lengths"] = np.diff(pb.cu_seqlens_q).tolist()
    return out


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        out = reference_arm(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    r = gpu_arm(args, rank, world, local_rank)
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    pb, w = r["pb"], r["w"]
    conv, alg = flop_counts(pb)
    peak_tf, peak_hbm, peak_kind = measured_peaks()
    value = job_tflops(conv, world, r["ms_step"])
    stages = stage_table(pb, r, peak_tf, peak_hbm)
    dom = max((st for st in stages.values() if st["bound"] == "tensor"), key=lambda st: st["ms"])
    out = {
        "metric": "attention-backward TFLOP/s (bf16) at 1 GB300 and % of dense tensor peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["ms_step"], "ms_per_step_with_stage_events": r["ms_step_split"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(pb, l2="flushed: 256 MB buffer written between timed steps (untimed)"),
        "dq_mode": "separate" if r["separate"] else "atomic",
        "pct_of_peak": 100.0 * value / world / peak_tf,
        "roofline": {"bound": "tensor", "achieved": dom["TFLOP/s"], "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": dom["TFLOP/s"] / peak_tf, "traffic": profile_traffic(w.name, dom["kernel"]),
                     "kernel": dom["kernel"], "peak_kind": f"{peak_kind} bf16 dense (burst)",
                     "algorithmic_flops_per_launch": dom["flops"], "ms_per_launch": dom["ms"],
                     "flops_per_pair": dom["flops_per_pair"],
                     "executed_frac": dom["executed_frac_of_peak"],
                     "executed_flops_per_pair": dom["executed_flops_per_pair"]},
        "kernels": stages,
        "workloads": workloads_table(r, peak_tf, peak_hbm, world),
        "flops_convention": conv, "flops_algorithmic": alg,
        "gpu_launches": (2 if r["merged"] else 3) * args.steps,
        "clocks": r["clocks"],
        "wall_s_timed_region": r["t_wall"],
    }
    if r.get("fwd"):
        ff = flop_counts(pb, per_pair=2 * (w.D + w.Dv))
        out["forward"] = {"kernel": "fabwd_fwd_kernel", "ms": r["fwd"]["ms"],
                          "TFLOP/s": ff[0] / (r["fwd"]["ms"] * 1e-3) / 1e12,
                          "algorithmic_TFLOP/s": ff[1] / (r["fwd"]["ms"] * 1e-3) / 1e12,
                          "frac_of_peak_algorithmic": ff[1] / (r["fwd"]["ms"] * 1e-3) / 1e12 / peak_tf,
                          "flops_convention": ff[0], "flops_per_pair": 2 * (w.D + w.Dv),
                          "note": "untimed side pass (10 launches, L2 flushed), not part of the step"}
    if r["e2e"]:
        out["e2e"] = {"value": job_tflops(conv, world, r["e2e_ms"]), "unit": "TFLOP/s",
                      "h2d_bytes_per_step": r["e2e"]["h2d_bytes_per_step"],
                      "d2h_bytes_per_step": r["e2e"]["d2h_bytes_per_step"], "ms_per_step": r["e2e_ms"],
                      "steps": r["e2e"]["steps"], "pipelining": r["e2e"]["pipelining"]}
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(pb, args.cpu_seconds)
    print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
