#!/usr/bin/env python
"""Benchmark: attention-backward TFLOP/s (bf16) on one GB300 and % of dense tensor peak.

One step = one pass of the whole backward path over one batch of synthetic input:
fabwd_preprocess (sfmg, lse rows, dq accumulator zeroing) -> fabwd_run_main (the dK/dV kernel,
or the fused kernel in the atomic dQ mode) -> fabwd_run_dq (the dQ kernel, or the convert pass),
all libfabwd kernels on one stream, with CUDA events between the stages.

`value` follows the measurement convention: per head 2·S1·S2·(3D + 2Dv), halved under a causal
mask, over the whole step.  `roofline` is the stage kernel with the longest time, credited with
its own algorithmic flops: 2·(inner dimensions of the products it forms) per visible (query, key)
pair — (3D + 2Dv) for the fused kernel, (2D + 2Dv) for the dK/dV kernel, (2D + Dv) for the dQ
kernel (which forms S and dP again).

Inputs: q, k, v, dout are the seeded draws of attention_backward_fabwd_gb300.inputs; attn_out
and softmax_lse come from a plain torch fp32 forward on the GPU (input synthesis, untimed).
The L2 cache (129 MB) is flushed between timed steps by writing a 256 MB buffer (untimed).
SM clocks and throttle reasons are sampled by nvidia-smi every 50 ms inside the timed region.

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
    """Per-stage timing with each kernel's algorithmic work: tensor stages count 2·(the inner
    dimensions of their own products) flops per visible (query, key) pair; HBM stages count the
    bytes they must read and write."""
    w = pb.w
    pairs = w.N1 * sum(visible_pairs(L1, L2, w) for L1, L2 in seq_lengths(pb))
    e = 2
    rows_pad = w.B * w.N1 * ((pb.S1 + 127) // 128 * 128)
    dq_acc = 0 if r["separate"] else 4 * r["dq_elems"]
    pre_bytes = e * 2 * pb.dout.numel() + 4 * w.N1 * pb.T1 + 2 * 4 * rows_pad + dq_acc

    def hbm(kernel, ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9 if ms > 0 else 0.0
        return {"kernel": kernel, "bound": "hbm", "ms": ms, "bytes": nbytes, "GB/s": gbs, "frac_of_hbm": gbs / peak_hbm}

    def tensor(kernel, ms, per_pair):
        f = per_pair * pairs
        tf = f / (ms * 1e-3) / 1e12 if ms > 0 else 0.0
        return {"kernel": kernel, "bound": "tensor", "ms": ms, "flops": f, "flops_per_pair": per_pair,
                "TFLOP/s": tf, "frac_of_peak": tf / peak_tf}

    out = {"preprocess": hbm("preprocess_kernel", r["ms_pre"], pre_bytes)}
    if r.get("merged"):
        # one grid of dK/dV CTAs (S, dP, dV, dK) and dQ CTAs (S, dP again, dQ)
        out["backward"] = tensor("fabwd_bwd_kernel" if w.D <= 128 else "fabwd_bwd_wide_kernel", r["ms_main"],
                                 2 * (2 * w.D + 2 * w.Dv) + 2 * (2 * w.D + w.Dv))
        if r.get("alone"):
            out["backward"]["launched_alone_ms"] = r["alone"]
    elif r["separate"]:
        out["dkdv"] = tensor("fabwd_kv_kernel" if w.D <= 128 else "fabwd_main_kernel", r["ms_main"],
                             2 * (2 * w.D + 2 * w.Dv))
        out["dq"] = tensor("fabwd_dq_kernel", r["ms_conv"], 2 * (2 * w.D + w.Dv))
    else:
        out["main"] = tensor("fabwd_main_kernel", r["ms_main"], 2 * (3 * w.D + 2 * w.Dv))
        out["convert"] = hbm("convert_kernel", r["ms_conv"], (4 + e) * r["dq_elems"])
    return out


# revision of each kernel's code that profiles/traffic.json must match
KERNEL_REV = {"fabwd_bwd_kernel": "bwd-v3", "fabwd_kv_kernel": "kv-v5", "fabwd_dq_kernel": "dq-v5",
              "fabwd_main_kernel": "main-v4"}


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


def replica_workload(w, rank):
    """Each rank draws its own batch of the same shape (independent replicas, weak scaling)."""
    from attention_backward_fabwd_gb300 import inputs

    return inputs.sized(w, seed=w.seed + 7919 * rank)


def gpu_arm(args, rank, world, local_rank):
    import torch
    from attention_backward_fabwd_gb300 import api, build, fabwd, inputs

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = inputs.WORKLOADS[args.workload]
    w = replica_workload(w, rank)
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
    p = api.make_params(q, k, v, dout, attn_out, lse, dq, dk, dv, cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv,
                        softmax_scale=w.softmax_scale, mask_mode=w.mask_mode, win_left=w.win_left,
                        win_right=w.win_right, layout=w.layout, dq_mode=args.dq_mode, **extra)
    nbytes = fabwd.fabwd_workspace_size(p)
    resolved = fabwd.fabwd_resolve_dq_mode(p)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream(dev)
    sp = st.cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    # separate dQ mode: fabwd_run launches the dK/dV and dQ CTAs as one grid
    merged = resolved == fabwd.FABWD_DQ_SEPARATE

    def step(evs=None):
        if evs:
            evs[0].record(st)
        fabwd.fabwd_preprocess(p, ws.data_ptr(), nbytes, sp)
        if evs:
            evs[1].record(st)
        if merged:
            fabwd.fabwd_run(p, ws.data_ptr(), nbytes, sp)
            if evs:
                evs[2].record(st)
                evs[3].record(st)
            return
        fabwd.fabwd_run_main(p, ws.data_ptr(), nbytes, sp)
        if evs:
            evs[2].record(st)
        fabwd.fabwd_run_dq(p, ws.data_ptr(), nbytes, sp)
        if evs:
            evs[3].record(st)

    for _ in range(max(args.warmup, 0)):
        flush.fill_(1)
        step()
    s_, bits = fabwd.fabwd_read_device_status(ws.data_ptr(), nbytes, sp)
    if s_ != fabwd.FABWD_OK:
        raise RuntimeError(f"device status {bits:#x} after warm-up")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
        bus = f"{bus:02x}" if isinstance(bus, int) else str(bus)
    except Exception:
        bus = None
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    with ClockSampler(bus) as clk:
        torch.cuda.synchronize(dev)
        barrier()
        t_wall0 = time.perf_counter()
        clk.mark_start()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            step(evs[i])
        torch.cuda.synchronize(dev)
        clk.mark_end()
        barrier()
        t_wall = time.perf_counter() - t_wall0
    pre = [e[0].elapsed_time(e[1]) for e in evs]
    main = [e[1].elapsed_time(e[2]) for e in evs]
    conv = [e[2].elapsed_time(e[3]) for e in evs]
    tot = [e[0].elapsed_time(e[3]) for e in evs]
    ms_step = statistics.mean(tot)
    ms_main = statistics.mean(main)
    s_, bits = fabwd.fabwd_read_device_status(ws.data_ptr(), nbytes, sp)
    if s_ != fabwd.FABWD_OK:
        raise RuntimeError(f"device status {bits:#x} after the timed steps")

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
            ps = api.make_params(*d_in, *d_out, cu_seqlens_q=cu_q, cu_seqlens_kv=cu_kv, softmax_scale=w.softmax_scale,
                                 mask_mode=w.mask_mode, win_left=w.win_left, win_right=w.win_right, layout=w.layout,
                                 dq_mode=args.dq_mode, **extra)
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

    ms_step, ms_main, ms_pre, ms_conv, e2e_ms, t_wall = max_over_ranks(
        [ms_step, ms_main, statistics.mean(pre), statistics.mean(conv), e2e["ms"] if e2e else 0.0, t_wall], world, dev)
    return dict(pb=pb, w=w, ms_step=ms_step, ms_main=ms_main, ms_pre=ms_pre, ms_conv=ms_conv, e2e=e2e, e2e_ms=e2e_ms,
                t_wall=t_wall, clocks=clk.summary(), dq_elems=dq.numel(), nbytes=nbytes,
                separate=resolved == fabwd.FABWD_DQ_SEPARATE, merged=merged, alone=alone, fwd=fwd)


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
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 numpy oracle backward of {heads} head(s) of the workload (S1xS2 {shape[0]}x{shape[1]}), "
                      f"{secs:.1f} s of CPU time, same flop convention"}


def reference_arm(args, rank, world):
    from attention_backward_fabwd_gb300 import inputs

    if rank != 0:
        return None
    w = inputs.WORKLOADS[args.workload]
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
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
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
        "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(pb, l2="flushed: 256 MB buffer written between timed steps (untimed)"),
        "dq_mode": "separate" if r["separate"] else "atomic",
        "pct_of_peak": 100.0 * value / world / peak_tf,
        "roofline": {"bound": "tensor", "achieved": dom["TFLOP/s"], "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": dom["TFLOP/s"] / peak_tf, "traffic": profile_traffic(w.name, dom["kernel"]),
                     "kernel": dom["kernel"], "peak_kind": f"{peak_kind} bf16 dense (burst)",
                     "algorithmic_flops_per_launch": dom["flops"], "ms_per_launch": dom["ms"],
                     "flops_per_pair": dom["flops_per_pair"]},
        "kernels": stages,
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
