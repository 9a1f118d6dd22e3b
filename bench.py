#!/usr/bin/env python
"""Benchmark of blockwise ring attention on GB300 (prints ONE JSON line).

A step is one pass of the whole hot path on the default workload: the causal
bf16 forward AND backward at batch 1, seq 65536, 32 heads, head_dim 128, 8
virtual ring shards (ra_fwd then ra_bwd).  The same run also times the
long-context forward (seq 131072, 32 heads, 16 shards) and reports it under
"fwd_s131072", and decoding one new token against that 131072-token K/V as
a full KV cache (ra_decode, HBM-bound) under "decode_s131072", and the blockwise
feed-forward at the 7B shape (ra_blockwise_ffn) under "ffn_7b".  Inputs are
seeded synthetic N(0,1) bf16 tensors, resident in
HBM before the timed region; every input set is larger than the 129 MB L2, so
no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the full workload on its own GPU as an
independent replica (the problem's batch x head units shard with no exchange);
the time is the max over ranks and `value` counts the work of all ranks.
`--impl reference` times the CPU float64 oracle on the host cores instead
(rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from long_context_exact_ra_gb300 import flops as F  # noqa: E402
from long_context_exact_ra_gb300.inputs import (DECODE_WORKLOADS, FFN_WORKLOADS, WORKLOADS,  # noqa: E402
                                                decode_cache_idx, make_ffn_inputs, make_inputs, tensor)

METRIC = "attention TFLOP/s (causal bf16 fwd/bwd, 1xGB300) and % of dense BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(mhz)}


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "long_context_exact_ra_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profile_traffic(key: str, sha: str):
    """DRAM bytes per launch recorded from an ncu capture in profiles/*.md, or None
    if absent or taken on a different kernel source."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    pat = re.compile(r"traffic:\s*key=(\S+)\s+bytes_per_launch=([0-9.eE+]+)\s+source_sha256=(\w+)")
    for fn in sorted(os.listdir(d)):
        if not fn.endswith(".md"):
            continue
        for line in open(os.path.join(d, fn)):
            m = pat.search(line)
            if m and m.group(1) == key and m.group(3) == sha:
                return float(m.group(2))
    return None


def max_over_ranks(x: float, ws: int, device=None) -> float:
    """Max of a per-rank scalar (step time) over all ranks; identity on one rank."""
    if ws <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(ws: int, flops_per_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every replica does flops_per_step in the (max-over-ranks) step time."""
    return ws * flops_per_step / (ms_per_step * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------------------- GPU arm
def to_dev(x, torch, dev):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)


def to_pinned(x, torch):
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory()


def time_fwd(ops, torch, w, steps, warmup, dev, keep_kv=False, with_seg=False):
    """Forward-only timing of workload w (device-resident inputs, with the
    workload's segment ids when it has them).  With keep_kv the device K and V are
    returned too (the decode leg reads them as its cache); with with_seg the host
    segment ids are returned too."""
    x = make_inputs(w, with_dout=False)
    q, k, v = (to_dev(getattr(x, n), torch, dev) for n in ("q", "k", "v"))
    seg_h = x.segment_ids
    seg = torch.from_numpy(np.ascontiguousarray(seg_h)).to(dev) if seg_h is not None else None
    del x
    out = torch.empty_like(q)
    lse = torch.empty((w.batch, w.heads, w.seq), dtype=torch.float32, device=dev)
    args = (seg, w.causal_block_size, w.num_shards, w.query_chunk_size, w.key_chunk_size)
    for _ in range(warmup):
        ops.fwd(q, k, v, *args, out=out, lse=lse)
    ops.sync_check()
    st = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(st)
        ops.fwd(q, k, v, *args, out=out, lse=lse)
        b.record(st)
    torch.cuda.synchronize()
    ops.sync_check()
    ms = [a.elapsed_time(b) for a, b in evs]
    fl = F.fwd_flops_nominal(w.batch, w.seq, w.heads, w.head_dim, w.causal_block_size > 0)
    if keep_kv:
        return fl, ms, (k, v)
    if with_seg:
        return fl, ms, seg_h
    return fl, ms


def time_decode(ops, torch, wd, kv, iters, warmup, dev):
    """ra_decode of the decode workload wd against the device cache kv = (k, v)
    ([B, S, H, D] bf16, S = wd.cache_len); the new tokens' q is drawn from the
    decode inputs' own stream.  Returns (ms per call, algorithmic bytes per call)."""
    k, v = kv
    B, T, S, H, D = wd.batch, wd.new_tokens, wd.cache_len, wd.heads, wd.head_dim
    assert tuple(k.shape) == (B, S, H, D)
    q = to_dev(tensor(wd.seed, 4, (B, T, H, D), wd.scale, wd.dtype), torch, dev)
    idx_h = decode_cache_idx(wd.seed, B, T, S, wd.fill)
    idx = torch.from_numpy(idx_h).to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev)
    work = torch.empty(max(16, ops.decode_workspace_size(B, T, S, H, D, wd.num_shards, torch.bfloat16)),
                       dtype=torch.uint8, device=dev)
    call = lambda: ops.decode(q, k, v, idx, None, None, wd.causal_block_size, wd.num_shards,  # noqa: E731
                              out=out, lse=lse, workspace=work)
    for _ in range(warmup):
        call()
    ops.sync_check()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(iters):
        call()
    e1.record(st)
    torch.cuda.synchronize()
    ops.sync_check()
    filled = np.clip(idx_h.astype(np.int64) + T, 0, S)
    byts = int(filled.sum()) * H * D * 2 * 2  # K and V rows of the filled cache, bf16
    return e0.elapsed_time(e1) / iters, byts


def run_e2e(args, torch, d, host, names, step, out, lse, backward, grads, st, ws, dev):
    """Same step through the public API with host buffers: H2D of the inputs from
    pinned memory, the step, D2H of every result, all inside the timed region."""
    B, S, H, _ = d["q"].shape
    hout = {n: torch.empty(d["q"].shape, dtype=torch.bfloat16).pin_memory()
            for n in (("out", "dq", "dk", "dv") if backward else ("out",))}
    hlse = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def e2e_step():
        for n in names:
            d[n].copy_(host[n], non_blocking=True)
        step()
        hout["out"].copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)
        if backward:
            hout["dq"].copy_(grads[0], non_blocking=True)
            hout["dk"].copy_(grads[1], non_blocking=True)
            hout["dv"].copy_(grads[2], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record(st)
    for _ in range(args.steps):
        e2e_step()
    e1.record(st)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, ws, dev)
    h2d = sum(host[n].numel() * host[n].element_size() for n in names)
    d2h = sum(t.numel() * 2 for t in hout.values()) + hlse.numel() * 4
    return e2e_ms, h2d, d2h


def workload_for(args):
    w = WORKLOADS[args.workload]
    if args.seq:  # a smaller case of the same workload (profiling); chunks shrink to fit the shard
        ssh = args.seq // w.num_shards
        ch = min(w.query_chunk_size, ssh)
        w = w.with_(name=f"{w.name} at seq {args.seq}", seq=args.seq, query_chunk_size=ch, key_chunk_size=ch)
    return w


def gpu_arm(args, peaks, peaks_src):
    import torch

    from long_context_exact_ra_gb300 import ops

    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    ops.lib()
    w = workload_for(args)
    backward = w.backward
    x = make_inputs(w, with_dout=backward)
    names = ("q", "k", "v") + (("dout",) if backward else ())
    host = {n: to_pinned(getattr(x, n), torch) for n in names}
    seg_h = x.segment_ids
    del x
    d = {n: host[n].to(dev) for n in names}
    if seg_h is not None:  # packed documents: the segment ids are an input like q, k, v
        host["seg"] = torch.from_numpy(np.ascontiguousarray(seg_h)).pin_memory()
        d["seg"] = host["seg"].to(dev)
        names = names + ("seg",)
    B, S, H, D = w.shape
    out = torch.empty_like(d["q"])
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    cargs = (d.get("seg"), w.causal_block_size, w.num_shards, w.query_chunk_size, w.key_chunk_size)
    if backward:
        dq, dk, dv = (torch.empty_like(d["q"]) for _ in range(3))
        wsz = ops.bwd_workspace_size(B, S, H, D, torch.bfloat16)
        work = torch.empty(wsz, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(rec=None):
        if rec is not None:
            rec[0].record(st)
        ops.fwd(d["q"], d["k"], d["v"], *cargs, out=out, lse=lse)
        if rec is not None:
            rec[1].record(st)
        if backward:
            ops.bwd(d["q"], d["k"], d["v"], out, lse, d["dout"], *cargs, dq=dq, dk=dk, dv=dv, workspace=work)
            if rec is not None:
                rec[2].record(st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ops.sync_check()
    if ws > 1:
        torch.distributed.barrier()
    recs = [(ev(), ev(), ev()) for _ in range(args.steps)]
    t0, t1 = ev(), ev()
    launches0 = ops.kernel_launches()
    try:
        sel = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        sel = str(local)
    clocks = ClockSampler(sel)
    clocks.start()
    torch.cuda.synchronize()
    t0.record(st)
    for i in range(args.steps):
        step(recs[i])
    t1.record(st)
    torch.cuda.synchronize()
    clk = clocks.stop()
    launches = ops.kernel_launches() - launches0
    ops.sync_check()
    total_ms = max_over_ranks(t0.elapsed_time(t1), ws, dev)
    fwd_ms = statistics.mean(r[0].elapsed_time(r[1]) for r in recs)
    bwd_ms = statistics.mean(r[1].elapsed_time(r[2]) for r in recs) if backward else 0.0
    causal = w.causal_block_size > 0
    fl_f = F.fwd_flops_nominal(B, S, H, D, causal)
    fl_b = F.bwd_flops_nominal(B, S, H, D, causal) if backward else 0.0
    per_step = fl_f + fl_b
    ms_step = total_ms / args.steps
    value = whole_job_tflops(ws, per_step, ms_step)

    # end-to-end through the public API with host buffers (copies inside the timed region)
    if args.no_e2e:
        e2e_ms, h2d, d2h = float("nan"), 0, 0
    else:
        e2e_ms, h2d, d2h = run_e2e(args, torch, d, host, names, step, out, lse, backward,
                                   (dq, dk, dv) if backward else None, st, ws, dev)

    peak = peaks["bf16_tflops"]
    peak_s = peaks.get("bf16_tflops_sustained", peak)
    fwd_tf = fl_f / (fwd_ms * 1e-3) / 1e12
    # visible-pair work (differs from the nominal formula when segments mask most of the square)
    fl_vis = F.fwd_flops_visible(B, S, H, D, w.causal_block_size, seg_h) if seg_h is not None else None
    fwd_sha = source_sha("attn_fwd_sm103.cu", "sm103.cuh")
    roof_fwd = {"bound": "tensor", "kernel": f"fwd_bf16_kernel<{D}>", "achieved": round(fwd_tf, 1),
                "peak": peak, "unit": UNIT, "frac": round(fwd_tf / peak, 4),
                "frac_sustained": round(fwd_tf / peak_s, 4), "peak_source": peaks_src,
                "traffic": profile_traffic(f"fwd{D}_cfg{args.workload}", fwd_sha),
                "ms_per_launch": round(fwd_ms, 3), "flops_per_launch": fl_f}
    if fl_vis is not None:
        vis_tf = fl_vis / (fwd_ms * 1e-3) / 1e12
        roof_fwd.update({"visible_flops_per_launch": fl_vis, "achieved_visible": round(vis_tf, 1),
                         "frac_visible": round(vis_tf / peak, 4)})
    roofline = roof_fwd
    extra = {}
    if backward:
        bwd_tf = fl_b / (bwd_ms * 1e-3) / 1e12
        bwd_sha = source_sha("attn_bwd_sm103.cu", "sm103.cuh")
        roof_bwd = {"bound": "tensor", "kernel": "ra_bwd (preprocess + main + finalize)",
                    "achieved": round(bwd_tf, 1), "peak": peak, "unit": UNIT, "frac": round(bwd_tf / peak, 4),
                    "frac_sustained": round(bwd_tf / peak_s, 4), "peak_source": peaks_src,
                    "traffic": profile_traffic(f"bwd{D}_cfg{args.workload}", bwd_sha),
                    "ms_per_launch": round(bwd_ms, 3), "flops_per_launch": fl_b}
        if bwd_ms >= fwd_ms:
            roofline, extra["roofline_fwd"] = roof_bwd, roof_fwd
        else:
            extra["roofline_bwd"] = roof_bwd
    # the long-context forward target (seq 131072), same run
    if args.workload != 4 and not args.no_secondary:
        del d, host, out, lse
        if backward:
            del dq, dk, dv, work
        torch.cuda.empty_cache()
        w4 = WORKLOADS[4]
        fl4, ms4, kv4 = time_fwd(ops, torch, w4, max(3, args.steps), args.warmup, dev, keep_kv=True)
        tf4 = fl4 / (statistics.mean(ms4) * 1e-3) / 1e12
        extra["fwd_s131072"] = {"workload": w4.name, "tflops": round(tf4, 1), "frac": round(tf4 / peak, 4),
                                "frac_sustained": round(tf4 / peak_s, 4), "ms": round(statistics.mean(ms4), 3),
                                "flops": fl4,
                                "traffic": profile_traffic("fwd128_cfg4", fwd_sha)}
        # decode: one new token against that 131072-token K/V as a full cache (HBM-bound)
        wd = DECODE_WORKLOADS["7b"]
        dms, dbytes = time_decode(ops, torch, wd, kv4, max(20, 10 * args.steps), max(3, args.warmup), dev)
        del kv4
        gbs = dbytes / (dms * 1e-3) / 1e9
        hbm = peaks["hbm_gbs"]
        dec_sha = source_sha("decode_sm103.cu")
        extra["decode_s131072"] = {
            "workload": wd.name, "ms": round(dms, 4), "tokens_per_s": round(wd.batch * wd.new_tokens / (dms * 1e-3), 1),
            "roofline": {"bound": "hbm", "kernel": "ra_decode (partial + combine)", "achieved": round(gbs, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4), "peak_source": peaks_src,
                         "algorithmic_bytes": dbytes,
                         "traffic": profile_traffic("decode128_7b", dec_sha)}}
        # the other forward evaluation workloads: causal B2 S8192 (config 2) and packed documents (config 3)
        for cfg in (2, 3):
            if cfg == args.workload:
                continue
            wc = WORKLOADS[cfg]
            flc, msc, segc = time_fwd(ops, torch, wc, max(10, args.steps), max(3, args.warmup), dev, with_seg=True)
            msm = statistics.mean(msc)
            tfc = flc / (msm * 1e-3) / 1e12
            line = {"workload": wc.name, "ms": round(msm, 4), "ms_min": round(min(msc), 4),
                    "roofline": {"bound": "tensor", "kernel": f"fwd_bf16_kernel<{wc.head_dim}>",
                                 "achieved": round(tfc, 1), "peak": peak, "unit": UNIT,
                                 "frac": round(tfc / peak, 4), "frac_sustained": round(tfc / peak_s, 4),
                                 "peak_source": peaks_src, "flops_per_launch": flc,
                                 "traffic": profile_traffic(f"fwd{wc.head_dim}_cfg{cfg}", fwd_sha)}}
            if segc is not None:  # packed documents: the visible pairs are the honest work
                flv = F.fwd_flops_visible(wc.batch, wc.seq, wc.heads, wc.head_dim, wc.causal_block_size, segc)
                tfv = flv / (msm * 1e-3) / 1e12
                line["roofline"].update({"visible_flops_per_launch": flv, "achieved_visible": round(tfv, 1),
                                         "frac_visible": round(tfv / peak, 4), "frac": round(tfv / peak, 4),
                                         "frac_sustained": round(tfv / peak_s, 4),
                                         "achieved": round(tfv, 1), "achieved_nominal": round(tfc, 1),
                                         "note": "achieved and frac count visible pairs only"})
            extra[f"fwd_cfg{cfg}"] = line
        # blockwise feed-forward at the 7B shape (the other half of a blockwise transformer layer)
        wf = FFN_WORKLOADS["7b"]
        fms, ffl = time_ffn(ops, torch, wf, max(5, args.steps), max(3, args.warmup), dev)
        ftf = ffl / (fms * 1e-3) / 1e12
        extra["ffn_7b"] = {
            "workload": wf.name, "ms": round(fms, 3),
            "roofline": {"bound": "tensor", "kernel": "gemm_bias_act_kernel (2 launches per chunk)",
                         "achieved": round(ftf, 1), "peak": peak, "unit": UNIT, "frac": round(ftf / peak, 4),
                         "frac_sustained": round(ftf / peak_s, 4), "peak_source": peaks_src,
                         "flops_per_launch": ffl,
                         "traffic": profile_traffic("ffn_7b", source_sha("ffn_sm103.cu", "sm103.cuh"))}}
        # the ring across devices, all ranks' steps on this one GPU (device work of the ring-step kernels)
        extra["ring_local_s65536"] = time_ring_local(ops, torch, WORKLOADS[5], max(2, args.steps // 2), dev, peak)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, no dataset)",
        "config": {"workload": w.name, "batch": B, "seq": S, "heads": H, "head_dim": D,
                   "num_shards": w.num_shards, "causal_block_size": w.causal_block_size,
                   "query_chunk_size": w.query_chunk_size, "key_chunk_size": w.key_chunk_size,
                   "step": "ra_fwd + ra_bwd" if backward else "ra_fwd",
                   "flops_per_step": per_step, "flop_convention": "4*b*h*s*s*d, /2 causal; bwd = 2.5x fwd",
                   "l2": "inputs larger than L2 (no flush needed)", "parallelism": f"replicas x{ws}"},
        "e2e": None if args.no_e2e else {"value": round(whole_job_tflops(ws, per_step, e2e_ms), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3)},
        "gpu_launches": launches,
        "roofline": roofline,
        "clocks": clk,
        **extra,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_seconds)
        if "decode_s131072" in result:
            result["decode_s131072"]["cpu_baseline"] = cpu_baseline_decode(DECODE_WORKLOADS["7b"])
        if "ffn_7b" in result:
            result["ffn_7b"]["cpu_baseline"] = cpu_baseline_ffn(FFN_WORKLOADS["7b"])
    if args.seq:
        result["config"]["note"] = "reduced seq for profiling: not the benchmark workload"
    if ws > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def decode_arm(args, peaks, peaks_src):
    """--decode-only: the decode leg alone (profiling; cache_len = --seq, default 131072)."""
    import torch

    from long_context_exact_ra_gb300 import ops
    from long_context_exact_ra_gb300.inputs import make_decode_inputs

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ops.lib()
    wd = DECODE_WORKLOADS["7b"]
    if args.seq:
        wd = wd.with_(name=f"{wd.name} at cache_len {args.seq}", cache_len=args.seq)
    x = make_decode_inputs(wd)
    kv = (to_dev(x.k_cache, torch, dev), to_dev(x.v_cache, torch, dev))
    del x
    dms, dbytes = time_decode(ops, torch, wd, kv, max(1, args.steps), max(1, args.warmup), dev)
    gbs = dbytes / (dms * 1e-3) / 1e9
    hbm = peaks["hbm_gbs"]
    print(json.dumps({"metric": "decode KV-cache read GB/s (ra_decode)", "value": round(gbs, 1), "unit": "GB/s",
                      "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dms, 4),
                      "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16)",
                      "config": {"workload": wd.name, "note": "decode leg alone, for profiling"},
                      "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                                   "frac": round(gbs / hbm, 4), "peak_source": peaks_src,
                                   "algorithmic_bytes": dbytes}}), flush=True)


def time_ring_local(ops, torch, w, iters, dev, peak):
    """The fwd+bwd workload as a ring of N = w.num_shards ranks run one after another on
    this GPU (ring.ring_forward_local / ring_backward_local): every ring-step kernel
    launch of every rank, contiguous and striped blocks.  This is the device work a
    rank does summed over the ring (no transfers), not the step time of a ring of
    N GPUs; the FLOPs are the workload's."""
    from long_context_exact_ra_gb300 import ring
    x = make_inputs(w, with_dout=True)
    q, k, v, do = (to_dev(getattr(x, n), torch, dev) for n in ("q", "k", "v", "dout"))
    del x
    B, S, H, D = q.shape
    fl_f = F.fwd_flops_nominal(B, S, H, D, True)
    fl_b = F.bwd_flops_nominal(B, S, H, D, True)
    res = {"workload": f"{w.name}, as a ring of {w.num_shards} ranks on one GPU", "ranks": w.num_shards}
    st = torch.cuda.current_stream()
    for layout in ring.LAYOUTS:
        n0 = ops.kernel_launches()
        out, lse = ring.ring_forward_local(q, k, v, None, 1, w.num_shards, layout)  # warm-up
        ring.ring_backward_local(q, k, v, out, lse, do, None, 1, w.num_shards, layout)
        launches = ops.kernel_launches() - n0
        ops.sync_check()
        tf, tb = [], []
        for _ in range(iters):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(st)
            out, lse = ring.ring_forward_local(q, k, v, None, 1, w.num_shards, layout)
            e[1].record(st)
            ring.ring_backward_local(q, k, v, out, lse, do, None, 1, w.num_shards, layout)
            e[2].record(st)
            torch.cuda.synchronize()
            tf.append(e[0].elapsed_time(e[1]))
            tb.append(e[1].elapsed_time(e[2]))
        ops.sync_check()
        mf, mb = statistics.mean(tf), statistics.mean(tb)
        res[layout] = {"fwd_ms": round(mf, 3), "bwd_ms": round(mb, 3),
                       "fwd_tflops": round(fl_f / (mf * 1e-3) / 1e12, 1), "bwd_tflops": round(fl_b / (mb * 1e-3) / 1e12, 1),
                       "fwd_frac": round(fl_f / (mf * 1e-3) / 1e12 / peak, 4),
                       "bwd_frac": round(fl_b / (mb * 1e-3) / 1e12 / peak, 4),
                       "launches_per_fwd_bwd": launches,
                       "note": "timed region includes the carries' allocation and the host-side block shuffles"}
    return res


def time_ffn(ops, torch, wf, iters, warmup, dev):
    """ra_blockwise_ffn on workload wf (device-resident inputs); returns (ms per call, FLOPs per call)."""
    xi = make_ffn_inputs(wf)
    x, w1, w2 = (to_dev(a, torch, dev) for a in (xi.x, xi.w1, xi.w2))
    b1 = torch.from_numpy(xi.b1).to(dev) if xi.b1 is not None else None
    b2 = torch.from_numpy(xi.b2).to(dev) if xi.b2 is not None else None
    del xi
    out = torch.empty_like(x)
    work = torch.empty(ops.ffn_workspace_size(wf.batch, wf.seq, wf.ffn_dim, wf.chunk_size), dtype=torch.uint8,
                       device=dev)
    for _ in range(warmup):
        ops.blockwise_ffn(x, w1, b1, w2, b2, wf.chunk_size, out=out, workspace=work)
    ops.sync_check()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(iters):
        ops.blockwise_ffn(x, w1, b1, w2, b2, wf.chunk_size, out=out, workspace=work)
    e1.record(st)
    torch.cuda.synchronize()
    ops.sync_check()
    flops = 2.0 * 2 * wf.batch * wf.seq * wf.model_dim * wf.ffn_dim  # two products
    return e0.elapsed_time(e1) / iters, flops


def ffn_arm(args, peaks, peaks_src):
    """--ffn-only: the blockwise feed-forward leg alone (profiling; rows = --seq, default 16384)."""
    import torch

    from long_context_exact_ra_gb300 import ops

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ops.lib()
    wf = FFN_WORKLOADS["7b"]
    if args.seq:
        wf = wf.with_(name=f"{wf.name} at {args.seq} rows", seq=args.seq, chunk_size=min(wf.chunk_size, args.seq))
    fms, ffl = time_ffn(ops, torch, wf, max(1, args.steps), max(1, args.warmup), dev)
    tf = ffl / (fms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    print(json.dumps({"metric": "blockwise feed-forward TFLOP/s (ra_blockwise_ffn)", "value": round(tf, 1),
                      "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": round(fms, 3), "higher_is_better": True, "dtype": "bf16",
                      "data": "synthetic (seeded, no dataset)",
                      "config": {"workload": wf.name, "note": "feed-forward leg alone, for profiling"},
                      "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak, "unit": UNIT,
                                   "frac": round(tf / peak, 4), "peak_source": peaks_src,
                                   "flops_per_launch": ffl}}), flush=True)


# ----------------------------------------------------------------------------- CPU oracle
def blas_threads():
    """Threads numpy's BLAS (which runs the oracle's float64 products) uses: from
    threadpoolctl when installed, else from the OpenBLAS query function of the
    library numpy ships; None when neither is available."""
    try:
        import threadpoolctl
        for info in threadpoolctl.threadpool_info():
            if info.get("user_api") == "blas":
                return int(info["num_threads"])
    except Exception:
        pass
    import ctypes
    import glob
    libdir = os.path.join(os.path.dirname(np.__file__), os.pardir, "numpy.libs")
    for path in sorted(glob.glob(os.path.join(libdir, "*openblas*"))):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for name in ("scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads",
                     "openblas_get_num_threads64_", "openblas_get_num_threads"):
            fn = getattr(lib, name, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    return None


def oracle_threads():
    """(cores the oracle runs on, BLAS threads or None): the BLAS thread count
    capped by the CPUs this process may use."""
    cpus = len(os.sched_getaffinity(0))
    bt = blas_threads()
    return (min(cpus, bt) if bt else cpus), bt


def oracle_rows_rate(w, budget_s, x=None, start_rows=32):
    """Time the float64 oracle on sampled query rows of workload w; return
    (algorithmic TFLOP/s, rows, seconds, cores)."""
    import oracle

    if x is None:
        x = make_inputs(w, with_dout=False)
    from long_context_exact_ra_gb300.inputs import bf16_bits_to_f32
    q, k, v = (bf16_bits_to_f32(getattr(x, n)) for n in ("q", "k", "v"))
    g = np.random.Generator(np.random.PCG64(7))
    n, total_t, total_f, total_rows = start_rows, 0.0, 0.0, 0
    c = w.causal_block_size
    while total_t < budget_s:
        bh = (int(g.integers(w.batch)), int(g.integers(w.heads)))
        rows = np.stack([np.full(n, bh[0]), np.full(n, bh[1]), g.integers(w.seq, size=n)], 1)
        t = time.perf_counter()
        oracle.ref_fwd_rows(q, k, v, rows, x.segment_ids, c)
        total_t += time.perf_counter() - t
        if x.segment_ids is not None:  # count the keys each sampled row actually sees
            kpos = np.arange(w.seq)
            seg = x.segment_ids[bh[0]]
            for i in rows[:, 2]:
                ok = seg == seg[i]
                if c > 0:
                    ok &= (kpos // c) <= (i // c)
                total_f += 4.0 * w.head_dim * np.count_nonzero(ok)
        elif c > 0:
            vis = ((rows[:, 2] // c) + 1) * c
            total_f += 4.0 * w.head_dim * np.minimum(vis, w.seq).sum()
        else:
            total_f += 4.0 * w.head_dim * w.seq * n
        total_rows += n
        n = min(n * 2, 4096)
    return total_f / total_t / 1e12, total_rows, total_t, oracle_threads()[0]


def oracle_bwd_rate(w, budget_s, x=None, prefix=8192):
    """Time the float64 backward oracle (ref_bwd_head_blocked) on whole heads of a
    prefix of workload w: the first `prefix` positions of a drawn (b, h) head are
    a complete attention problem of their own under the causal mask (no query of
    the prefix sees a later key).  Returns (algorithmic TFLOP/s of the backward
    under the metric's convention, heads, seconds)."""
    import oracle

    from long_context_exact_ra_gb300.inputs import bf16_bits_to_f32
    if x is None:
        x = make_inputs(w, with_dout=True)
    n = min(prefix, w.seq) if w.causal_block_size > 0 else w.seq
    g = np.random.Generator(np.random.PCG64(8))
    rows = np.arange(n)
    total_t, total_f, heads = 0.0, 0.0, 0
    while total_t < budget_s or heads == 0:
        b, h = int(g.integers(w.batch)), int(g.integers(w.heads))
        Q, K, V, dO = (bf16_bits_to_f32(getattr(x, a)[b, :n, h]).astype(np.float64) for a in ("q", "k", "v", "dout"))
        seg = None if x.segment_ids is None else x.segment_ids[b, :n]
        t0 = time.perf_counter()
        oracle.ref_bwd_head_blocked(Q, K, V, dO, seg, w.causal_block_size, rows, rows, block=2048)
        total_t += time.perf_counter() - t0
        total_f += F.bwd_flops_nominal(1, n, 1, w.head_dim, w.causal_block_size > 0)
        heads += 1
    return total_f / total_t / 1e12, heads, total_t, n


def oracle_step_rate(w, budget_s, x=None):
    """CPU oracle rate for one step of workload w: the forward on sampled query rows
    and, for a forward+backward workload, the backward on whole prefix heads; the
    step's FLOPs divided by the time the two rates imply for them."""
    tf_f, rows, secs_f, cores = oracle_rows_rate(w, budget_s / (2 if w.backward else 1), x)
    fl_f = F.fwd_flops_nominal(w.batch, w.seq, w.heads, w.head_dim, w.causal_block_size > 0)
    if not w.backward:
        return tf_f, cores, (f"float64 oracle forward on {rows} sampled query rows of '{w.name}' "
                             f"(full key range per row, {secs_f:.1f} s); algorithmic FLOPs of the visible pairs")
    tf_b, heads, secs_b, n = oracle_bwd_rate(w, budget_s / 2, x)
    fl_b = F.bwd_flops_nominal(w.batch, w.seq, w.heads, w.head_dim, w.causal_block_size > 0)
    value = (fl_f + fl_b) / (fl_f / (tf_f * 1e12) + fl_b / (tf_b * 1e12)) / 1e12
    return value, cores, (f"float64 oracle: forward on {rows} sampled query rows of '{w.name}' ({secs_f:.1f} s, "
                          f"{tf_f:.4f} TFLOP/s) and backward on {heads} whole heads of its first {n} positions "
                          f"({secs_b:.1f} s, {tf_b:.4f} TFLOP/s); combined over the step's forward and backward "
                          f"FLOPs (bwd = 2.5x fwd)")


def cpu_baseline(w, budget_s=15.0):
    value, cores, sample = oracle_step_rate(w, budget_s)
    return {"value": value, "unit": UNIT, "cores": cores, "blas_threads": oracle_threads()[1], "kind": "oracle",
            "sample": sample}


def cpu_baseline_decode(wd, budget_s=5.0, cache_len=16384):
    """The float64 decode oracle on one new token per sampled head against a cache of
    `cache_len` entries (the decode workload's layout and distributions, a shorter
    cache); reported as GB/s of K/V cache processed, the decode leg's unit."""
    import oracle

    from long_context_exact_ra_gb300.inputs import bf16_bits_to_f32, make_decode_inputs
    w = wd.with_(cache_len=cache_len)
    x = make_decode_inputs(w)
    q = bf16_bits_to_f32(x.q).astype(np.float64)
    g = np.random.Generator(np.random.PCG64(11))
    t_sum, byts, rows = 0.0, 0, 0
    while t_sum < budget_s:
        h = int(g.integers(w.heads))
        t0 = time.perf_counter()
        oracle.ref_decode_rows(q, x.k_cache, x.v_cache, x.cache_idx, np.array([[0, h, 0]]), w.causal_block_size)
        t_sum += time.perf_counter() - t0
        byts += 2 * cache_len * w.head_dim * 2
        rows += 1
    cores, bt = oracle_threads()
    return {"value": byts / t_sum / 1e9, "unit": "GB/s", "cores": cores, "blas_threads": bt, "kind": "oracle",
            "sample": f"float64 decode oracle on {rows} (head, token) rows against a {cache_len}-entry cache of "
                      f"the same layout ({t_sum:.1f} s); bytes = the bf16 K/V rows each row reads"}


def cpu_baseline_ffn(wf, budget_s=5.0):
    """The float64 feed-forward oracle on sampled rows of the feed-forward workload (TFLOP/s)."""
    import oracle

    from long_context_exact_ra_gb300.inputs import make_ffn_inputs
    xi = make_ffn_inputs(wf)
    w1, w2 = xi.as_f64("w1"), xi.as_f64("w2")
    b1 = xi.as_f64("b1") if xi.b1 is not None else np.zeros(wf.ffn_dim)
    b2 = xi.as_f64("b2") if xi.b2 is not None else np.zeros(wf.model_dim)
    xflat = xi.as_f64("x").reshape(-1, wf.model_dim)
    g = np.random.Generator(np.random.PCG64(12))
    t_sum, rows = 0.0, 0
    while t_sum < budget_s:
        r = g.integers(wf.batch * wf.seq, size=16)
        xr = xflat[r]
        t0 = time.perf_counter()
        oracle.ffn_rows(xr, w1, b1, w2, b2)
        t_sum += time.perf_counter() - t0
        rows += len(r)
    flops = 2.0 * 2 * rows * wf.model_dim * wf.ffn_dim
    cores, bt = oracle_threads()
    return {"value": flops / t_sum / 1e12, "unit": UNIT, "cores": cores, "blas_threads": bt, "kind": "oracle",
            "sample": f"float64 feed-forward oracle on {rows} sampled rows of '{wf.name}' ({t_sum:.1f} s)"}


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    w = workload_for(args)
    x = make_inputs(w, with_dout=w.backward)
    per_step = max(4.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_step_rate(w, per_step, x)
    rates, secs = [], 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        tf, cores, sample = oracle_step_rate(w, per_step, x)
        secs += time.perf_counter() - t0
        rates.append(tf)
    value = statistics.mean(rates)
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1) bf16 inputs, computed in float64)",
           "config": {"workload": w.name, "batch": w.batch, "seq": w.seq, "heads": w.heads,
                      "head_dim": w.head_dim, "num_shards": w.num_shards},
           "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle", "cores": cores,
                            "blas_threads": oracle_threads()[1],
                            "sample": f"each step (~{per_step:.0f} s): {sample}"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, choices=[2, 3, 4, 5], default=5)
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode leg (cache_len = --seq, default 131072); for profiling")
    ap.add_argument("--ffn-only", action="store_true",
                    help="time only the blockwise feed-forward leg (rows = --seq, default 16384); for profiling")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the seq-131072 forward, decode and feed-forward lines")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--seq", type=int, default=0, help="run a smaller seq of the workload (profiling)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    peaks, src = load_peaks()
    if args.impl == "reference":
        reference_arm(args)
    elif args.decode_only:
        decode_arm(args, peaks, src)
    elif args.ffn_only:
        ffn_arm(args, peaks, src)
    else:
        gpu_arm(args, peaks, src)


if __name__ == "__main__":
    main()
