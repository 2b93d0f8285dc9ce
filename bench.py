"""Benchmark of the GatedDeltaNet layer on GB300.

One step = one ``gdn_prefill`` call over the long packed prefill (131072
tokens = 16 sequences x 8192, H_qk = 16, H_v = 32, d_k = d_v = 128, bf16
streams, fp32 state, final state returned), the largest single-GPU workload,
inputs resident in HBM, L2 flushed between steps.  Prints one JSON line.  Also
measured, in ``extra``: the 4096-token single-sequence prefill, the
32768-token varlen prefill and the 256-sequence decode step, each with its
roofline fraction and per-kernel split.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick]

Under torchrun (N > 1) every rank runs its own copy of the workload on its
own GPU (sequences are independent: no data-path collective), the per-step
time is the max over ranks and ``value`` counts the tokens of all ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead
(rank 0 only), each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gateddeltanet_layer_gb300 import synth  # noqa: E402

METRIC = "GatedDeltaNet prefill tokens/s & decode seqs/s on 1 GB300; % of roofline"
BYTES_PER_TOKEN = 32896          # q 4096 + k 4096 + v 8192 + z 8192 + a 64 + b 64 + out 8192 (bf16)
STATE_BYTES = 32 * 128 * 128 * 4  # one sequence's fp32 state, all 32 value heads
FLOPS_PER_TOKEN = 32 * (10 * 64 * 128 + 6 * 128 * 128)
DECODE_BYTES_PER_SEQ = 2 * STATE_BYTES + 32896 + 2 * 8192 * 3 * 2
DECODE_FLOPS_PER_SEQ = 32 * 6 * 128 * 128
L2_FLUSH_BYTES = 512 << 20


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def prefill_work(cfg) -> tuple[int, float]:
    """Algorithmic bytes and flops of one prefill call (streams, states, no intermediates):
    per token q, k [h_qk, d_k], v, z and out [h_v, d_v], a, b [h_v] in the stream dtype; per
    sequence the fp32 state [h_v, d_k, d_v] written (and read when there is an initial one).
    32,896 B and FLOPS_PER_TOKEN per token at 16/32 heads, d = 128, bf16."""
    es = 4 if cfg.dtype == "fp32" else 2
    per_token = es * (2 * cfg.h_qk * cfg.d_k + 3 * cfg.h_v * cfg.d_v + 2 * cfg.h_v)
    state = 4 * cfg.h_v * cfg.d_k * cfg.d_v
    nbytes = cfg.T * per_token + cfg.N * state               # final state written
    if cfg.init_std > 0:
        nbytes += cfg.N * state                              # initial state read
    flops = float(cfg.T) * cfg.h_v * (10 * 64 * cfg.d_v + 6 * cfg.d_k * cfg.d_v)
    return nbytes, flops


def max_over_ranks(values, device):
    """Elementwise maximum of `values` over the ranks of the default process
    group (the values themselves without one, or with a single rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


# ---------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi SM clock / throttle reasons sampled every 200 ms during a timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz)}


_INPUTS = {}


def inputs_of(cfg):
    """The seeded inputs of a prefill workload, drawn once per run."""
    if cfg.name not in _INPUTS:
        _INPUTS[cfg.name] = synth.make_prefill(cfg)
    return _INPUTS[cfg.name]


# ---------------------------------------------------------------------- GPU arm
def _device_inputs(inp, dev, fp32=False):
    import torch
    t = {}
    sdt = torch.float32 if fp32 else torch.bfloat16
    for key in ("x_q", "x_k", "x_v", "z", "a", "b"):
        t[key] = torch.from_numpy(inp[key]).to(dev).to(sdt)
    for key in ("conv_w", "A_log", "dt_bias", "norm_w"):
        t[key] = torch.from_numpy(inp[key]).to(dev)
    t["cu_seqlens"] = torch.from_numpy(inp["cu_seqlens"]).to(dev)
    t["init_state"] = None if inp.get("init_state") is None else torch.from_numpy(inp["init_state"]).to(dev)
    return t


def time_prefill(cfg, steps, warmup, dev, flush, with_e2e=False, trace=False, seg_chunks=0):
    """Per-step device time (CUDA events on the launching stream, L2 flushed
    between steps) of one gdn_prefill call; optionally the end-to-end time with
    pinned-host inputs copied in and outputs copied out every step, and the
    library's per-kernel trace (CUDA events around each of its launches, on the
    same stream) over as many steps again, run right after the timed ones: the
    trace's events between launches hold back the early start of the next
    kernel (programmatic dependent launch), so they stay out of the timed steps.
    seg_chunks > 0 times gdn_prefill_segmented with segments of that many chunks."""
    import torch

    import gateddeltanet_layer_gb300 as gdn
    inp = inputs_of(cfg)
    fp32 = cfg.dtype == "fp32"
    t = _device_inputs(inp, dev, fp32)
    T, N = cfg.T, cfg.N
    out = torch.empty((T, cfg.h_v, cfg.d_v), dtype=torch.float32 if fp32 else torch.bfloat16, device=dev)
    fs = torch.empty((N, cfg.h_v, cfg.d_k, cfg.d_v), dtype=torch.float32, device=dev)
    if seg_chunks:
        ws_bytes = gdn.prefill_segmented_workspace_bytes(T, N, cfg.h_qk, cfg.h_v, cfg.d_k, cfg.d_v, seg_chunks)
    else:
        ws_bytes = gdn.prefill_workspace_bytes(T, N, cfg.h_qk, cfg.h_v, cfg.d_k, cfg.d_v, not fp32)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        args = (t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"], t["dt_bias"],
                t["norm_w"], t["cu_seqlens"], t["init_state"])
        if seg_chunks:
            gdn.prefill_segmented(*args, seg_chunks=seg_chunks, out=out, final_state=fs, workspace=ws,
                                  stream=stream)
        else:
            gdn.prefill(*args, out=out, final_state=fs, workspace=ws, stream=stream)

    for _ in range(warmup):
        flush.zero_()
        call()
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in ev:
        flush.zero_()
        s.record(stream)
        call()
        e.record(stream)
    torch.cuda.synchronize(dev)
    ms = [s.elapsed_time(e) for s, e in ev]
    kernels = None
    if trace:
        gdn.trace_enable(True)
        gdn.trace_read()
        for _ in range(steps):
            flush.zero_()
            call()
        torch.cuda.synchronize(dev)
        kernels = gdn.trace_read()
        gdn.trace_enable(False)
    status = gdn.workspace_status(ws, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed prefill")
    res = {"ms": ms, "kernels": kernels}
    if with_e2e:
        res["e2e"] = _prefill_e2e(t, cfg, steps, warmup, dev, flush, out, fs, ws, stream)
    del t
    return res


def _prefill_e2e(t, cfg, steps, warmup, dev, flush, out, fs, ws, stream):
    """End-to-end through the public API: every step copies its inputs from
    pinned host memory, runs gdn_prefill and copies out and the final state back
    to pinned host memory.  Steps are pipelined over two device buffer sets and
    three streams (copy-in of step k+1 and copy-out of step k-1 run beside the
    compute of step k), as a serving loop would; the time is from the first
    timed copy-in to the last copy-out, over the timed steps.  No L2 flush here:
    each step's inputs are fresh from the host and its working set (inputs,
    workspace, outputs) exceeds L2."""
    import torch

    import gateddeltanet_layer_gb300 as gdn
    keys = ["x_q", "x_k", "x_v", "z", "a", "b", "cu_seqlens"] + (["init_state"] if t["init_state"] is not None else [])
    # one pinned host buffer and, per buffer set, one device buffer holding every
    # input at 256-byte aligned offsets: one large copy per step
    offs, total = {}, 0
    for k in keys:
        offs[k] = total
        total += (t[k].numel() * t[k].element_size() + 255) // 256 * 256
    host_flat = torch.empty(total, dtype=torch.uint8, pin_memory=True)

    def views(flat):
        return {k: flat[offs[k]:offs[k] + t[k].numel() * t[k].element_size()].view(t[k].dtype).view(t[k].shape)
                for k in keys}
    host = views(host_flat)
    for k in keys:
        host[k].copy_(t[k])
    dev_flat = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    sets = [dict(t), dict(t)]
    for i in range(2):
        sets[i].update(views(dev_flat[i]))
    outs = [(out, fs), (torch.empty_like(out), torch.empty_like(fs))]
    out_h = [(torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
              torch.empty(fs.shape, dtype=fs.dtype, pin_memory=True)) for _ in range(2)]
    h2d = sum(host[k].numel() * host[k].element_size() for k in keys)
    d2h = out.numel() * out.element_size() + fs.numel() * fs.element_size()
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), stream, torch.cuda.Stream(dev)
    ev_cmp = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]
    used = [False, False]

    def step(k):
        i = k % 2
        d = sets[i]
        o, f = outs[i]
        with torch.cuda.stream(s_in):
            if used[i]:
                s_in.wait_event(ev_cmp[i])  # step k-2 has read this input set
            dev_flat[i].copy_(host_flat, non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        s_cmp.wait_event(ev_in)
        if used[i]:
            s_cmp.wait_event(ev_out[i])  # step k-2's results have left this output set
        gdn.prefill(d["x_q"], d["x_k"], d["x_v"], d["a"], d["b"], d["z"], d["conv_w"], d["A_log"], d["dt_bias"],
                    d["norm_w"], d["cu_seqlens"], d["init_state"], out=o, final_state=f, workspace=ws, stream=s_cmp)
        ev_cmp[i].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[i])
            out_h[i][0].copy_(o, non_blocking=True)
            out_h[i][1].copy_(f, non_blocking=True)
            ev_out[i].record(s_out)
        used[i] = True

    for k in range(warmup):
        step(k)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for k in range(warmup, warmup + steps):
        step(k)
    end.record(s_out)
    end.synchronize()
    torch.cuda.synchronize(dev)
    return {"ms": start.elapsed_time(end) / steps, "h2d": h2d, "d2h": d2h, "pipelined": "2 buffer sets, 3 streams"}


def time_backward(cfg, steps, warmup, dev, flush):
    """Per-step device time of one gdn_prefill_backward call (all gradients,
    dy of the output, no final-state gradient), L2 flushed between steps."""
    import torch

    import gateddeltanet_layer_gb300 as gdn
    inp = inputs_of(cfg)
    fp32 = cfg.dtype == "fp32"
    t = _device_inputs(inp, dev, fp32)
    dy = torch.randn((cfg.T, cfg.h_v, cfg.d_v), generator=torch.Generator().manual_seed(1)).to(
        dev, torch.float32 if fp32 else torch.bfloat16)
    ws = torch.empty(gdn.prefill_backward_workspace_bytes(cfg.T, cfg.N, cfg.h_qk, cfg.h_v, cfg.d_k, cfg.d_v),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        gdn.prefill_backward(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                             t["dt_bias"], t["norm_w"], t["cu_seqlens"], dy, t["init_state"], workspace=ws,
                             stream=stream)

    for _ in range(warmup):
        flush.zero_()
        call()
    ms = []
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        call()
        e.record(stream)
        e.synchronize()
        ms.append(s.elapsed_time(e))
    gdn.trace_enable(True)
    gdn.trace_read()
    call()
    torch.cuda.synchronize(dev)
    kernels = {k: v[1] for k, v in gdn.trace_read().items()}
    gdn.trace_enable(False)
    return {"ms": ms, "kernels": kernels}


def time_decode(cfg, steps, warmup, dev, flush):
    import torch

    import gateddeltanet_layer_gb300 as gdn
    inp = synth.make_decode(cfg)
    t = {}
    for key in ("x_q", "x_k", "x_v", "z", "a", "b", "conv_state"):
        t[key] = torch.from_numpy(inp[key]).to(dev).to(torch.bfloat16)
    for key in ("conv_w", "A_log", "dt_bias", "norm_w", "state"):
        t[key] = torch.from_numpy(inp[key]).to(dev)
    out = torch.empty((cfg.batch, cfg.h_v, cfg.d_v), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        gdn.decode_step(t["x_q"], t["x_k"], t["x_v"], t["a"], t["b"], t["z"], t["conv_w"], t["A_log"],
                        t["dt_bias"], t["norm_w"], t["conv_state"], t["state"], out=out, stream=stream)

    for _ in range(warmup):
        flush.zero_()
        call()
    ms = []
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        call()
        e.record(stream)
        e.synchronize()
        ms.append(s.elapsed_time(e))
    return {"ms": ms}


def roofline_of(nbytes, flops, ms, pk, peak_key="hbm_gbs"):
    t = ms * 1e-3
    gbs = nbytes / t / 1e9
    tfl = flops / t / 1e12
    t_roof = max(nbytes / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
    return {"achieved_gbs": gbs, "achieved_tflops": tfl, "roofline_frac": t_roof / t,
            "hbm_frac": gbs / pk["hbm_gbs"]}


HEADLINE = synth.LONG_128K
# A smaller copy of the headline workload (2 of its 16 sequences) for ncu
# captures; per sequence it does the same work, so its DRAM traffic scales to
# the headline call by the number of sequences.
LONG_2X8192 = synth.scaled(synth.LONG_128K, name="prefill_long_T16384", lengths=(8192,) * 2)
# the shapes the token-sequential fp32 kernel serves: more than 8 value heads per q/k head, fp32 streams
GQA16_4K = synth.scaled(synth.SINGLE_4K, name="prefill_T4096_gqa16", h_qk=2)
FP32_4K = synth.scaled(synth.SINGLE_4K, name="prefill_T4096_fp32", dtype="fp32")
PROFILE_CASES = {c.name: c for c in (LONG_2X8192, synth.FEW_CHAINS_16K, GQA16_4K, FP32_4K)}


def prefill_line(cfg, res, steps, pk, dev):
    """Roofline of one prefill workload: the whole call against the slower of
    its byte and flop bounds, and the per-kernel split of the call."""
    ms, = max_over_ranks([statistics.mean(res["ms"])], dev)
    nbytes, flops = prefill_work(cfg)
    rf = roofline_of(nbytes, flops, ms, pk)
    bound = "hbm" if nbytes / pk["hbm_gbs"] >= flops / (pk["bf16_tflops"] * 1e3) else "tensor"
    per_kernel = {}
    traffic = profiled_traffic(cfg)
    kernels = res["kernels"] or {}
    for name, (n, total) in kernels.items():
        k_ms = total / steps
        entry = {"ms_per_call": k_ms, "share_of_traced_call": None, "launches_per_call": n / steps}
        kt = (traffic or {}).get("kernels", {}).get(name)
        if kt is not None:
            entry["dram_bytes_per_call"] = kt
            entry["dram_gbs"] = kt / (k_ms * 1e-3) / 1e9
            entry["dram_frac_of_peak"] = entry["dram_gbs"] / pk["hbm_gbs"]
        per_kernel[name] = entry
    traced = sum(e["ms_per_call"] for e in per_kernel.values())
    for e in per_kernel.values():
        e["share_of_traced_call"] = e["ms_per_call"] / traced if traced > 0 else None
    if bound == "hbm":
        achieved, peak, unit = rf["achieved_gbs"], pk["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = rf["achieved_tflops"], pk["bf16_tflops"], "TFLOP/s"
    return ms, {
        "bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": rf["roofline_frac"],
        "traffic": None if traffic is None else traffic["call"],
        "scope": "whole gdn_prefill call (every kernel it launches)",
        "peak_source": pk["source"] + (" (burst copy)" if bound == "hbm" else " (burst cuBLAS bf16)"),
        "algorithmic_bytes_per_call": nbytes, "algorithmic_flops_per_call": flops,
        "flop_bound_frac": flops / (pk["bf16_tflops"] * 1e12) / (ms * 1e-3),
        "byte_bound_frac": nbytes / (pk["hbm_gbs"] * 1e9) / (ms * 1e-3),
        "per_kernel": per_kernel,
    }


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    pk = peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cfg = HEADLINE

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # ---- the headline: the 131072-token long prefill
    barrier()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0 = time.perf_counter()
        res = time_prefill(cfg, args.steps, args.warmup, dev, flush, with_e2e=True, trace=True)
        barrier()
        wall = time.perf_counter() - t0
    ms, roof = prefill_line(cfg, res, args.steps, pk, dev)
    e2e_ms, = max_over_ranks([res["e2e"]["ms"]], dev)
    launches = int(round(sum(e["launches_per_call"] for e in roof["per_kernel"].values()) * args.steps))

    extra = {}
    if not args.quick:
        for c in (synth.SINGLE_4K, synth.VARLEN_32K):
            n_steps = args.steps
            r = time_prefill(c, n_steps, args.warmup, dev, flush, trace=True)
            m, rl = prefill_line(c, r, n_steps, pk, dev)
            extra[c.name] = {"tokens_per_s": c.T / (m * 1e-3), "ms": m, "roofline_frac": rl["frac"],
                             "achieved_gbs": rl["achieved"] if rl["unit"] == "GB/s" else None,
                             "flop_bound_frac": rl["flop_bound_frac"], "byte_bound_frac": rl["byte_bound_frac"],
                             "per_kernel": rl["per_kernel"], "traffic": rl["traffic"]}
        # the segment-parallel prefill, next to the plain one on the same input: the few-chain
        # workload it is for, and the 4096-token one (32 chains, where the plain pass already
        # keeps 128 SMs busy)
        for c, seg in ((synth.FEW_CHAINS_16K, 16), (synth.SINGLE_4K, 22)):
            ent = {}
            for label, sc in (("plain", 0), ("segmented", seg)):
                r = time_prefill(c, args.steps, args.warmup, dev, flush, trace=True, seg_chunks=sc)
                m, rl = prefill_line(c, r, args.steps, pk, dev)
                ent[label] = {"tokens_per_s": c.T / (m * 1e-3), "ms": m, "roofline_frac": rl["frac"],
                              "per_kernel": rl["per_kernel"]}
            ent["segmented"]["seg_chunks"] = seg
            ent["speedup"] = ent["plain"]["ms"] / ent["segmented"]["ms"]
            extra[f"{c.name}_segmented"] = ent
        # the token-sequential fp32 kernel (one CTA per chain) on the shapes the chunked path leaves to it
        for c in (GQA16_4K, FP32_4K, synth.TINY):
            n_steps = max(3, args.steps // 4)
            r = time_prefill(c, n_steps, args.warmup, dev, flush, trace=True)
            m, rl = prefill_line(c, r, n_steps, pk, dev)
            extra[c.name] = {"tokens_per_s": c.T / (m * 1e-3), "ms": m, "roofline_frac": rl["frac"],
                             "per_kernel": rl["per_kernel"], "h_qk": c.h_qk, "h_v": c.h_v, "d": c.d_k,
                             "dtype": c.dtype}
        r = time_backward(synth.SINGLE_4K, max(3, args.steps // 4), args.warmup, dev, flush)
        m, = max_over_ranks([statistics.mean(r["ms"])], dev)
        extra["prefill_backward_T4096"] = {"tokens_per_s": synth.SINGLE_4K.T / (m * 1e-3), "ms": m,
                                           "kernels": "token_inputs_kernel, bwd_fwd_kernel, bwd_norm_kernel, bwd_rev_kernel, bwd_prologue_kernel, bwd_gate_kernel, bwd_param_kernel",
                                           "kernels_ms_per_step": r["kernels"]}
        dc = synth.DECODE_256
        r = time_decode(dc, args.steps, args.warmup, dev, flush)
        m, = max_over_ranks([statistics.mean(r["ms"])], dev)
        extra[dc.name] = {"seqs_per_s": dc.batch / (m * 1e-3), "ms": m,
                          **roofline_of(dc.batch * DECODE_BYTES_PER_SEQ, dc.batch * DECODE_FLOPS_PER_SEQ, m, pk)}
    if rank != 0:
        return
    cpu = cpu_baseline(cfg)
    line = {
        "metric": METRIC,
        "value": world * cfg.T / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; distributions of the workload definitions)",
        "config": headline_config(cfg, world),
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": {"value": world * cfg.T / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": res["e2e"]["h2d"], "d2h_bytes_per_step": res["e2e"]["d2h"],
                "ms_per_step": e2e_ms, "pipelined": res["e2e"]["pipelined"]},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "wall_s_timed_region": wall,
        "extra": extra,
    }
    print(json.dumps(line), flush=True)


def headline_config(cfg, world):
    """The `config` of the headline line (both arms print the same one)."""
    return {"workload": cfg.name, "tokens": cfg.T, "seqs": cfg.N, "seq_len": max(cfg.lengths), "h_qk": cfg.h_qk,
            "h_v": cfg.h_v, "d_k": cfg.d_k, "d_v": cfg.d_v, "state": "fp32", "init_state": cfg.init_std > 0,
            "final_state": True,
            "l2": "flushed between steps (512 MiB write); e2e: not flushed, fresh inputs each step",
            "parallelism": f"replicas x{world}"}


# The sources of the chunked prefill's kernels (the ones the DRAM summary measures): its translation
# unit and the headers it includes.
PREFILL_TC_SOURCES = ("gateddeltanet_layer_gb300/csrc/prefill_tc.cu", "gateddeltanet_layer_gb300/csrc/tc_ptx.cuh",
                      "gateddeltanet_layer_gb300/csrc/gdn_common.cuh", "gateddeltanet_layer_gb300/csrc/gdn_internal.h",
                      "include/gdn.h", "include/gdn_trace.h")


def _source_digest():
    """sha256 over the chunked prefill's sources (PREFILL_TC_SOURCES, in that order)."""
    import hashlib
    h = hashlib.sha256()
    for f in PREFILL_TC_SOURCES:
        h.update(f.encode())
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()


def profiled_traffic(cfg):
    """DRAM bytes (read + write) of one call on workload `cfg`, whole call and
    per kernel, from the committed ncu summary ``profiles/dram_<workload>.md``,
    or None when that summary is missing or was taken on other library sources.
    The summary holds lines ``traffic_bytes_per_call: N`` and
    ``traffic_<kernel>: N`` (already scaled to the named workload)."""
    path = os.path.join(ROOT, "profiles", f"dram_{cfg.name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if line.startswith(("traffic_", "sources_sha256")) and ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    try:
        if fields["sources_sha256"] != _source_digest():
            return None
        call = int(fields.pop("traffic_bytes_per_call"))
    except (KeyError, ValueError):
        return None
    kernels = {k[len("traffic_"):]: int(v) for k, v in fields.items() if k.startswith("traffic_")}
    return {"call": call, "kernels": kernels}


# ---------------------------------------------------------------------- CPU oracle
def _oracle_sample(cfg, n_chains):
    """(sequence, head) chains of the first sequences of `cfg`, all heads of each."""
    return [(n, h) for n in range(cfg.N) for h in range(cfg.h_v)][:n_chains]


def _sample_tokens(cfg, chains):
    """Tokens of the whole layer (all heads) the chains amount to."""
    return float(sum(int(cfg.lengths[n]) for n, _ in chains)) / cfg.h_v


def cpu_baseline(cfg, n_chains=64):
    """The fp64 oracle, as it is, on the host cores: a bounded sample of the
    workload's (sequence, head) chains, as tokens/s of the whole layer."""
    from oracle import oracle as ref
    cores = os.cpu_count() or 1
    inp = inputs_of(cfg)
    chains = _oracle_sample(cfg, n_chains)
    t0 = time.perf_counter()
    ref.prefill(inp, inp["cu_seqlens"], inp["init_state"], chains=chains, threads=cores)
    dt = time.perf_counter() - t0
    return {"value": _sample_tokens(cfg, chains) / dt, "unit": "tokens/s", "cores": min(cores, len(chains)),
            "kind": "oracle",
            "sample": f"{len(chains)} of {cfg.h_v * cfg.N} (sequence, head) chains of {cfg.name} (all tokens of "
                      f"each), {dt:.2f} s wall on {min(cores, len(chains))} threads; tokens/s of the whole layer = "
                      f"the chains' tokens / {cfg.h_v} heads / wall time"}


def run_reference(args):
    """The reference arm: the fp64 CPU oracle, timed on the host cores.  Each
    step runs one chain per host core of the headline workload (a bounded
    sample of it); ms_per_step is that step's measured wall time and value the
    tokens/s of the whole layer the sample amounts to."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = HEADLINE
    from oracle import oracle as ref
    ref.build()
    cores = os.cpu_count() or 1
    inp = synth.make_prefill(cfg)
    chains = _oracle_sample(cfg, min(cores, cfg.h_v * cfg.N))
    for _ in range(args.warmup):
        ref.prefill(inp, inp["cu_seqlens"], chains=chains, threads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        ref.prefill(inp, inp["cu_seqlens"], chains=chains, threads=cores)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    value = _sample_tokens(cfg, chains) / dt
    sample = (f"{len(chains)} of {cfg.h_v * cfg.N} (sequence, head) chains of {cfg.name} per step, all tokens of "
              f"each; tokens/s of the whole layer = the chains' tokens / {cfg.h_v} heads / step time")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)", "config": headline_config(cfg, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": min(cores, len(chains)), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_case(args):
    """Only the GPU call of one workload (warm-up + steps), for profilers."""
    import torch

    import gateddeltanet_layer_gb300 as gdn
    gdn.library()
    dev = torch.device("cuda", 0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cfg = {**synth.CONFIGS, **PROFILE_CASES}[args.case]
    if isinstance(cfg, synth.DecodeConfig):
        r = time_decode(cfg, args.steps, args.warmup, dev, flush)
    elif args.backward:
        r = time_backward(cfg, args.steps, args.warmup, dev, flush)
    else:
        r = time_prefill(cfg, args.steps, args.warmup, dev, flush, seg_chunks=args.seg_chunks)
    print(json.dumps({"case": args.case, "backward": args.backward, "seg_chunks": args.seg_chunks, "ms": r["ms"]}),
          flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--case", choices=sorted({**synth.CONFIGS, **PROFILE_CASES}),
                    help="run only this workload's GPU call")
    ap.add_argument("--seg-chunks", type=int, default=0,
                    help="with --case: time the segment-parallel prefill with segments of this many chunks")
    ap.add_argument("--backward", action="store_true", help="with --case: time the backward of that prefill")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
