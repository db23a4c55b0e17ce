"""Benchmark of the absorbed causal Gated-MLA forward on GB300.

A step is one causal prefill of the K3-size layer (B=1, T=8192, H=96,
d_q=d_v=128, r=512, bf16, scale 1): the W_UK absorb, the latent scores, the
causal softmax, the latent weighting, the W_UV up-projection and the gate, all
in the library's fused kernel.  The cached-latent decode (B=64, cache lengths
uniform in [1024, 32768], H=96, r=512) is timed in the same run and reported
under "decode", and the whole layer at the prefill's size (step-1 projections
with RMSNorm, the attention, W_o: x [B,T,D] -> y) under "layer".  The
mid-size prefill (B=4, T=4096, H=16) runs under "mid_prefill".  The two
small configurations run under "small_prefill" (r=32 at T=2048, bf16, bound by
the exponential unit), "toy_layer" (the fp32 toy layer, bound by launch
latency), "toy_backward" (the gradients of the toy layer's attention, fp32) and
"small_backward" (the same at the toy long-context sizes with bf16 inputs).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on stdout (rank 0), ending with ``summary``: every section's
headline figure and roofline fraction.  ``value`` is TFLOP/s on the algorithmic
causal FLOP count B*H*[2 r T(T+1) + 2 T r (d_q+d_v)], device time of the
kernel launches, L2 flushed between steps; ``e2e`` is the same metric through
the public API with pinned host buffers, copies included.  Under torchrun each
rank runs its own replica (the path needs no exchange: weak scaling).
``--impl reference`` times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from latent_compressed_attention_gb300 import workloads as W  # noqa: E402

PREFILL = W.K3_PREFILL_BF16
DECODE = W.K3_DECODE_BF16
KERNEL_SRC = os.path.join(ROOT, "latent_compressed_attention_gb300", "csrc", "prefill_bf16_r512.cu")
DECODE_SRC = os.path.join(ROOT, "latent_compressed_attention_gb300", "csrc", "decode_bf16.cu")
_CSRC = os.path.join(ROOT, "latent_compressed_attention_gb300", "csrc")
LAYER_SRCS = [os.path.join(_CSRC, f) for f in ("gemm_bf16.cu", "layer.cu", "prefill_bf16_r512.cu")]
LAYER_DECODE_SRCS = [os.path.join(_CSRC, f) for f in ("gemm_bf16.cu", "layer_decode.cu", "decode_bf16.cu")]
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
L2_FLUSH_BYTES = 512 << 20   # > 129 MB L2


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def src_hash(paths):
    """First 16 hex digits of the SHA-256 of the files' bytes, concatenated in order."""
    h = hashlib.sha256()
    for path in ([paths] if isinstance(paths, str) else paths):
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, src):
    """DRAM bytes per launch (or per call) from a committed ncu capture, if the sources are unchanged since."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)[kernel]
        if d.get("src_sha") == src_hash(src):
            return float(d["bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples (every 50 ms) taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 6:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[2 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# ----------------------------------------------------------------------------- distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- our arm
def prefill_inputs(torch, dev, w=None):
    d = W.draw_prefill_direct(PREFILL if w is None else w, seed=0)
    to = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)  # noqa: E731
    host = {k: to(v).pin_memory() for k, v in d.items() if v is not None}
    devt = {k: v.to(dev) for k, v in host.items()}
    return host, devt


def decode_inputs(torch, dev):
    d = W.draw_decode(DECODE, seed=0)
    lens = d["lens"]
    cache = torch.empty((DECODE.B, DECODE.max_len, DECODE.r), dtype=torch.bfloat16, device=dev)
    for b in range(DECODE.B):
        rows = W.decode_cache_rows(DECODE, b, int(lens[b]), seed=0)
        cache[b, : lens[b]].copy_(torch.from_numpy(rows.astype(np.float32)).to(torch.bfloat16))
        cache[b, lens[b]:].zero_()
    to = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(dev)  # noqa: E731
    return dict(q_abs=to(d["q_abs"]), w_uv=to(d["w_uv"]), cache=cache,
                lens=torch.from_numpy(lens).to(dev), lens_np=lens)


def timed_steps(torch, fn, steps, flush, stream):
    """Per-step CUDA-event times (ms) on `stream`, L2 flushed before each step (outside the events),
    and the number of kernels the library launched over the steps (its own launch counter)."""
    import latent_compressed_attention_gb300 as lca

    times = []
    first = lca.mla_kernel_launches()
    for _ in range(steps):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        e.synchronize()
        times.append(s.elapsed_time(e))
    return times, lca.mla_kernel_launches() - first


def run_ours(args):
    import torch

    import latent_compressed_attention_gb300 as lca

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    if world == 1:
        lca.build()
    lca.library()
    pk = peaks()

    host, d = prefill_inputs(torch, dev)
    out = torch.empty((PREFILL.B, PREFILL.T, PREFILL.H * PREFILL.d_v), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ws = prefill_workspace(torch, lca, PREFILL, dev)
    step = lambda: lca.mla_absorbed_attn_fwd(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"],  # noqa: E731
                                             PREFILL.scale, out=out, workspace=ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if lca.mla_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        times, launches = timed_steps(torch, step, args.steps, flush, stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = max_over_ranks(sum(times), world)
    flops = PREFILL.prefill_flops()
    ms_per_step = total_ms / args.steps
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12
    kernel_ms = statistics.mean(times)
    achieved = flops / (kernel_ms * 1e-3) / 1e12

    # end to end through the public API: every step copies its inputs in from pinned host memory and its
    # result out to pinned host memory; as in a serving loop, step i's copies run on their own streams and
    # overlap the neighbouring steps' kernels (two device buffer sets, ordered by events)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out.numel() * out.element_size()
    e2e_value = e2e_ms = None
    if not args.no_e2e:
        e2e_ms = max_over_ranks(e2e_pipelined(torch, lca, dev, stream, host, out, ws, max(4, args.steps // 2)),
                                world)
        e2e_value = world * flops / (e2e_ms * 1e-3) / 1e12

    mid = run_mid_prefill(torch, lca, dev, stream, flush, args, pk) \
        if not args.no_mid and PREFILL.name != W.MID_PREFILL_BF16.name else None
    decode = run_decode(torch, lca, dev, stream, flush, args, pk) if not args.no_decode else None
    layer_line = run_layer(torch, lca, dev, stream, flush, args, pk) if not args.no_layer else None
    layer_dec = run_layer_decode(torch, lca, dev, stream, flush, args, pk) \
        if not (args.no_layer or args.no_decode) else None
    small = run_small_prefill(torch, lca, dev, stream, flush, args) if not args.no_small else None
    toy = run_toy_layer(torch, lca, dev, stream, flush, args) if not args.no_small else None
    toy_bwd = run_toy_backward(torch, lca, dev, stream, flush, args) if not args.no_small else None
    small_bwd = run_toy_backward(torch, lca, dev, stream, flush, args, W.TOY_LONG_BF16) if not args.no_small else None
    mid_bwd = run_backward_r512(torch, lca, dev, stream, flush, args, pk) if not args.no_bwd else None
    if lca.mla_get_device_error() != 0:
        raise RuntimeError("device error word set after the timed region")

    if rank == 0:
        line = {
            "metric": "MLA fwd TFLOP/s (causal) and decode GB/s, % of GB300 roofline, vs CPU oracle",
            "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": PREFILL.name, "B": PREFILL.B, "T": PREFILL.T, "H": PREFILL.H,
                       "d_q": PREFILL.d_q, "d_v": PREFILL.d_v, "r": PREFILL.r, "scale": PREFILL.scale,
                       "causal": True, "gate": True, "flops_per_step": flops,
                       "l2": "flushed between steps (512 MB write outside the timed events)",
                       "parallelism": f"replicas x{world}"},
            "e2e": None if e2e_value is None else {
                "value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "schedule": "every step: pinned H2D of its inputs, the prefill call, D2H of its output; copies "
                            "on separate streams overlap the neighbouring steps' kernels (double-buffered)"},
            "roofline": {"kernel": "prefill_r512_kernel", "bound": "tensor", "achieved": round(achieved, 2),
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 4),
                         "peak_source": pk["source"] + " (burst bf16)",
                         "traffic": committed_traffic("prefill_r512_kernel", KERNEL_SRC)},
            "gpu_launches": launches,
            "clocks": clk.summary(),
        }
        sections = [("mid_prefill", mid), ("decode", decode), ("layer", layer_line), ("layer_decode", layer_dec),
                    ("small_prefill", small), ("toy_layer", toy), ("toy_backward", toy_bwd),
                    ("small_backward", small_bwd), ("mid_backward", mid_bwd)]
        for name, sec in sections:
            if sec is not None:
                line[name] = sec
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        line["summary"] = summary(line, sections)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def summary(line, sections):
    """Every section's headline figure and roofline fraction in a few hundred bytes, last on the line."""
    def brief(sec):
        if "unavailable" in sec:
            return {"unavailable": sec["unavailable"]}
        rf = sec.get("roofline", {})
        return {"value": sec["value"], "unit": sec["unit"], "frac": rf.get("frac"), "bound": rf.get("bound")}
    out = {line["config"]["workload"]: {"value": line["value"], "unit": line["unit"],
                                        "frac": line["roofline"]["frac"], "bound": "tensor"}}
    if line.get("e2e"):
        out["e2e_ms_per_step"] = line["e2e"]["ms_per_step"]
    for name, sec in sections:
        if sec is not None:
            out[name] = brief(sec)
            if name == "decode" and sec.get("fp8"):
                out["decode_fp8"] = brief(sec["fp8"])
                out["decode_rows_per_s"] = {"bf16": sec.get("rows_per_s"), "fp8": sec["fp8"].get("rows_per_s")}
    if "cpu_baseline" in line:
        out["cpu_oracle_tflops"] = line["cpu_baseline"]["value"]
    return out


def prefill_workspace(torch, lca, w, dev):
    """The prefill's device workspace for workload w, allocated once outside every timed region (None if none)."""
    need = lca.mla_absorbed_attn_fwd_workspace_size(w.B, w.T, w.H, w.d_q, w.d_v, w.r, torch.bfloat16)
    return torch.empty(need, dtype=torch.uint8, device=dev) if need > 0 else None


def e2e_pipelined(torch, lca, dev, stream, host, out, ws, steps):
    """Per-step milliseconds of `steps` end-to-end prefill steps: step i copies its inputs host -> device on a
    copy stream, runs the prefill on `stream`, copies its output device -> host on a third stream; two device
    buffer sets let step i+1's input copy and step i-1's output copy overlap step i's kernel.  Timed with CUDA
    events from the first input copy to the last output copy (warm-up steps outside)."""
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bufs = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    wss = [ws, None if ws is None else torch.empty_like(ws)]
    outs_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    in_ready, comp_done, out_read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    used = [False, False]

    def step(i):
        j = i % 2
        with torch.cuda.stream(h2d_s):
            if used[j]:
                h2d_s.wait_event(comp_done[j])   # buffer set j's previous kernel has read its inputs
            for k, v in host.items():
                bufs[j][k].copy_(v, non_blocking=True)
            in_ready[j].record(h2d_s)
        stream.wait_event(in_ready[j])
        if used[j]:
            stream.wait_event(out_read[j])       # the previous output of set j has been copied out
        b = bufs[j]
        lca.mla_absorbed_attn_fwd(b["q"], b["c"], b["w_uk"], b["w_uv"], b["gate"], PREFILL.scale, out=outs[j],
                                  workspace=wss[j], stream=stream)
        comp_done[j].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(comp_done[j])
            outs_host[j].copy_(outs[j], non_blocking=True)
            out_read[j].record(d2h_s)
        used[j] = True

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(h2d_s)
    for i in range(steps):
        step(i)
    t1.record(d2h_s)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


def run_mid_prefill(torch, lca, dev, stream, flush, args, pk):
    """The mid-size prefill (B=4, T=4096, H=16, d_q=d_v=128, r=512, bf16, scale 1/sqrt(128)): the same fused
    kernel as the step, with 16 heads instead of 96 sharing each latent tile and 4x shorter key rows."""
    w = W.MID_PREFILL_BF16
    _, d = prefill_inputs(torch, dev, w)
    out = torch.empty((w.B, w.T, w.H * w.d_v), dtype=torch.bfloat16, device=dev)
    ws = prefill_workspace(torch, lca, w, dev)
    step = lambda: lca.mla_absorbed_attn_fwd(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], w.scale,  # noqa: E731
                                             out=out, workspace=ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    times, launches = timed_steps(torch, step, args.steps, flush, stream)
    ms = statistics.mean(times)
    tf = w.prefill_flops() / (ms * 1e-3) / 1e12
    return {"workload": w.name, "value": round(tf, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "flops_per_step": w.prefill_flops(),
            "config": {"B": w.B, "T": w.T, "H": w.H, "d_q": w.d_q, "d_v": w.d_v, "r": w.r, "scale": w.scale,
                       "l2": "flushed between steps"},
            "roofline": {"kernel": "prefill_r512_kernel", "bound": "tensor", "achieved": round(tf, 2),
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(tf / pk["bf16_tflops"], 4),
                         "peak_source": pk["source"] + " (burst bf16)", "traffic": None},
            "gpu_launches": launches}


def run_decode(torch, lca, dev, stream, flush, args, pk):
    try:
        ws_bytes = lca.mla_latent_decode_workspace_size(DECODE.B, DECODE.H, DECODE.r, DECODE.max_len)
        if ws_bytes == 0:
            return {"unavailable": "decode kernel not built for this shape"}
    except Exception as e:  # noqa: BLE001
        return {"unavailable": str(e)}
    d = decode_inputs(torch, dev)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty((DECODE.B, DECODE.H * DECODE.d_v), dtype=torch.bfloat16, device=dev)
    step = lambda: lca.mla_latent_decode(d["q_abs"], d["cache"], d["lens"], d["w_uv"], None,  # noqa: E731
                                         DECODE.scale, out=out, workspace=ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    times, launches = timed_steps(torch, step, args.steps, flush, stream)
    ms = statistics.mean(times)
    cache_bytes = int(d["lens_np"].astype(np.int64).sum()) * DECODE.r * 2
    gbs = cache_bytes / (ms * 1e-3) / 1e9
    fp8 = run_decode_fp8(torch, lca, dev, stream, flush, args, pk, d) if not args.no_fp8 else None
    return {"workload": DECODE.name, "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "rows_per_s": round(int(d["lens_np"].sum()) / (ms * 1e-3), 1),
            "cache_bytes_per_step": cache_bytes, "sum_lens": int(d["lens_np"].sum()), "fp8": fp8,
            "roofline": {"kernel": "decode (pair + merge)", "bound": "hbm", "achieved": round(gbs, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                         "peak_source": pk["source"],
                         "traffic": committed_traffic("decode", DECODE_SRC)},
            "gpu_launches": launches}


FP8_CACHE_SCALE = 0.0625   # RMSNorm rows (|c| <= sqrt(512)) map inside e4m3's +-448


def run_decode_fp8(torch, lca, dev, stream, flush, args, pk, d):
    """The decode workload over the same cache stored as e4m3 (quantised once, outside the timed region):
    half the bytes per cached token."""
    c8 = lca.mla_quantize_latent_fp8(d["cache"], FP8_CACHE_SCALE)
    ws = torch.empty(lca.library().mla_latent_decode_fp8_workspace_size(DECODE.B, DECODE.H, DECODE.r,
                                                                        DECODE.max_len), dtype=torch.uint8, device=dev)
    out = torch.empty((DECODE.B, DECODE.H * DECODE.d_v), dtype=torch.bfloat16, device=dev)
    step = lambda: lca.mla_latent_decode_fp8(d["q_abs"], c8, d["lens"], d["w_uv"], FP8_CACHE_SCALE, None,  # noqa: E731
                                             DECODE.scale, out=out, workspace=ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    times, launches = timed_steps(torch, step, args.steps, flush, stream)
    del c8
    ms = statistics.mean(times)
    sum_lens = int(d["lens_np"].astype(np.int64).sum())
    cache_bytes = sum_lens * DECODE.r
    gbs = cache_bytes / (ms * 1e-3) / 1e9
    return {"workload": DECODE.name.replace("bf16", "fp8"), "value": round(gbs, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "rows_per_s": round(sum_lens / (ms * 1e-3), 1),
            "cache_bytes_per_step": cache_bytes, "cache_scale": FP8_CACHE_SCALE,
            "roofline": {"kernel": "decode over the e4m3 cache (query split, pair + merge)", "bound": "hbm",
                         "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / pk["hbm_gbs"], 4), "peak_source": pk["source"], "traffic": None},
            "gpu_launches": launches}


def layer_flops(w) -> dict:
    """Algorithmic FLOPs of the whole layer: the five projections plus the absorbed attention."""
    M = w.B * w.T
    gemm = 2 * M * (w.D * w.r_q + w.r_q * w.H * w.d_q + w.D * w.r + w.D * w.H * w.d_v + w.H * w.d_v * w.D)
    attn = w.B * w.H * (2 * w.r * w.T * (w.T + 1) + 2 * w.T * w.r * (w.d_q + w.d_v))
    return {"gemm": gemm, "attention": attn, "total": gemm + attn}


def run_layer(torch, lca, dev, stream, flush, args, pk):
    """The whole layer (x -> y through step 1, the attention and W_o) at the prefill workload's size."""
    w = PREFILL
    p = W.draw_layer(w, seed=0)
    to = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(dev)  # noqa: E731
    t = {k: to(v) for k, v in p.items()}
    del p
    ws_bytes = lca.mla_gated_layer_workspace_size(w.B, w.T, w.D, w.H, w.d_q, w.d_v, w.r, w.r_q, torch.bfloat16)
    if ws_bytes == 0:
        return {"unavailable": "layer shape not supported"}
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    y = torch.empty((w.B, w.T, w.D), dtype=torch.bfloat16, device=dev)
    step = lambda: lca.mla_gated_layer_fwd(t["x"], t["q_down"], t["q_up"], t["kv_down"], t["kv_up"],  # noqa: E731
                                           t["gate"], t["o_proj"], w.H, w.d_q, w.d_v, w.scale, out=y, workspace=ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    times, launches = timed_steps(torch, step, args.steps, flush, stream)
    ms = statistics.mean(times)
    fl = layer_flops(w)
    tf = fl["total"] / (ms * 1e-3) / 1e12
    return {"workload": w.name.replace("prefill", "layer"), "value": round(tf, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "flops_per_step": fl["total"], "gemm_flops": fl["gemm"],
            "attention_flops": fl["attention"],
            "config": {"B": w.B, "T": w.T, "D": w.D, "H": w.H, "d_q": w.d_q, "d_v": w.d_v, "r": w.r, "r_q": w.r_q,
                       "inputs": "x ~ N(0,1), weights ~ N(0, 0.02^2), bf16"},
            "roofline": {"kernel": "layer (5 tensor-core GEMMs, the latent's row pass, prefill_r512_kernel)",
                         "bound": "tensor", "achieved": round(tf, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tf / pk["bf16_tflops"], 4), "peak_source": pk["source"] + " (burst bf16)",
                         "traffic": committed_traffic("layer", LAYER_SRCS)},
            "gpu_launches": launches}


def run_layer_decode(torch, lca, dev, stream, flush, args, pk):
    """One decode step of the whole layer (step 1, latent append, cached-latent attention, W_o) for the
    decode workload's sequences, with the prefill workload's layer sizes."""
    w = PREFILL
    dw = DECODE
    p = W.draw_layer(dataclasses.replace(w, B=dw.B, T=1), seed=1)
    to = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).to(dev)  # noqa: E731
    t = {k: to(v) for k, v in p.items()}
    del p
    x = t["x"].reshape(dw.B, w.D)
    d = decode_inputs(torch, dev)
    lens = d["lens"].clone()
    ok = lens < dw.max_len            # a sequence at the cache's end keeps its length (no free row)
    lens = torch.where(ok, lens, lens - 1).to(torch.int32)
    y = torch.empty((dw.B, w.D), dtype=torch.bfloat16, device=dev)
    need = lca.library().mla_gated_layer_decode_workspace_size(dw.B, w.D, w.H, w.d_q, w.d_v, w.r, w.r_q,
                                                               dw.max_len, lca.DTYPE_BF16)
    if need == 0:
        return {"unavailable": "layer decode shape not supported"}
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    step = lambda: lca.mla_gated_layer_decode(x, t["q_down"], t["q_up"], t["kv_down"], t["kv_up"],  # noqa: E731
                                              t["gate"], t["o_proj"], d["cache"], lens, w.H, w.d_q, w.d_v,
                                              dw.scale, out=y, workspace=ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    times, launches = timed_steps(torch, step, args.steps, flush, stream)
    ms = statistics.mean(times)
    cache_bytes = int((lens.to(torch.int64) + 1).sum().item()) * w.r * 2
    weight_bytes = sum(int(v.numel()) * 2 for k, v in t.items() if k != "x")
    gbs = (cache_bytes + weight_bytes) / (ms * 1e-3) / 1e9
    return {"workload": "k3_layer_decode_bf16", "value": round(dw.B / (ms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(ms, 4), "tokens_per_step": dw.B, "cache_bytes_per_step": cache_bytes,
            "weight_bytes_per_step": weight_bytes,
            "roofline": {"kernel": "layer decode step (5 GEMMs with M = B and their row passes, append, absorb, "
                                   "pair + merge)",
                         "bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / pk["hbm_gbs"], 4), "peak_source": pk["source"],
                         "traffic": committed_traffic("layer_decode", LAYER_DECODE_SRCS)},
            "gpu_launches": launches}


# Exponentials per clock per SM on the multi-function unit: measured on GB300 by a throughput probe (152 SMs x
# 2048 threads, eight independent ex2.approx.ftz.f32 chains per thread, CUDA events): 9.47e12 ex2/s, 30.1 per
# clock per SM at 2070 MHz (the f16x2 and bf16x2 forms give the same 32 exponentials per clock).  fp32 FMA
# lanes per SM (the same probe measured 121.7 FMA per clock per SM).
MUFU_EX2_PER_CLK_SM = 30.1
FP32_LANES_SM = 128
SM_MAX_MHZ = 2070.0


def run_small_prefill(torch, lca, dev, stream, flush, args):
    """The small-rank prefill (r = 32, d = 16, T = 2048, bf16): one exponential per causal score and only
    4 r = 128 tensor-core FLOPs per exponential, so the exponential unit bounds it."""
    w = W.TOY_LONG_BF16
    d = W.draw_prefill_direct(w, seed=0)
    t = {k: torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).to(dev) for k, v in d.items() if v is not None}
    out = torch.empty((w.B, w.T, w.H * w.d_v), dtype=torch.bfloat16, device=dev)
    ws = prefill_workspace(torch, lca, w, dev)
    step = lambda: lca.mla_absorbed_attn_fwd(t["q"], t["c"], t["w_uk"], t["w_uv"], t["gate"], w.scale,  # noqa: E731
                                             out=out, workspace=ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    times, launches = timed_steps(torch, step, args.steps, flush, stream)
    ms = statistics.mean(times)
    exps = w.B * w.H * w.T * (w.T + 1) // 2
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = MUFU_EX2_PER_CLK_SM * sms * SM_MAX_MHZ * 1e6 / 1e9   # G ex2/s
    achieved = exps / (ms * 1e-3) / 1e9
    return {"workload": w.name, "value": round(w.prefill_flops() / (ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 5), "flops_per_step": w.prefill_flops(), "exp_per_step": exps,
            "config": {"B": w.B, "T": w.T, "H": w.H, "d_q": w.d_q, "d_v": w.d_v, "r": w.r, "scale": w.scale,
                       "l2": "flushed between steps"},
            "roofline": {"kernel": "prefill_small_kernel", "bound": "alu", "achieved": round(achieved, 1),
                         "peak": round(peak, 1), "unit": "G ex2/s", "frac": round(achieved / peak, 4),
                         "peak_source": f"measured ex2 throughput: {MUFU_EX2_PER_CLK_SM} ex2/clk/SM x {sms} SMs x "
                                        f"{SM_MAX_MHZ:.0f} MHz",
                         "traffic": None},
            "gpu_launches": launches}


def run_toy_layer(torch, lca, dev, stream, flush, args):
    """The fp32 toy layer (B=2, T=128, D=256, H=8, d=16, r=32, r_q=64) through step 1, the attention and W_o:
    2.1e7 attention FLOPs, so launch latency bounds it."""
    w = W.TOY_LAYER_F32
    p = W.draw_layer(w, seed=0)
    t = {k: torch.from_numpy(v.astype(np.float32)).to(dev) for k, v in p.items()}
    ws = torch.empty(lca.mla_gated_layer_workspace_size(w.B, w.T, w.D, w.H, w.d_q, w.d_v, w.r, w.r_q, torch.float32),
                     dtype=torch.uint8, device=dev)
    y = torch.empty((w.B, w.T, w.D), dtype=torch.float32, device=dev)
    step = lambda: lca.mla_gated_layer_fwd(t["x"], t["q_down"], t["q_up"], t["kv_down"], t["kv_up"],  # noqa: E731
                                           t["gate"], t["o_proj"], w.H, w.d_q, w.d_v, w.scale, out=y, workspace=ws)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    times, launches = timed_steps(torch, step, args.steps, flush, stream)
    ms = statistics.mean(times)
    fl = layer_flops(w)["total"]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = 2 * FP32_LANES_SM * sms * SM_MAX_MHZ * 1e6 / 1e12
    tf = fl / (ms * 1e-3) / 1e12
    return {"workload": w.name, "value": round(ms * 1e3, 2), "unit": "us/call", "higher_is_better": False,
            "ms_per_step": round(ms, 5), "flops_per_step": fl, "kernels_per_call": launches // max(args.steps, 1),
            "config": {"B": w.B, "T": w.T, "D": w.D, "H": w.H, "d_q": w.d_q, "d_v": w.d_v, "r": w.r, "r_q": w.r_q,
                       "dtype": "f32 (fp32 FMAs, no TF32)", "l2": "flushed between steps"},
            "roofline": {"kernel": "toy layer (fp32 SIMT kernels)", "bound": "alu", "achieved": round(tf, 4),
                         "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(tf / peak, 5),
                         "peak_source": f"derived: fp32 FMA {FP32_LANES_SM} lanes/SM x 2 x {sms} SMs x "
                                        f"{SM_MAX_MHZ:.0f} MHz; the call is launch-latency bound",
                         "traffic": None},
            "gpu_launches": launches}


def backward_flops(w) -> float:
    """Algorithmic FLOPs of the attention's backward: per causal pair and head the scores, the latent
    weighting, do_lat . c, dq_abs, and the two parts of dc (2r each); per token and head the absorb, W_UV,
    do_lat, dW_UV, dq and dW_UK products."""
    pairs = w.T * (w.T + 1) / 2
    return w.B * w.H * (12.0 * w.r * pairs + 6.0 * w.T * w.r * (w.d_q + w.d_v))


def run_toy_backward(torch, lca, dev, stream, flush, args, w=None):
    """Gradients of the attention for a random dout: at the toy layer's sizes (fp32, B=2, T=128, H=8, d=16,
    r=32) or, given the toy long-context workload, at its sizes with bf16 inputs (B=4, T=2048); q, c, W_UK,
    W_UV and the gate logits are the workload's seeded direct draws.  Gradients are fp32 either way."""
    w = W.TOY_LAYER_F32 if w is None else w
    d = W.draw_prefill_direct(w, seed=0)
    dout = W.round_to(np.random.default_rng(1).standard_normal((w.B, w.T, w.H * w.d_v)), w.dtype)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    t = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(dt).to(dev)  # noqa: E731
    q, c, g, w_uk, w_uv, dout = (t(a) for a in (d["q"], d["c"], d["gate"], d["w_uk"], d["w_uv"], dout))
    code = lca.DTYPE_BF16 if w.dtype == "bf16" else lca.DTYPE_F32
    ws = torch.empty(lca.library().mla_absorbed_attn_bwd_workspace_size(w.B, w.T, w.H, w.d_q, w.d_v, w.r, code),
                     dtype=torch.uint8, device=dev)
    step = lambda: lca.mla_absorbed_attn_bwd(q, c, w_uk, w_uv, g, w.scale, dout, workspace=ws)  # noqa: E731
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    times, launches = timed_steps(torch, step, args.steps, flush, stream)
    ms = statistics.mean(times)
    fl = backward_flops(w)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = 2 * FP32_LANES_SM * sms * SM_MAX_MHZ * 1e6 / 1e12
    tf = fl / (ms * 1e-3) / 1e12
    return {"workload": w.name.replace("toy_layer_f32", "toy_backward_f32").replace("toy_long_bf16",
                                                                                      "toy_long_backward_bf16"),
            "value": round(ms * 1e3, 2), "unit": "us/call", "higher_is_better": False,
            "ms_per_step": round(ms, 5), "flops_per_step": fl, "kernels_per_call": launches // max(args.steps, 1),
            "config": {"B": w.B, "T": w.T, "H": w.H, "d_q": w.d_q, "d_v": w.d_v, "r": w.r,
                       "inputs": "direct draws of the workload, dout ~ N(0,1)",
                       "dtype": f"{w.dtype} inputs, f32 arithmetic and gradients",
                       "l2": "flushed between steps"},
            "roofline": {"kernel": "bwd_query_kernel + bwd_key_kernel (fp32 SIMT)", "bound": "alu",
                         "achieved": round(tf, 4), "peak": round(peak, 1), "unit": "TFLOP/s",
                         "frac": round(tf / peak, 5),
                         "peak_source": f"derived: fp32 FMA {FP32_LANES_SM} lanes/SM x 2 x {sms} SMs x "
                                        f"{SM_MAX_MHZ:.0f} MHz" + ("; the call is latency bound at this size" if w.T <= 256 else ""),
                         "traffic": None},
            "gpu_launches": launches}


def run_backward_r512(torch, lca, dev, stream, flush, args, pk):
    """Gradients of the attention at the mid-size prefill's shape (B=4, T=4096, H=16, r=512, d=128, bf16 inputs,
    fp32 gradients) on the tensor cores: the chain rule's products as batched GEMMs over per-head attention
    matrices.  The timed call is the backward of a training step: it is given the forward's output and each row's
    log-sum-exp (mla_absorbed_attn_fwd(..., return_lse=True), run once before the timed region), so the forward is
    not run again; `with_forward_recompute` times the call that recomputes them itself."""
    w = W.MID_PREFILL_BF16
    if args.bwd_T != w.T:   # a shorter sequence, for profiling only
        w = dataclasses.replace(w, T=args.bwd_T, name=f"{w.name}_t{args.bwd_T}")
    d = W.draw_prefill_direct(w, seed=0)
    dout = W.round_bf16(np.random.default_rng(1).standard_normal((w.B, w.T, w.H * w.d_v)))
    t = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).to(dev)  # noqa: E731
    q, c, g, w_uk, w_uv, dout = (t(a) for a in (d["q"], d["c"], d["gate"], d["w_uk"], d["w_uv"], dout))
    ws = torch.empty(lca.library().mla_absorbed_attn_bwd_workspace_size(w.B, w.T, w.H, w.d_q, w.d_v, w.r,
                                                                        lca.DTYPE_BF16), dtype=torch.uint8, device=dev)
    out_fwd, lse = lca.mla_absorbed_attn_fwd(q, c, w_uk, w_uv, g, w.scale, return_lse=True)
    saved = lambda: lca.mla_absorbed_attn_bwd(q, c, w_uk, w_uv, g, w.scale, dout, workspace=ws,  # noqa: E731
                                              out=out_fwd, lse=lse)
    recompute = lambda: lca.mla_absorbed_attn_bwd(q, c, w_uk, w_uv, g, w.scale, dout, workspace=ws)  # noqa: E731
    res = {}
    for name, step in (("recompute", recompute), ("saved", saved)):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        res[name] = timed_steps(torch, step, args.steps, flush, stream)
    del ws
    times, launches = res["saved"]
    ms = statistics.mean(times)
    ms_re = statistics.mean(res["recompute"][0])
    fl = backward_flops(w)
    tf = fl / (ms * 1e-3) / 1e12
    return {"workload": w.name.replace("prefill", "backward"), "value": round(tf, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "flops_per_step": fl, "kernels_per_call": launches // max(args.steps, 1),
            "with_forward_recompute": {"ms_per_step": round(ms_re, 4), "value": round(fl / (ms_re * 1e-3) / 1e12, 2),
                                       "unit": "TFLOP/s"},
            "config": {"B": w.B, "T": w.T, "H": w.H, "d_q": w.d_q, "d_v": w.d_v, "r": w.r, "scale": w.scale,
                       "inputs": "direct draws of the mid-size workload, dout ~ N(0,1), bf16; the forward's output "
                                 "and log-sum-exp from one forward call before the timed region",
                       "dtype": "bf16 operands, fp32 accumulation and gradients", "l2": "flushed between steps"},
            "roofline": {"kernel": "backward given the forward's output and lse (gate, 10 batched tcgen05 GEMMs)",
                         "bound": "tensor", "achieved": round(tf, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tf / pk["bf16_tflops"], 4), "peak_source": pk["source"] + " (burst bf16)",
                         "traffic": None},
            "gpu_launches": launches}


# ----------------------------------------------------------------------------- CPU oracle (baseline / reference arm)
def oracle_inputs():
    return W.draw_prefill_direct(PREFILL, seed=0)


def oracle_sample(d, seconds: float, seed: int = 0):
    """Time the fp64 oracle on sampled query rows (all heads) of the K3 prefill.

    Returns (tflops, rows, elapsed, threads).  Rows are drawn uniformly over
    the sequence; work per row is counted with the same algorithmic formula.
    """
    import oracle

    w = PREFILL
    rng = np.random.default_rng(seed)
    per_row = lambda t: w.H * (4.0 * w.r * (t + 1) + 2.0 * w.r * (w.d_q + w.d_v))  # noqa: E731
    # calibrate on two rows, then size the sample to about `seconds`
    rows = rng.integers(0, w.T, 2)
    t0 = time.perf_counter()
    oracle.prefill(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], w.scale, rows=rows)
    dt = max(time.perf_counter() - t0, 1e-3)
    rate = sum(per_row(int(t)) for t in rows) / dt
    n = int(max(2, min(4096, seconds * rate / per_row(w.T // 2))))
    rows = rng.integers(0, w.T, n)
    t0 = time.perf_counter()
    oracle.prefill(d["q"], d["c"], d["w_uk"], d["w_uv"], d["gate"], w.scale, rows=rows)
    elapsed = time.perf_counter() - t0
    flops = sum(per_row(int(t)) for t in rows)
    return flops / elapsed / 1e12, n, elapsed, oracle.num_threads()


def cpu_baseline(seconds: float):
    tflops, n, elapsed, threads = oracle_sample(oracle_inputs(), seconds)
    return {"value": round(tflops, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} query rows x {PREFILL.H} heads of {PREFILL.name}, uniform over t, {elapsed:.1f} s"}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    d = oracle_inputs()
    per_step = []
    rows_total, threads = 0, 1
    seconds = min(args.ref_seconds, 150.0 / (args.warmup + args.steps))
    for i in range(args.warmup + args.steps):
        tflops, n, elapsed, threads = oracle_sample(d, seconds, seed=100 + i)
        if i >= args.warmup:
            per_step.append((tflops, n, elapsed))
            rows_total += n
    value = statistics.mean(t for t, _, _ in per_step)
    ms = statistics.mean(e for _, _, e in per_step) * 1e3
    line = {
        "impl": "reference", "metric": "MLA fwd TFLOP/s (causal) and decode GB/s, % of GB300 roofline, vs CPU oracle",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 1), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": PREFILL.name, "B": PREFILL.B, "T": PREFILL.T, "H": PREFILL.H, "d_q": PREFILL.d_q,
                   "d_v": PREFILL.d_v, "r": PREFILL.r, "scale": PREFILL.scale, "causal": True, "gate": True},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows_total} query rows x {PREFILL.H} heads over {args.steps} steps "
                                   f"(about {seconds:.1f} s each)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-layer", action="store_true")
    ap.add_argument("--no-mid", action="store_true", help="skip the mid-size prefill section")
    ap.add_argument("--no-fp8", action="store_true", help="skip the e4m3-cache decode")
    ap.add_argument("--no-bwd", action="store_true", help="skip the r = 512 backward")
    ap.add_argument("--bwd-T", type=int, default=W.MID_PREFILL_BF16.T,
                    help="sequence length of the r = 512 backward (4096 is the benchmark; shorter is for profiling)")
    ap.add_argument("--no-small", action="store_true", help="skip the small-rank prefill and the fp32 toy layer")
    ap.add_argument("--workload", choices=["k3_prefill_bf16", "mid_prefill_bf16"], default="k3_prefill_bf16",
                    help="prefill workload of a step (the K3 size is the benchmark; the mid size is for profiling)")
    ap.add_argument("--decode-batch", type=int, default=W.K3_DECODE_BF16.B,
                    help="sequences of the decode workload (64 is the benchmark; fewer is for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    global PREFILL, DECODE
    PREFILL = W.WORKLOADS[args.workload]
    if args.decode_batch != DECODE.B:
        DECODE = dataclasses.replace(DECODE, B=args.decode_batch, name=f"{DECODE.name}_b{args.decode_batch}")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
