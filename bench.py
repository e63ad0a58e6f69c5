#!/usr/bin/env python3
"""Benchmark of the fused MLA attention prolog on GB300.

One step = one pass of the whole prolog (compression projection, split,
RMSNorm, RoPE, expansion projection, split/assemble, and the q path + INT8
quant when the workload has one) over one batch of T tokens.

Default workload: the DeepSeek-V3-shaped full prolog long prefill
(T=16384, q path + per-token INT8 quant), the largest of the five
configurations; the others are selected with
--workload {tiny,v2lite_decode,v2lite_prefill,v3_decode,v3_prefill}.

Timing: K steps are captured into one CUDA graph, each step on its own
buffer set (inputs, weights and outputs), with enough sets that the sets
together exceed 3x the L2 size; the graph is replayed between CUDA events on
the launching stream after W warm-up replays.  Per-kernel durations come from
a second graph of the same K steps with the library's timing hook on.
`e2e` is the same metric through the public call with host buffers: each
step copies x and positions from pinned host memory, runs, and copies every
output back, all inside the timed region.  When a step copies at least
8 MB the loop is pipelined as a serving loop would run it: copies in on one
stream, the call on another, copies out on a third, over two device buffer
sets, so step k+1's input copy and step k-1's output copy overlap step k's
kernels; below that the cross-stream events cost more than they hide and
the steps run in order on one stream.
Under torchrun each rank runs its own replica of the workload (no collective
on the data path); value = tokens of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mla_attention_prolog_gb300 import workloads as wl  # noqa: E402

METRIC = "MLA prolog tokens/s on 1 GB300; % HBM roofline (decode) / % BF16 TC peak (prefill)"
L2_BYTES = 126 * 1024 * 1024
DEFAULT_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(DEFAULT_PEAKS), "fallback"


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int) -> float:
    """Max of a per-rank number over all ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(tokens_per_rank: int, ms_max: float, world: int) -> float:
    """Whole-job throughput: the tokens every rank processed over the slowest
    rank's time (each rank runs its own replica; weak scaling)."""
    return tokens_per_rank * world / (ms_max / 1e3)


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    @staticmethod
    def now():
        import datetime
        return datetime.datetime.now()

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen; samples inside
        [t0, t1] (the timed region) when there are at least 3 of them, else
        every sample of the run."""
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((ts, float(parts[1]), float(parts[2]),
                             [n for n, v in zip(names, parts[4:8]) if v.lower() == "active"]))
            except ValueError:
                continue
        window = "timed region"
        sel = [r for r in rows if t0 is not None and t0 <= r[0] <= t1]
        if len(sel) < 3:
            sel, window = rows, "whole run"
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        reasons = sorted({n for r in sel for n in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel), "window": window}


# ------------------------------------------------------ per-kernel accounting

def kernel_work(d: wl.Dims, cache: bool = False, names=()):
    """Algorithmic bytes and flops attributed to each kernel of one run.

    Bytes: every input a kernel must read once plus every output it must write
    once (workspace traffic excluded); they add up to the whole op's count.
    The per-head quant writes its codes and scales from the expansion kernel;
    the latent cache rows are written by the norm kernel.
    Flops: 2 * T * N * K of the projection the kernel computes.
    """
    T, H, Dn, Dv, R = d.T, d.num_heads, d.nope_dim, d.v_dim, d.rope_dim
    q_out = (T * d.n_q + 4 * T * d.n_scales) if d.quant_q else 0
    w8 = d.w8a8  # INT8 weights (1 byte) and their row scales; x is read by the x-quant kernel
    nq_rows = d.n_q if d.q_lora_rank else 0
    b = {
        "mla_quant_x_kernel": 2 * T * d.D if w8 else 0,
        "mla_compress_kernel": (d.n_a * d.D + 4 * d.n_a) if w8 else 2 * T * d.D + 2 * d.n_a * d.D,
        "mla_norm_rope_kernel": 2 * (d.q_lora_rank + d.kv_lora_rank) + 4 * T + 4 * T * R
                                + 2 * T * R + 2 * T * H * R
                                + ((4 * T + 2 * T * (d.kv_lora_rank + R)) if cache else 0),
        "mla_expand_kernel": (d.w_b_elems + 4 * (nq_rows + d.n_kv) if w8 else 2 * d.w_b_elems)
                             + 2 * T * H * Dn + 2 * T * H * Dv + (q_out if d.quant_per_head else 0),
        "mla_quant_kernel": 0 if d.quant_per_head else q_out,
    }
    f = {
        "mla_quant_x_kernel": 0,
        "mla_compress_kernel": 2 * T * d.n_a * d.D,
        "mla_norm_rope_kernel": 0,
        "mla_expand_kernel": 2 * T * (d.n_q * d.q_lora_rank + d.n_kv * d.kv_lora_rank),
        "mla_quant_kernel": 0,
    }
    assert sum(b.values()) == wl.algorithmic_bytes(d, cache)
    # the kernels on CTA pairs do the work of their one-CTA counterparts
    b["mla_compress_pair_kernel"] = b["mla_compress_kernel"]
    f["mla_compress_pair_kernel"] = f["mla_compress_kernel"]
    b["mla_expand_pair_kernel"] = b["mla_expand_kernel"]
    f["mla_expand_pair_kernel"] = f["mla_expand_kernel"]
    if "mla_expand_kv_pair_kernel" in names:
        # the kv tiles on their own pair kernel; the pair expansion keeps the q tiles
        b_kv = 2 * d.n_kv * d.kv_lora_rank + 2 * T * H * Dn + 2 * T * H * Dv
        b["mla_expand_kv_pair_kernel"] = b_kv
        f["mla_expand_kv_pair_kernel"] = 2 * T * d.n_kv * d.kv_lora_rank
        b["mla_expand_pair_kernel"] = b["mla_expand_kernel"] - b_kv
        f["mla_expand_pair_kernel"] = 2 * T * d.n_q * d.q_lora_rank
    # the cluster kernel runs the compression and the norm step
    b["mla_compress_norm_kernel"] = b["mla_compress_kernel"] + b["mla_norm_rope_kernel"]
    f["mla_compress_norm_kernel"] = f["mla_compress_kernel"]
    # the cooperative decode kernel runs every step in one launch
    b["mla_decode_kernel"] = wl.algorithmic_bytes(d, cache)
    f["mla_decode_kernel"] = wl.algorithmic_flops(d)
    return b, f


def csrc_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_attention_prolog_gb300", "csrc")
    for n in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, n), "rb") as fh:
            h.update(n.encode() + fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.md")
    if not os.path.exists(p):
        return None
    vals = {}
    for ln in open(p):
        if ":" in ln and ln.strip().startswith("- "):
            k, v = ln.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("csrc_digest") != csrc_digest():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------- GPU arm

def run_gpu(args):
    from mla_attention_prolog_gb300 import binding

    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = wl.WORKLOADS[args.workload]
    variants = parse_variants(args.variant)
    d = w.dims if not args.tokens else w.dims.with_T(args.tokens)
    d = dataclasses.replace(d, flags=d.flags | sum(wl.VARIANTS[v] for v in variants))
    cached = "cache" in variants
    inp = wl.make_inputs(w, d)
    ww = wl.make_w8a8_weights(w, d) if d.w8a8 else None
    H, Dn, Dv, R = d.num_heads, d.nope_dim, d.v_dim, d.rope_dim

    def bf(a, shape):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).reshape(shape).to(dev)

    # W8A8: the weights live in the handle (loaded once below), not in the sets
    base = dict(x=bf(inp.x, (d.T, d.D)), gamma=bf(inp.gamma, (-1,)),
                W_a=None if ww else bf(inp.W_a, (d.n_a, d.D)), W_b=None if ww else bf(inp.W_b, (-1,)),
                positions=torch.from_numpy(inp.positions).to(dev), cos_sin=torch.from_numpy(inp.cos_sin).to(dev))

    def new_outputs():
        o = dict(out_k=torch.empty((d.T, H, Dn + R), dtype=torch.bfloat16, device=dev),
                 out_v=torch.empty((d.T, H, Dv), dtype=torch.bfloat16, device=dev),
                 out_kpe=torch.empty((d.T, R), dtype=torch.bfloat16, device=dev),
                 out_q_int8=None, out_scale=None)
        if d.q_lora_rank:
            o["out_q_int8"] = torch.empty((d.T, H, Dn + R), dtype=torch.int8, device=dev)
            o["out_scale"] = torch.empty((d.T, H) if d.quant_per_head else (d.T,), dtype=torch.float32,
                                         device=dev)
        if cached:  # a latent cache of 2T slots, token t -> a seeded slot
            o["kv_cache"] = torch.empty((2 * d.T, d.kv_lora_rank + R), dtype=torch.bfloat16, device=dev)
        return o

    if cached:
        base["slot_mapping"] = torch.from_numpy(
            np.random.default_rng(1).permutation(2 * d.T)[:d.T].astype(np.int32)).to(dev)
    set_bytes = sum(t.numel() * t.element_size() for t in base.values() if t is not None)
    set_bytes += sum(t.numel() * t.element_size() for t in new_outputs().values() if t is not None)
    n_sets = max(2, -(-3 * L2_BYTES // set_bytes))
    n_sets = min(n_sets, max(2, int(8e9 // set_bytes)))
    sets = []
    for i in range(n_sets):
        s = {k: (v if i == 0 or v is None else v.clone()) for k, v in base.items()}
        s.update(new_outputs())
        sets.append(s)

    clk = ClockSampler(local).__enter__()
    p = binding.MlaProlog.from_dims(d)
    if ww is not None:
        p.load_w8a8(torch.from_numpy(ww.W_a).to(dev), torch.from_numpy(ww.W_b).to(dev),
                    torch.from_numpy(ww.w_scale).to(dev), stream=torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)
    names = p.kernel_names()
    active = [n for n in names if n != "mla_quant_kernel" or (d.q_lora_rank and not d.quant_per_head)]
    stream = torch.cuda.Stream(device=dev)

    def one(s):
        if cached:
            p.run_cached(s["x"], s["gamma"], s["W_a"], s["W_b"], s["positions"], s["cos_sin"], s["out_k"],
                         s["out_v"], s["out_kpe"], s["out_q_int8"], s["out_scale"], s["slot_mapping"],
                         s["kv_cache"], stream=stream)
        else:
            p.run(s["x"], s["gamma"], s["W_a"], s["W_b"], s["positions"], s["cos_sin"], s["out_k"], s["out_v"],
                  s["out_kpe"], s["out_q_int8"], s["out_scale"], stream=stream)

    # eager warm-up (also builds the tensor maps of each set)
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, n_sets)):
            one(sets[i % n_sets])
    stream.synchronize()
    assert p.device_status(stream) == 0

    # Step time estimate from eager runs, to size K when it is not given.
    t_est0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_sets):
            one(sets[i % n_sets])
    stream.synchronize()
    t_step = (time.perf_counter() - t_est0) / n_sets
    K = args.steps if args.steps else int(min(100000, max(50, 1.0 / t_step)))
    G = K if K <= 200 else 100                     # steps per captured graph
    reps, rem = divmod(K, G)

    def capture(nsteps, hook=None):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(nsteps):
                if hook is not None:
                    p.set_timing_events(hook[i])
                one(sets[i % n_sets])
            if hook is not None:
                p.set_timing_events([])
        return gr

    g = capture(G)
    g_rem = capture(rem) if rem else None
    # instrumented graph: per-step events around every kernel (G steps)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(G)]
    for row in ev:  # create the CUDA events before the capture
        for e in row:
            e.record(stream)
    stream.synchronize()
    gi = capture(G, ev)

    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-args.warmup // G))):
            g.replay()
    stream.synchronize()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = ClockSampler.now()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    stream.synchronize()
    t_wall1 = ClockSampler.now()
    torch.cuda.synchronize()
    barrier(world)
    ms_total = start.elapsed_time(end)
    with torch.cuda.stream(stream):
        gi.replay()
    stream.synchronize()
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / K
    per_kernel = {n: statistics.mean(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(G))
                  for j, n in enumerate(names) if n in active}

    # e2e: host buffers through the public call, pipelined over two device sets
    pin = lambda t: t.cpu().pin_memory()
    hx, hpos = pin(base["x"]), pin(base["positions"])
    outs_h = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in sets[0].items()
              if (k.startswith("out_") or k == "kv_cache") and v is not None}
    h2d = hx.numel() * hx.element_size() + hpos.numel() * hpos.element_size()
    d2h = sum(v.numel() * v.element_size() for v in outs_h.values())
    pipelined = h2d + d2h >= (8 << 20)
    s_in, s_out = (torch.cuda.Stream(), torch.cuda.Stream()) if pipelined else (stream, stream)
    K_e2e = min(K, 2000)
    n_ev = K_e2e + args.warmup
    ev_in = [torch.cuda.Event() for _ in range(n_ev)]
    ev_run = [torch.cuda.Event() for _ in range(n_ev)]
    ev_out = [torch.cuda.Event() for _ in range(n_ev)]

    def e2e_steps(first, n):
        if not pipelined:  # in order on one stream
            s = sets[0]
            with torch.cuda.stream(stream):
                for k in range(first, first + n):
                    s["x"].copy_(hx, non_blocking=True)
                    s["positions"].copy_(hpos, non_blocking=True)
                    one(s)
                    for name, v in outs_h.items():
                        v.copy_(s[name], non_blocking=True)
                ev_out[first + n - 1].record(stream)
            return
        for k in range(first, first + n):
            s = sets[k % 2]
            with torch.cuda.stream(s_in):  # set k % 2 is free once step k - 2 has run
                if k >= 2:
                    s_in.wait_event(ev_run[k - 2])
                s["x"].copy_(hx, non_blocking=True)
                s["positions"].copy_(hpos, non_blocking=True)
                ev_in[k].record(s_in)
            with torch.cuda.stream(stream):  # outputs of set k % 2 copied out by step k - 2
                stream.wait_event(ev_in[k])
                if k >= 2:
                    stream.wait_event(ev_out[k - 2])
                one(s)
                ev_run[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[k])
                for name, v in outs_h.items():
                    v.copy_(s[name], non_blocking=True)
                ev_out[k].record(s_out)

    e2e_steps(0, args.warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    e2e_steps(args.warmup, K_e2e)
    stream.wait_event(ev_out[n_ev - 1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    assert p.device_status(stream) == 0
    clk.__exit__(None, None, None)
    clocks = clk.summary(t_wall0, t_wall1)

    value = whole_job_tokens_per_s(d.T * K, ms_total, world)
    peaks, peak_src = load_peaks()
    kb, kf = kernel_work(d, cached, names)
    dom = max(per_kernel, key=per_kernel.get)
    dom_ms = per_kernel[dom]
    if w.bound == "tensor":
        ach = kf[dom] / (dom_ms / 1e3) / 1e12
        # the burst peak for a kernel timed in a short loop, the sustained
        # (power-capped) one for a kernel timed inside a seconds-long loop
        long_loop = ms_total >= 1000.0 and "bf16_tflops_sustained" in peaks
        peak = peaks["bf16_tflops_sustained"] if long_loop else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "peak_kind": "sustained" if long_loop else "burst"}
    else:
        ach = kb[dom] / (dom_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4)}
    wname = "+".join([args.workload] + variants)
    roof.update({"kernel": dom, "kernel_ms": round(dom_ms, 5), "peak_source": peak_src,
                 "traffic": committed_traffic(dom, wname)})
    abytes = wl.algorithmic_bytes(d, cached)
    whole = {"algorithmic_bytes": abytes, "algorithmic_flops": wl.algorithmic_flops(d),
             "hbm_frac": round(abytes / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
             "tc_frac": round(wl.algorithmic_flops(d) / (ms_step / 1e3) / 1e12 / peaks["bf16_tflops"], 4)}
    if "bf16_tflops_sustained" in peaks:
        whole["tc_frac_of_sustained"] = round(
            wl.algorithmic_flops(d) / (ms_step / 1e3) / 1e12 / peaks["bf16_tflops_sustained"], 4)
    if clocks.get("sm_mhz"):
        # step time x median SM clock: compares runs taken at different
        # (power-capped) clocks
        whole["ms_x_sm_mhz"] = round(ms_step * clocks["sm_mhz"], 2)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 x int8 -> int32 (on bf16 tensor cores)" if d.w8a8 else "bf16",
        "data": "synthetic",
        "config": {"workload": wname, "T": d.T, "D": d.D, "q_lora_rank": d.q_lora_rank,
                   "kv_lora_rank": d.kv_lora_rank, "rope_dim": d.rope_dim, "num_heads": d.num_heads,
                   "nope_dim": d.nope_dim, "v_dim": d.v_dim, "quant_q": d.quant_q, "flags": d.flags,
                   "kv_cache_write": cached,
                   "l2": f"{n_sets} rotating buffer sets of {set_bytes / 1e6:.1f} MB (> 3x L2)",
                   "timing": f"{reps} replay(s) of a {G}-step CUDA graph" + (f" + {rem}" if rem else "")
                             + " between CUDA events", "parallelism": f"replicas x{world}",
                   "schedule": p.schedule(), "inputs_sha256": inp.sha256()[:16]},
        "roofline": roof,
        "whole_step": whole,
        "per_kernel_ms": {k: round(v, 5) for k, v in per_kernel.items()},
        "e2e": {"value": round(whole_job_tokens_per_s(d.T * K_e2e, e2e_ms, world), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K_e2e,
                "pipelined": pipelined},
        "gpu_launches": K * len(active),
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, d)
    p.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def parse_variants(spec: str):
    """'' or a comma list of interleaved, head_norm, per_head, cache."""
    out = [v for v in (x.strip() for x in spec.split(",")) if v]
    for v in out:
        if v not in wl.VARIANTS:
            raise SystemExit(f"unknown variant {v!r}; choose from {sorted(wl.VARIANTS)}")
    return sorted(set(out), key=list(wl.VARIANTS).index)


# ------------------------------------------------------------------ CPU arm

def oracle_sample(w: wl.Workload, max_tokens: int, dims=None):
    """Inputs and a token sample of the workload for the oracle (bounded)."""
    inp = wl.make_inputs(w, dims)
    T = inp.dims.T
    if T <= max_tokens:
        return inp, None
    rng = np.random.default_rng(3)
    return inp, np.sort(rng.choice(T, max_tokens, replace=False)).astype(np.int32)


def oracle_call(w: wl.Workload, inp: wl.Inputs, tok):
    """One oracle pass over the sampled tokens (the W8A8 oracle for W8A8 dims)."""
    import oracle
    d = inp.dims
    if d.w8a8:
        ww = wl.make_w8a8_weights(w, d)
        return lambda: oracle.mla_prolog_w8a8(d, inp.x, inp.gamma, ww.W_a, ww.W_b, ww.w_scale, inp.positions,
                                              inp.cos_sin, tokens=tok)
    return lambda: oracle.mla_prolog(d, inp.x, inp.gamma, inp.W_a, inp.W_b, inp.positions, inp.cos_sin, tokens=tok)


def cpu_baseline(w: wl.Workload, seconds: float, dims=None):
    import oracle
    oracle.build()
    dims = dims or w.dims
    per_tok = wl.algorithmic_flops(dims) / max(1, dims.T)
    max_tokens = max(1, min(dims.T, int(4e10 / per_tok)))  # ~40 GFLOP of fp64 work per call at most
    inp, tok = oracle_sample(w, max_tokens, dims)
    d = inp.dims
    n = d.T if tok is None else len(tok)
    run = oracle_call(w, inp, tok)
    t0 = time.perf_counter()
    calls = 0
    while True:
        run()
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds or el / calls * (calls + 1) > 3 * seconds:
            break
    return {"value": round(n * calls / el, 2), "unit": "tokens/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{calls} call(s) of {n} of the workload's {d.T} tokens ({el:.1f} s wall)"}


def run_reference(args):
    rank, world, _ = dist_info()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = wl.WORKLOADS[args.workload]
    variants = parse_variants(args.variant)  # the same config as the GPU arm's line
    dims = w.dims if not args.tokens else w.dims.with_T(args.tokens)
    dims = dataclasses.replace(dims, flags=dims.flags | sum(wl.VARIANTS[v] for v in variants))
    per_tok = wl.algorithmic_flops(dims) / max(1, dims.T)
    max_tokens = max(1, min(dims.T, int(1e10 / per_tok)))
    inp, tok = oracle_sample(w, max_tokens, dims)
    d = inp.dims
    n = d.T if tok is None else len(tok)
    call = oracle_call(w, inp, tok)
    steps = args.steps or 10
    for _ in range(args.warmup):
        call()
    t0 = time.perf_counter()
    for _ in range(steps):
        call()
    el = time.perf_counter() - t0
    v = n * steps / el
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int64+f32" if d.w8a8 else "f64+f32",
            "data": "synthetic", "config": {"workload": "+".join([args.workload] + variants), "T": d.T},
            "cpu_baseline": {"value": round(v, 2), "unit": "tokens/s", "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": f"{n} of {d.T} tokens per step"},
            "e2e": {"value": round(v, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (default: about one second of steps)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="v3_prefill", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=0,
                    help="override T of the workload (small profiling cases; not a bench line)")
    ap.add_argument("--variant", default="",
                    help="comma list of interleaved, head_norm, per_head (dims flags) and cache "
                         "(the latent KV-cache write); default: the base path")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
