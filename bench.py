#!/usr/bin/env python
"""Throughput of the fused MoE layer forward (libmoe, sm_103a) on GB300.

One step = one moe_forward of a whole layer (routing, align/permute, grouped
SiLU-gated MLP of the local and shared experts, combine) over one batch of
synthetic tokens. The default workload is the Mixtral-8x7B-shape prefill layer
(T=4096, H=4096, I=14336, E=8, top_k=2). Prints one JSON line. On one GPU
the line also carries the other workloads (Qwen3-MoE-shape decode at T = 1, 8
and 64, the DeepSeek-V2-shape prefill, the EP shard), each timed the same way,
under "workloads" (--no-extra skips them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

With N > 1 (torchrun, one rank per GPU) every rank runs its own batch through
its own copy of the layer (replicas: weak scaling, no collective on the data
path). Rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE layer tokens/s and TFLOP/s (bf16) on 1 GB300, % of tensor/HBM roofline"
DATA = ("synthetic: seeded counter-based normals (SplitMix64 + Box-Muller), "
        "random-init weights std 1/sqrt(fan_in)")
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Empties L2 between steps: writes a buffer twice the size of L2, then
    reads another one, so the step starts with no useful and no dirty lines
    (the write alone would leave ~126 MB of dirty lines whose write-back then
    lands inside the next timed step)."""

    def __init__(self, device):
        self.wr = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.rd = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.wr.zero_()
        return self.rd.amax()

WORKLOADS = {w.name: w for w in (synth.TINY, synth.MIXTRAL, synth.DEEPSEEK, synth.EP_SHARD)}
for _t in synth.DECODE_TOKENS:
    WORKLOADS[f"qwen3_decode_T{_t}"] = synth.QWEN_DECODE.with_(name=f"qwen3_decode_T{_t}", T=_t)
# timed beside the headline workload in the same run; the decode sizes last,
# largest T last (their weights are drawn once, with that T's x)
EXTRA_WORKLOADS = ["deepseek_v2_prefill", "ep_shard", "mixtral_prefill",
                   *[f"qwen3_decode_T{t}" for t in sorted(synth.DECODE_TOKENS)]]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                source="fallback")


# --------------------------------------------------------------------------- inputs
def _pinned_bits(seed, tid, row0, nrows, ncols, std):
    t = torch.empty(nrows * ncols, dtype=torch.int16, pin_memory=True)
    synth.draw_bf16_bits(seed, tid, row0, nrows, ncols, std, out_ptr=t.data_ptr())
    return t


def device_layer(wl, device, seed=0):
    """Device tensors of a layer, drawn from synth (no tie-gap redraws: the
    bench measures speed; parity is the tests' job)."""
    bf = wl.act == "bf16"
    e0 = wl.ep_rank * wl.E_local

    def dev(seedrows, shape, f32=False):
        tid, row0, nrows, ncols, std = seedrows
        if bf and not f32:
            t = _pinned_bits(seed, tid, row0, nrows, ncols, std)
            return t.to(device).view(torch.bfloat16).view(*shape)
        a = synth.draw(seed, tid, row0, nrows, ncols, std, False)
        return torch.from_numpy(a).to(device).view(*shape)

    d = {}
    d["x"] = dev((synth.X, 0, wl.T, wl.H, wl.std(synth.X)), (wl.T, wl.H))
    if wl.router == "bf16":
        d["router_w"] = dev((synth.ROUTER_W, 0, wl.E, wl.H, wl.std(synth.ROUTER_W)), (wl.E, wl.H))
    else:
        d["router_w"] = dev((synth.ROUTER_W, 0, wl.E, wl.H, wl.std(synth.ROUTER_W)),
                            (wl.E, wl.H), f32=True)
    d["router_b"] = None
    if wl.router_bias:
        d["router_b"] = torch.from_numpy(synth.draw_tensor(wl, synth.ROUTER_B, seed)).to(device)
    d["w13"] = dev((synth.W13, e0 * 2 * wl.I, wl.E_local * 2 * wl.I, wl.H, wl.std(synth.W13)),
                   (wl.E_local, 2 * wl.I, wl.H))
    d["w2"] = dev((synth.W2, e0 * wl.H, wl.E_local * wl.H, wl.I, wl.std(synth.W2)),
                  (wl.E_local, wl.H, wl.I))
    d["shared_w13"] = d["shared_w2"] = None
    if wl.n_shared:
        d["shared_w13"] = dev((synth.SHARED_W13, 0, wl.n_shared * 2 * wl.I_shared, wl.H,
                               wl.std(synth.SHARED_W13)), (wl.n_shared, 2 * wl.I_shared, wl.H))
        d["shared_w2"] = dev((synth.SHARED_W2, 0, wl.n_shared * wl.H, wl.I_shared,
                              wl.std(synth.SHARED_W2)), (wl.n_shared, wl.H, wl.I_shared))
    return d


def cfg_of(wl):
    from expert_moe_layer_gb300 import binding as B
    return B.make_config(wl.E, wl.K, wl.H, wl.I, wl.renormalize, wl.n_group, wl.topk_group,
                         wl.rsf, wl.n_shared, wl.I_shared, wl.ep_size, wl.ep_rank, wl.act,
                         wl.router, wl.scoring, wl.bias_mode)


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, interval_ms=50):
        import tempfile
        self.proc = None
        # the raw samples go to a temporary file; only their summary is kept
        fd, self.path = tempfile.mkstemp(prefix=f"moe_clocks_gpu{gpu_index}_", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(interval_ms)],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            if getattr(self, "fh", None) is not None:
                self.fh.close()
            os.remove(self.path)
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as fh:
            summary = summarize_clocks(fh)
        os.remove(self.path)
        return summary


def summarize_clocks(lines):
    """Median SM clock, the largest max clock and the throttle reasons that
    were active in any sample, from nvidia-smi CSV rows in ClockSampler.FIELDS
    order (no header, no units). Rows that do not parse are skipped; None when
    no row does."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        f = [c.strip() for c in line.split(",")]
        if len(f) < 9:
            continue
        try:
            sm.append(float(f[1]))
            mx.append(float(f[2]))
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
            "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- ranks
def aggregate_over_ranks(local_ms, tokens_per_rank, steps, world, device=None):
    """Whole-job numbers of a replicated run: the slowest rank's time over the
    K steps, and every rank's tokens. Returns (max total ms, tokens/s)."""
    total = float(local_ms)
    if world > 1:
        t = torch.tensor([total], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total = float(t.item())
    return total, world * tokens_per_rank * steps / (total / 1e3)


# --------------------------------------------------------------------------- our arm
def dominant_kernel_roofline(wl, plan, A, touched, rows, k_ms, peaks):
    """Roofline of the layer's dominant kernel: GEMM1 (gate/up with the SiLU
    epilogue), or for decode-sized batches the fused kernel that runs GEMM1
    and GEMM2 together. GEMM1 on CTA pairs reads the A permuted token rows;
    on single CTAs it gathers them from x itself, where the algorithmic
    bytes count each of the `rows` distinct token rows once (the repeats of
    a row hit L2). Algorithmic FLOPs and bytes per launch over its
    measured duration, against the measured peak: the bf16 burst peak for a
    tensor-bound kernel (the timed regions here last milliseconds, not the
    seconds of the sustained figure, which is reported beside it), the HBM
    copy peak otherwise."""
    eb = 2 if wl.act == "bf16" else 4
    w13_bytes = touched * 2 * wl.I * wl.H * eb
    w2_bytes = touched * wl.H * wl.I * eb
    if plan.fused_mlp:
        kname, ksrc = "moe_mlp_fused (GEMM1 + GEMM2)", "kernels_mlp_fused.cu"
        k_flops = 6 * A * wl.H * wl.I
        # weights once; x rows in, h out and back in, y out
        k_bytes = w13_bytes + w2_bytes + (2 * A * wl.H + 2 * A * wl.I) * eb
    else:
        kname, ksrc = (("moe_gemm_pair<SiLU> (GEMM1, CTA pairs)", "kernels_gemm_pair.cu")
                       if plan.cta_pairs else
                       ("moe_gemm_tc<SiLU> (GEMM1)", "kernels_gemm.cu"))
        k_flops = 4 * A * wl.H * wl.I
        x_rows = A if plan.cta_pairs else rows
        k_bytes = w13_bytes + x_rows * wl.H * eb + A * wl.I * eb
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if k_flops / max(k_bytes, 1) >= ridge:
        ach = k_flops / (k_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4),
                "peak_basis": f"{peaks['source']} bf16 burst (the kernel runs inside a "
                              "timed region of milliseconds)",
                "frac_of_sustained": round(ach / peaks["bf16_tflops_sustained"], 4)}
    else:
        ach = k_bytes / (k_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_basis": f"{peaks['source']} HBM copy",
                "frac_of_nominal_8TBs": round(ach / 8000.0, 4)}
    roof.update({"kernel": kname, "ms_per_launch": round(k_ms, 4),
                 "algorithmic_flops": k_flops, "algorithmic_bytes": k_bytes,
                 "traffic": traffic_from_profile(wl.name, ksrc)})
    return roof


def layer_work(wl, A, touched):
    """Algorithmic FLOPs and bytes of one layer forward: the expert MLPs of
    the A local assignments, the router and shared experts; the weights of
    each touched expert, the router and shared weights, x in and out once."""
    rb = 2 if wl.router == "bf16" else 4
    eb = 2 if wl.act == "bf16" else 4
    alg_bytes = (touched * 3 * wl.H * wl.I * eb + wl.E * wl.H * rb
                 + wl.n_shared * 3 * wl.H * wl.I_shared * eb + 2 * wl.T * wl.H * eb)
    return wl.flops(A), alg_bytes


def layer_roofline(flops, alg_bytes, ms, peaks):
    """The whole layer against both roofs: algorithmic bytes over the HBM copy
    peak, FLOPs over the bf16 burst peak."""
    gbs = alg_bytes / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    return {"gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "tflops": round(tfs, 2), "frac_of_bf16_burst": round(tfs / peaks["bf16_tflops"], 4)}


def time_layer(args, wl, d, device, world, headline):
    """Times moe_forward on one workload: K steps (L2 flush + layer forward)
    captured into one CUDA graph and replayed once, step times from CUDA events
    the library records at each step's start and end. With headline, also the
    eager pass and the per-rank aggregation of the JSON line's main value."""
    from expert_moe_layer_gb300 import binding as B
    peaks = load_peaks()
    cfg = cfg_of(wl)
    T, H = wl.T, wl.H
    ws = torch.empty(B.workspace_size(cfg, T), dtype=torch.uint8, device=device)
    out = torch.empty(T, H, dtype=d["x"].dtype, device=device)
    flush = L2Flush(device)
    stream = torch.cuda.current_stream(device)

    def fwd(events=None):
        if events is None:
            B.moe_forward(cfg, T, d["x"], d["router_w"], d["router_b"], d["w13"], d["w2"],
                          d["shared_w13"], d["shared_w2"], None, out, ws,
                          torch.cuda.current_stream(device))
            return 0
        return B.moe_forward_timed(cfg, T, d["x"], d["router_w"], d["router_b"], d["w13"],
                                   d["w2"], d["shared_w13"], d["shared_w2"], None, out, ws,
                                   events, torch.cuda.current_stream(device))

    for _ in range(args.warmup):
        flush()
        fwd()
    torch.cuda.synchronize(device)
    rc, flags = B.moe_get_status(ws, stream)
    if rc != 0:
        raise RuntimeError(f"{wl.name}: device status {rc} flags {flags:#x} after warm-up")

    # routing statistics of this batch (for the algorithmic work counts)
    lay = B.workspace_layout(cfg, T)
    El = wl.E_local
    counts = ws[lay.counts:lay.counts + 4 * El].view(torch.int32).cpu().numpy()
    A = int(counts.sum())
    touched = int((counts > 0).sum())
    # distinct token rows with at least one local assignment
    tk = ws[lay.topk_ids:lay.topk_ids + 4 * T * wl.K].view(torch.int32).view(T, wl.K)
    rows = int(((tk // El) == wl.ep_rank).any(dim=1).sum().item())

    def new_events(n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(n)]
        for row in evs:             # create the CUDA events (torch creates them lazily)
            for ev in row:
                ev.record(stream)
        return evs

    eager_ms = None
    if headline:
        # Eager pass (host launches every kernel): a secondary number.
        eager_ev = new_events(args.steps)
        torch.cuda.synchronize(device)
        for i in range(args.steps):
            flush()
            fwd(eager_ev[i])
        torch.cuda.synchronize(device)
        eager_ms = statistics.mean(eager_ev[i][0].elapsed_time(eager_ev[i][7])
                                   for i in range(args.steps))

    def capture(evs):
        g = torch.cuda.CUDAGraph()
        cap_stream = torch.cuda.Stream(device)
        cap_stream.wait_stream(stream)
        torch.cuda.synchronize(device)
        n = 0
        with torch.cuda.graph(g, stream=cap_stream):
            for i in range(args.steps):
                flush()
                n += fwd(evs[i])
        torch.cuda.synchronize(device)
        return g, n

    # Timed region: the K steps (L2 flush + layer forward) are captured into one
    # CUDA graph and replayed once, as a serving engine replays its layers. The
    # library records only each step's start and end events, as graph nodes.
    events = new_events(args.steps)
    edges = [[ev[0], None, None, None, None, None, None, ev[7]] for ev in events]
    graph, launches = capture(edges)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    t_start = time.time()
    graph.replay()
    torch.cuda.synchronize(device)
    if world > 1:
        torch.distributed.barrier()
    step_ms = [events[i][0].elapsed_time(events[i][7]) for i in range(args.steps)]
    rc, flags = B.moe_get_status(ws, stream)
    if rc != 0:
        raise RuntimeError(f"{wl.name}: device status {rc} flags {flags:#x} in the timed region")

    # Per-stage breakdown (and the dominant kernel's live duration): a second
    # graph of the same K steps with events at every stage boundary, replayed
    # right after the timed one, under the same clocks.
    sevents = new_events(args.steps)
    sgraph, _ = capture(sevents)
    sgraph.replay()
    torch.cuda.synchronize(device)
    del sgraph

    # nvidia-smi samples every 50 ms and takes a moment to start: a timed
    # region shorter than that is followed by untimed replays of the same
    # graph, so that the clock record covers this workload
    extra = 0
    while time.time() - t_start < 0.6:
        graph.replay()
        torch.cuda.synchronize(device)
        extra += 1
    clocks = sampler.stop()
    if clocks is not None:
        clocks["untimed_replays"] = extra
    del graph

    def span(a, b):
        return [sevents[i][a].elapsed_time(sevents[i][b]) for i in range(args.steps)]

    if headline:
        total_ms, tokens_per_s = aggregate_over_ranks(sum(step_ms), T, args.steps, world,
                                                      device)
    else:
        total_ms = sum(step_ms)
        tokens_per_s = T * args.steps / (total_ms / 1e3)
    stage_names = ["route", "align", "tiles_gather", "gemm1_silu", "gemm2", "shared", "combine"]
    stages = {n: statistics.mean(span(i, i + 1)) for i, n in enumerate(stage_names)}
    ms_per_step = total_ms / args.steps
    flops, alg_bytes = layer_work(wl, A, touched)
    plan = B.forward_plan(cfg, T)
    roof = dominant_kernel_roofline(wl, plan, A, touched, rows, stages["gemm1_silu"], peaks)
    path = {f: getattr(plan, f) for f, _ in B.Plan._fields_}
    e2e = run_e2e(args, wl, cfg, d, ws, out, flush, stream, device, world, alg_bytes)
    res = {
        "value": round(tokens_per_s, 1), "unit": "tokens/s",
        "ms_per_step": round(ms_per_step, 4),
        "tflops": round(flops / (ms_per_step / 1e3) / 1e12, 2),
        "gbs": round(alg_bytes / (ms_per_step / 1e3) / 1e9, 1),
        "layer_roofline": layer_roofline(flops, alg_bytes, ms_per_step, peaks),
        "roofline": roof,
        "config": {"workload": wl.name, "T": T, "H": wl.H, "I": wl.I, "E": wl.E, "K": wl.K,
                   "E_local": El, "shared_experts": wl.n_shared,
                   "ep": [wl.ep_size, wl.ep_rank], "assignments": A,
                   "experts_touched": touched},
        "alg_flops_per_step": flops, "alg_bytes_per_step": alg_bytes,
        "stages_ms": {k: round(v, 4) for k, v in stages.items()},
        "staged_ms_per_step": round(statistics.mean(span(0, 7)), 4),
        "path": path,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if eager_ms is not None:
        res["eager_ms_per_step"] = round(eager_ms, 4)
    return res


L2_NOTE = (f"flushed before every step, outside the timed events: a {L2_FLUSH_BYTES >> 20} "
           f"MiB write, then a {L2_FLUSH_BYTES >> 20} MiB read so that no dirty flush lines "
           "are written back inside the step")
TIMING_NOTE = ("one CUDA graph of the K steps replayed once; step times from CUDA events "
               "the library records at each step's start and end; stage times from a "
               "second graph with events at every stage boundary")


def run_ours(args, wl, rank, world, device):
    from expert_moe_layer_gb300 import binding as B
    B.lib()
    torch.cuda.set_device(device)
    d = device_layer(wl, device)
    r = time_layer(args, wl, d, device, world, headline=True)
    del d
    res = {
        "metric": METRIC, "value": r["value"], "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.act == "bf16" else "f32",
        "data": DATA,
        "config": {**r["config"], "l2": L2_NOTE,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "timing": TIMING_NOTE,
    }
    res.update({k: v for k, v in r.items() if k not in res})
    return res


def extra_workloads(args, headline, device):
    """The other workloads of the layer, each timed as the headline one (graph
    of K steps, L2 flushed outside the events), on this GPU. The decode sizes
    share one set of weights."""
    out = {}
    decode_d = None
    for name in EXTRA_WORKLOADS:
        if name == headline:
            continue
        wl = WORKLOADS[name]
        if name.startswith("qwen3_decode_T"):
            if decode_d is None:
                decode_d = device_layer(WORKLOADS[EXTRA_WORKLOADS[-1]], device)
            d = dict(decode_d)
            d["x"] = decode_d["x"][:wl.T].contiguous()
        else:
            d = device_layer(wl, device)
        r = time_layer(args, wl, d, device, 1, headline=False)
        del d
        torch.cuda.empty_cache()
        out[name] = r
    return out


def run_e2e(args, wl, cfg, d, ws, out, flush, stream, device, world, step_bytes):
    """The layer through moe_forward with every step's input copied in from
    pinned host memory and its output copied back.

    When a step reads more than three times the L2 size (so no flush is
    needed between steps), the steps are pipelined as a serving loop runs them:
    copy streams upload step i+1's tokens and download step i-1's output
    while step i computes, with two input and two output buffers. The time is
    from the first upload to the last download, over the steps. Smaller
    layers run step by step with an L2 flush before each, timed per step."""
    from expert_moe_layer_gb300 import binding as B
    T, H = wl.T, wl.H
    x_host = torch.empty(T, H, dtype=d["x"].dtype, pin_memory=True)
    x_host.copy_(d["x"].cpu())
    n = max(3, min(args.steps, 50))
    nbytes = T * H * x_host.element_size()
    pipelined = step_bytes > 3 * 129 * 2 ** 20

    def fwd(xd, od):
        B.moe_forward(cfg, T, xd, d["router_w"], d["router_b"], d["w13"], d["w2"],
                      d["shared_w13"], d["shared_w2"], None, od, ws, stream)

    if pipelined:
        up = torch.cuda.Stream(device)    # uploads
        down = torch.cuda.Stream(device)  # downloads
        x_dev = [torch.empty_like(d["x"]) for _ in range(2)]
        o_dev = [torch.empty_like(out) for _ in range(2)]
        o_host = [torch.empty(T, H, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        ev = lambda: torch.cuda.Event(enable_timing=True)
        warm = 2
        total = n + warm
        h2d = [ev() for _ in range(total)]
        done = [ev() for _ in range(total)]
        d2h = [ev() for _ in range(total)]
        start = [ev() for _ in range(total)]
        torch.cuda.synchronize(device)
        for i in range(total):
            b = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(done[i - 2])  # step i-2 no longer reads x_dev[b]
                start[i].record(up)
                x_dev[b].copy_(x_host, non_blocking=True)
                h2d[i].record(up)
            stream.wait_event(h2d[i])
            if i >= 2:
                stream.wait_event(d2h[i - 2])  # step i-2's output is downloaded
            fwd(x_dev[b], o_dev[b])
            done[i].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(done[i])
                o_host[b].copy_(o_dev[b], non_blocking=True)
                d2h[i].record(down)
        torch.cuda.synchronize(device)
        ms = start[warm].elapsed_time(d2h[total - 1]) / n
        mode = ("pipelined: copy streams upload step i+1 and download step i-1 while step "
                "i computes; no L2 flush (a step reads over 3x the L2 size)")
    else:
        out_host = torch.empty(T, H, dtype=out.dtype, pin_memory=True)
        x_dev = torch.empty_like(d["x"])
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        for i in range(n + 2):
            flush()
            if i >= 2:
                evs[i - 2][0].record(stream)
            x_dev.copy_(x_host, non_blocking=True)
            fwd(x_dev, out)
            out_host.copy_(out, non_blocking=True)
            if i >= 2:
                evs[i - 2][1].record(stream)
        torch.cuda.synchronize(device)
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        mode = "step by step, L2 flushed before each step, outside the timed copies"
    if world > 1:
        t = torch.tensor([ms], device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    return {"value": round(world * T / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
            "ms_per_step": round(ms, 4), "steps": n, "mode": mode}


def traffic_from_profile(workload, kernel_source, root=ROOT):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when there is none for this workload or the kernel's
    source changed since the capture."""
    import hashlib
    p = os.path.join(root, "profiles", "dominant_kernel_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    v = d["workloads"].get(workload)
    if v is None or os.path.basename(v["kernel_source"]) != kernel_source:
        return None
    with open(os.path.join(root, v["kernel_source"]), "rb") as fh:
        if hashlib.sha256(fh.read()).hexdigest() != v["kernel_sha256"]:
            return None
    return v.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------- oracle arms
def oracle_sample(wl, n_tokens, seed=0):
    """Host inputs for the oracle on the first n_tokens of the workload."""
    bf = wl.act == "bf16"
    e0 = wl.ep_rank * wl.E_local
    x = synth.draw(seed, synth.X, 0, n_tokens, wl.H, wl.std(synth.X), bf)
    rw = synth.draw_tensor(wl, synth.ROUTER_W, seed)
    rb = synth.draw_tensor(wl, synth.ROUTER_B, seed) if wl.router_bias else None
    if bf:
        w13 = synth.BF16Experts(synth.draw_bf16_bits(
            seed, synth.W13, e0 * 2 * wl.I, wl.E_local * 2 * wl.I, wl.H,
            wl.std(synth.W13)).reshape(wl.E_local, 2 * wl.I, wl.H))
        w2 = synth.BF16Experts(synth.draw_bf16_bits(
            seed, synth.W2, e0 * wl.H, wl.E_local * wl.H, wl.I,
            wl.std(synth.W2)).reshape(wl.E_local, wl.H, wl.I))
    else:
        w13 = synth.draw_tensor(wl, synth.W13, seed)
        w2 = synth.draw_tensor(wl, synth.W2, seed)
    s13 = synth.draw_tensor(wl, synth.SHARED_W13, seed) if wl.n_shared else None
    s2 = synth.draw_tensor(wl, synth.SHARED_W2, seed) if wl.n_shared else None
    return x, rw, rb, w13, w2, s13, s2


def oracle_step(wl, inputs):
    from oracle import moe_oracle as O
    x, rw, rb, w13, w2, s13, s2 = inputs
    return O.moe_forward(x, rw, w13, w2, top_k=wl.K, renormalize=wl.renormalize,
                         n_group=wl.n_group, topk_group=wl.topk_group, rsf=wl.rsf, router_b=rb,
                         shared_w13=s13, shared_w2=s2,
                         emap=O.expert_map(wl.E, wl.ep_size, wl.ep_rank),
                         scoring=wl.scoring, bias_mode=wl.bias_mode)


def oracle_tokens(wl):
    # bounded sample: roughly 5-20 s of host work per call on the prefill layers
    return min(wl.T, {"mixtral_prefill": 64, "deepseek_v2_prefill": 32,
                      "ep_shard": 128}.get(wl.name, wl.T))


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(wl):
    n = oracle_tokens(wl)
    inputs = oracle_sample(wl, n)
    t0 = time.perf_counter()
    oracle_step(wl, inputs)
    dt = time.perf_counter() - t0
    return {"value": round(n / dt, 3), "unit": "tokens/s", "cores": cores_used(),
            "kind": "oracle",
            "sample": f"first {n} of {wl.T} tokens of {wl.name}, one oracle forward "
                      f"(numpy fp64 MLP, fp32 softmax), {dt:.1f} s"}


def run_reference(args, wl):
    n = oracle_tokens(wl)
    inputs = oracle_sample(wl, n)
    for _ in range(args.warmup):
        oracle_step(wl, inputs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(wl, inputs)
    dt = time.perf_counter() - t0
    v = n * args.steps / dt
    return {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E,
                       "K": wl.K, "tokens_per_step": n},
            "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": cores_used(),
                             "kind": "oracle",
                             "sample": f"first {n} of {wl.T} tokens per step"},
            "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------------- EP dispatch
def run_ep_dispatch(args, device):
    """One expert-parallel rank's step at the EP-shard shape (T=8192 own tokens,
    E=256, K=8, ep 4, rank 1): route, dispatch, the exchange, expert compute on
    what the rank receives, the return, combine. No collective runs here; the
    exchange stand-in is device copies. This rank receives its own segment for
    rank 1 from each of the 4 ranks (the sources are assumed alike), so it
    computes about T*K items as a real rank does. The rows returned for its
    items sent elsewhere are zero, a stand-in for the other ranks' results,
    and do not change the work. Timed per call with CUDA events, eager, L2
    flushed before each step."""
    from expert_moe_layer_gb300 import binding as B
    wl = synth.EP_SHARD
    T, H, K, E, ep, r = wl.T, wl.H, wl.K, wl.E, wl.ep_size, wl.ep_rank
    cfg = cfg_of(wl)
    d = device_layer(wl, device)
    peaks = load_peaks()
    n = T * K
    stream = torch.cuda.current_stream(device)
    ids = torch.empty(T, K, dtype=torch.int32, device=device)
    w = torch.empty(T, K, dtype=torch.float32, device=device)
    rws = torch.empty(B.route_workspace_size(cfg, T), dtype=torch.uint8, device=device)
    counts = torch.empty(ep, dtype=torch.int32, device=device)
    offsets = torch.empty(ep + 1, dtype=torch.int32, device=device)
    pos = torch.empty(n, dtype=torch.int32, device=device)
    sx = torch.empty(n, H, dtype=torch.bfloat16, device=device)
    sids = torch.empty(n, dtype=torch.int32, device=device)
    sw = torch.empty(n, dtype=torch.float32, device=device)
    stok = torch.empty(n, dtype=torch.int32, device=device)
    dws = torch.empty(B.ep_dispatch_workspace_size(cfg, T), dtype=torch.uint8, device=device)
    # the receive side is sized from one routing of this batch
    B.moe_route(cfg, T, d["x"], d["router_w"], d["router_b"], ids, w, rws)
    B.moe_ep_dispatch(cfg, T, d["x"], ids, w, counts, offsets, pos, sx, sids, sw, stok, dws)
    off = offsets.cpu().numpy()
    c_r = int(off[r + 1] - off[r])
    R = ep * c_r
    rx = torch.empty(R, H, dtype=torch.bfloat16, device=device)
    rids = torch.empty(R, dtype=torch.int32, device=device)
    rw = torch.empty(R, dtype=torch.float32, device=device)
    y = torch.empty(R, H, dtype=torch.bfloat16, device=device)
    ret = torch.zeros(n, H, dtype=torch.bfloat16, device=device)
    cws = torch.empty(B.ep_expert_compute_workspace_size(cfg, R), dtype=torch.uint8,
                      device=device)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    sws = torch.zeros(256, dtype=torch.uint8, device=device)
    flush = L2Flush(device)
    names = ["route", "dispatch", "exchange", "expert_compute", "return", "combine"]

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        B.moe_route(cfg, T, d["x"], d["router_w"], d["router_b"], ids, w, rws, stream)
        mark(1)
        B.moe_ep_dispatch(cfg, T, d["x"], ids, w, counts, offsets, pos, sx, sids, sw, stok,
                          dws, stream)
        mark(2)
        seg = slice(int(off[r]), int(off[r + 1]))
        for s in range(ep):
            rx[s * c_r:(s + 1) * c_r].copy_(sx[seg])
            rids[s * c_r:(s + 1) * c_r].copy_(sids[seg])
            rw[s * c_r:(s + 1) * c_r].copy_(sw[seg])
        mark(3)
        B.moe_ep_expert_compute(cfg, R, rx, rids, rw, d["w13"], d["w2"], y, cws, stream)
        mark(4)
        ret[seg].copy_(y[:c_r])
        mark(5)
        B.moe_ep_combine(cfg, T, ret, pos, None, out, sws, stream)
        mark(6)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(device)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    sampler = ClockSampler(device.index if device.index is not None else 0)
    for i in range(args.steps):
        flush()
        step(evs[i])
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    for ws in (rws, dws, cws, sws):
        rc, flags = B.moe_get_status(ws, stream)
        if rc != 0:
            raise RuntimeError(f"device status {rc} flags {flags:#x}")
    per = {nm: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
           for j, nm in enumerate(names)}
    ms = statistics.mean(e[0].elapsed_time(e[6]) for e in evs)
    eb = 2
    # algorithmic bytes: dispatch reads x once and writes the send buffers;
    # combine reads the returned rows and writes out
    disp_bytes = T * H * eb + n * H * eb + n * 16
    comb_bytes = n * H * eb + T * H * eb + n * 4
    hbm = peaks["hbm_gbs"]
    return {"metric": "EP rank step tokens/s (route, dispatch, expert compute, combine; "
                      "exchange stand-in: device copies)",
            "value": round(T / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "dtype": "bf16", "data": DATA,
            "config": {"workload": "ep_dispatch", "T": T, "H": H, "I": wl.I, "E": E, "K": K,
                       "ep": [ep, r], "items_sent": n, "items_received": R,
                       "l2": "flushed before every step, outside the timed events"},
            "calls_ms": {k: round(v, 4) for k, v in per.items()},
            "dispatch": {"bytes": disp_bytes, "gbs": round(disp_bytes / per["dispatch"] / 1e6, 1),
                         "frac_of_hbm": round(disp_bytes / per["dispatch"] / 1e6 / hbm, 4)},
            "combine": {"bytes": comb_bytes, "gbs": round(comb_bytes / per["combine"] / 1e6, 1),
                        "frac_of_hbm": round(comb_bytes / per["combine"] / 1e6 / hbm, 4)},
            "peak_basis": f"{peaks['source']} HBM copy {hbm} GB/s",
            "clocks": clocks}


# --------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["ep_dispatch"],
                    default="mixtral_prefill")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only --workload (by default rank 0 of a 1-GPU run also times "
                         "the other workloads and reports them under 'workloads')")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload == "ep_dispatch":
        print(json.dumps(run_ep_dispatch(args, torch.device("cuda", 0))), flush=True)
        return
    wl = WORKLOADS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, wl)), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local_rank)
    res = run_ours(args, wl, rank, world, device)
    if rank == 0:
        if world == 1 and not args.no_extra:
            res["workloads"] = extra_workloads(args, wl.name, device)
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(wl)
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
