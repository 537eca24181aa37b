"""Benchmark of one MoE layer's prefill on GB300 (tokens/s and grouped-GEMM
TFLOP/s), with the CPU oracle timed beside it.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config c5] [--configs c2,c3,c4,c5]
                [--impl ours|reference]

One step = the MoE-layer prefill of one config through the C ABI over T
tokens of seeded synthetic input (every layer of the config: routing + route
map, gate/up GEMM with the row gather, SwiGLU, down GEMM + scatter-add,
shared experts and layer chaining where the config has them), experts
resident in HBM. The headline line is the Mixtral-shaped layer (T=4096,
H=4096, F=14336: the largest config, tensor-core bound); every config of
--configs is measured the same way under "configs" (resident, end to end,
4-bit experts, router, and the arena-paged call, whose bound is the host
link, in the three loading schedules of EStream Fig. 6: after routing,
prefetch before routing, and on demand through one bank). Under torchrun each rank runs its own replica on its own T tokens
(weak scaling, no collective on the data path).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from routed_expert_ffn_topk_gb300 import workloads as W  # noqa: E402  (seeded inputs only)

METRIC = "MoE-layer prefill tokens/sec and grouped-GEMM TFLOP/s vs bf16 peak (1 GB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one fused expert-kernel launch on the
# OLMoE-shaped layer, from an ncu capture of that kernel. Reported only while
# the kernel source is the one that was captured.
PROFILED_TRAFFIC = {
    "c2": {"kernel_sha256_16": "069fc538aec109ce", "bytes": 858343936},
}
KERNEL_SRC = [os.path.join(ROOT, "routed_expert_ffn_topk_gb300", "csrc", f)
              for f in ("expert_gemm.cu", "tc_ptx.cuh")]


def kernel_source_hash() -> str:
    """sha256 prefix of the expert kernel's sources with comments and blank
    lines removed, so that the traffic record survives comment-only edits."""
    import hashlib
    import re
    h = hashlib.sha256()
    for path in KERNEL_SRC:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for line in text.splitlines():
            line = re.sub(r"//.*$", "", line).rstrip()
            if line.strip():
                h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(config: str):
    rec = PROFILED_TRAFFIC.get(config)
    if not rec:
        return None
    return rec["bytes"] if kernel_source_hash() == rec["kernel_sha256_16"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


# --------------------------------------------------------------------------
# distributed plumbing (timing only)
# --------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str | None):
        self.path = path
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            out = open(self.path, "w") if self.path else subprocess.PIPE
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=out, stderr=subprocess.DEVNULL, text=True)
            self._out = out
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.path:
            self._out.close()
            with open(self.path) as f:
                self.lines = f.read().splitlines()
        else:
            self.lines = self.proc.stdout.read().splitlines()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# workload accounting
# --------------------------------------------------------------------------

def algorithmic(cfg, n_active_per_layer):
    """Algorithmic (minimum) bytes and FLOPs of one layer's routed fused
    expert kernel: the weights of the experts with routes (gate, up, down:
    3*H*F*2 bytes each), X read once (T*H*2) and Y read and written
    (2*T*H*4). The fp16 h intermediate (2*R*F*2 bytes, L2-resident at these
    sizes) is implementation traffic and not counted. Returned as the old
    (gate/up, down) split so callers can sum them."""
    H, F, T, R = cfg.H, cfg.F, cfg.T, cfg.T * cfg.k
    gu = n_active_per_layer * 2 * H * F * 2 + T * H * 2
    dn = n_active_per_layer * H * F * 2 + 2 * T * H * 4
    return gu, dn, 4.0 * H * F * R, 2.0 * H * F * R


def active_experts(cfg, logits_layers):
    """Experts with at least one route (ties at the k-th logit do not occur
    with continuous random logits)."""
    import torch
    out = []
    for lg in logits_layers:
        ids = torch.topk(lg, cfg.k, dim=1).indices
        out.append(int(torch.unique(ids).numel()))
    return out


# --------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# --------------------------------------------------------------------------

def oracle_tokens_per_s(cfg, wl, target_s=10.0, max_tokens=None):
    """Time the oracle as it stands on a bounded sample of tokens of layer 0:
    routing over all T tokens, Eq. 2 for the sampled rows."""
    import numpy as np

    import oracle
    from routed_expert_ffn_topk_gb300 import workloads as W
    lw = wl.layers[0]
    shared = (lw.Sg, lw.Su, lw.Sd) if cfg.n_shared else None
    n = 4
    while True:
        rows = W.sample_rows(cfg.T, n, seed=1).numpy()
        t0 = time.perf_counter()
        ids, alpha = oracle.route_topk(wl.logits[0].numpy(), cfg.k, cfg.renorm)
        oracle.moe_layer_rows(wl.X, lw.Wg, lw.Wu, lw.Wd, ids, alpha, rows=rows, shared=shared)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or len(rows) >= cfg.T or (max_tokens and len(rows) >= max_tokens):
            break
        n = int(min(cfg.T, max(n * 2, n * target_s / max(dt, 1e-3))))
    return len(rows) / dt, len(rows), dt, oracle.num_threads()


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def roofline_of(cfg, stats, steps, n_active, peaks, form="auto"):
    """Roofline of the routed fused expert kernel from the library's CUDA-event
    times (launching stream): algorithmic bytes (active experts' weights + X
    once + Y read and written) or FLOPs (6*H*F per route) per launch over the
    average launch time. Tensor roof (sustained bf16) when the arithmetic
    intensity is above the ridge, HBM roof below it."""
    from routed_expert_ffn_topk_gb300 import estream as es
    L = cfg.layers
    ffn_b = ffn_f = 0.0
    for l in range(L):
        a, b, c, d = algorithmic(cfg, n_active[l])
        ffn_b += a + b
        ffn_f += c + d
    n_ffn = max(1, stats["n_ffn"])
    ffn_ms = stats["ms_ffn"] / n_ffn
    launches_per_step = n_ffn / steps
    per_launch_bytes = ffn_b / launches_per_step
    per_launch_flops = ffn_f / launches_per_step
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    pair = form == "pair" or (form == "auto" and   # the library's automatic choice
                              cfg.T * cfg.k >= es.PAIR_MIN_ROWS * cfg.E)
    kname = ("k_expert_ffn_pair (CTA pairs, 256-record tiles" if pair else
             "k_expert_ffn (128-record tiles") + ": gather + gate/up + SwiGLU + down + scatter)"
    if ffn_f / ffn_b < ridge:
        achieved = per_launch_bytes / (ffn_ms / 1e3) / 1e9
        roof = {"kernel": kname, "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None}
    else:
        # timed inside seconds of back-to-back steps: the sustained (power-capped)
        # bf16 figure is the denominator; the burst one is kept beside it
        sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        achieved = per_launch_flops / (ffn_ms / 1e3) / 1e12
        roof = {"kernel": kname, "bound": "tensor", "achieved": round(achieved, 1),
                "peak": sus, "peak_kind": "sustained", "unit": "TFLOP/s",
                "frac": round(achieved / sus, 4),
                "frac_of_burst_peak": round(achieved / peaks["bf16_tflops"], 4), "traffic": None}
    roof["peak_source"] = peaks["source"]
    roof["traffic"] = profiled_traffic(cfg.key) if L == 1 else None
    roof["algorithmic_bytes_per_launch"] = int(per_launch_bytes)
    roof["algorithmic_flops_per_launch"] = int(per_launch_flops)
    roof["arithmetic_intensity"] = round(ffn_f / ffn_b, 1)
    roof["ms_per_launch"] = round(ffn_ms, 4)
    kernels = {
        "route_ms": round(stats["ms_route"] / steps, 4),
        "ffn_ms": round(stats["ms_ffn"] / steps, 4),
        "shared_ms": round(stats["ms_shared"] / steps, 4),
        "ffn_GBps": round(ffn_b / (stats["ms_ffn"] / steps / 1e3) / 1e9, 1),
        "ffn_TFLOPs": round(ffn_f / (stats["ms_ffn"] / steps / 1e3) / 1e12, 1),
    }
    return roof, kernels


def measure_config(args, cfg, wl, dev, flush, peaks, world, rank):
    """One config's resident step (every layer: routing + route map, the
    fused expert kernel, shared experts and layer chaining where the config
    has them), experts resident in HBM:
      - device throughput: the step replayed from one CUDA graph, L2 flushed
        before every step (outside the timed events), CUDA events on the
        launching stream; per-kernel times from the library's own events on
        an eager pass of the same steps;
      - e2e: the same step as eager C-ABI calls with every step's inputs
        copied from pinned host memory and Y read back to pinned host memory
        inside the timed events, same L2 policy;
      - e2e_pipelined_graph: requests pipelined over two buffer sets and two
        copy streams around graph replays (a serving loop's form).
    Then the router, the 4-bit experts and the arena-paged run of the config."""
    import torch

    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack

    stream = torch.cuda.current_stream()
    L = cfg.layers
    X0 = wl.X.to(dev)
    logits = [lg.to(dev) for lg in wl.logits]
    Xbuf = [X0] + [torch.empty_like(X0) for _ in range(L - 1)]
    Y = [torch.empty(cfg.T, cfg.H, dtype=torch.float32, device=dev) for _ in range(L)]
    one = cfg.__class__(**{**cfg.__dict__, "layers": 1})
    # one resident arena per layer (every expert of every layer in HBM)
    form = {"auto": es.FFN_AUTO, "single": es.FFN_SINGLE, "pair": es.FFN_PAIR}[args.ffn_form]
    stacks = [BoundLayerStack(W.Workload(one, [wl.logits[l]], wl.X, [wl.layers[l]]), mode="resident",
                              ffn_form=form)
              for l in range(L)]

    def make_step(X_in, lg_in, Y_out):
        """One step over the layer stack reading X_in / lg_in and leaving the
        last layer's Y in Y_out (the intermediate buffers are shared)."""
        def run():
            for l in range(L):
                X_l = X_in if l == 0 else Xbuf[l]
                Y_l = Y_out if l == L - 1 else Y[l]
                # Y_l = X_l + MoE_l(X_l): the residual of Eq. 2 is the layer input
                stacks[l].prefill(0, X_l, lg_in[l], Y_l, residual=X_l)
                if l + 1 < L:
                    es.cast_f32_bf16(Y_l, Xbuf[l + 1])
        return run

    step = make_step(Xbuf[0], logits, Y[L - 1])

    def for_all(fn, *a):
        return [fn(st.ctx, *a) for st in stacks]

    def merged_stats():
        out = None
        for st in stacks:
            s_ = es.last_stats(st.ctx)
            if out is None:
                out = dict(s_)
            else:
                for k_, v in s_.items():
                    out[k_] += v
        return out

    def timed_loop(n, fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for i in range(n):
            flush.zero_()
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    # ---- warm-up, then the timed region (clocks sampled throughout) ----
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    for_all(es.reset_stats)
    for_all(es.set_timing, True)
    clocks = ClockSampler(dev.index, None)
    graph, graph_note = None, "eager (--no-graph)"
    with clocks:
        t_end = time.time() + 0.6   # let the sampler see the GPU under this load
        while time.time() < t_end:
            step()
        torch.cuda.synchronize()
        # per-kernel times from the library's own CUDA events (eager steps)
        for_all(es.reset_stats)
        timed_loop(args.steps, step)
        stats = merged_stats()
        for_all(es.set_timing, False)
        assert all(e == es.OK for e in for_all(es.get_device_error))
        # the timed step: one CUDA-graph replay of the whole step (the L2 flush
        # stays outside the graph); eager launches if capture is refused
        if not args.no_graph:
            try:
                graph = capture_graph(step)
                graph_note = "cuda-graph replay"
            except Exception as ex:  # capture refused: time eager launches
                graph, graph_note = None, f"eager (graph capture failed: {type(ex).__name__})"
        barrier(world)
        torch.cuda.synchronize()
        times = timed_loop(args.steps, graph.replay if graph is not None else step)
        barrier(world)
    assert all(e == es.OK for e in for_all(es.get_device_error))
    ms_per_step = max_over_ranks(sum(times), world, dev) / args.steps
    tokens = cfg.T * world
    value = tokens / (ms_per_step / 1e3)
    gpu_launches = stats["launches"] + (L - 1) * args.steps   # + the bf16 casts between layers

    n_active = active_experts(cfg, wl.logits)
    roof, kernels = roofline_of(cfg, stats, args.steps, n_active, peaks, args.ffn_form)
    flops_step = cfg.flops_per_layer() * L
    gemm_ms = (stats["ms_ffn"] + stats["ms_shared"]) / args.steps
    tflops = flops_step / (ms_per_step / 1e3) / 1e12
    gemm_tflops = flops_step / (gemm_ms / 1e3) / 1e12

    # ---- end to end through the C ABI with host buffers, eager calls ----
    Xh = wl.X.pin_memory()
    lgh = [lg.pin_memory() for lg in wl.logits]
    Yh = torch.empty(cfg.T, cfg.H, dtype=torch.float32).pin_memory()
    h2d_b = Xh.numel() * Xh.element_size() + sum(t.numel() * 4 for t in lgh)
    d2h_b = Yh.numel() * 4

    def api_step():
        Xbuf[0].copy_(Xh, non_blocking=True)
        for l in range(L):
            logits[l].copy_(lgh[l], non_blocking=True)
        step()
        Yh.copy_(Y[L - 1], non_blocking=True)

    for _ in range(2):
        api_step()
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(sum(timed_loop(args.steps, api_step)), world, dev) / args.steps
    assert all(e == es.OK for e in for_all(es.get_device_error))
    e2e = {"value": round(tokens / (e2e_ms / 1e3), 1), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
           "mode": "eager C-ABI calls (estream_moe_layer_prefill_residual per layer) each step, "
                   "inputs copied from pinned host memory and Y read back to pinned host memory "
                   "inside the timed events on the compute stream",
           "l2": "flushed before every step (outside the timed events), as for value"}

    # ---- requests pipelined around graph replays (two buffer sets, two copy streams) ----
    e2e_pipe = None
    if graph is not None:
        Yh2 = [Yh, torch.empty_like(Yh).pin_memory()]
        # the second set starts as a copy of the first: the capture's warm-up
        # runs read it before the pipelined loop writes it
        sets = [(Xbuf[0], logits, Y[L - 1]),
                (Xbuf[0].clone(), [t.clone() for t in logits], torch.empty_like(Y[L - 1]))]
        try:
            graphs_b = [graph, capture_graph(make_step(*sets[1]))]
        except Exception:
            graphs_b = None
        if graphs_b is not None:
            h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
            ev = {k_: [torch.cuda.Event() for _ in range(2)] for k_ in ("h2d", "comp", "d2h")}

            def pipe_run(n):
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(h2d_s)
                for i in range(n):
                    b = i % 2
                    Xd, lgd, Yd = sets[b]
                    with torch.cuda.stream(h2d_s):
                        if i >= 2:
                            h2d_s.wait_event(ev["comp"][b])     # step i-2 has read this set
                        Xd.copy_(Xh, non_blocking=True)
                        for l in range(L):
                            lgd[l].copy_(lgh[l], non_blocking=True)
                        ev["h2d"][b].record(h2d_s)
                    stream.wait_event(ev["h2d"][b])
                    if i >= 2:
                        stream.wait_event(ev["d2h"][b])         # step i-2's Y has left the device
                    graphs_b[b].replay()
                    ev["comp"][b].record(stream)
                    with torch.cuda.stream(d2h_s):
                        d2h_s.wait_event(ev["comp"][b])
                        Yh2[b].copy_(Yd, non_blocking=True)
                        ev["d2h"][b].record(d2h_s)
                t1.record(d2h_s)
                torch.cuda.synchronize()
                return t0.elapsed_time(t1)

            pipe_run(4)
            barrier(world)
            pipe_ms = max_over_ranks(pipe_run(args.steps), world, dev) / args.steps
            assert all(e == es.OK for e in for_all(es.get_device_error))
            e2e_pipe = {"value": round(tokens / (pipe_ms / 1e3), 1), "unit": "tokens/s",
                        "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
                        "mode": "requests pipelined: two device buffer sets, inputs copied on one "
                                "copy stream and Y returned on another while the neighbouring "
                                "steps' graph replays compute",
                        "l2": "not flushed"}
            graphs_b = None
    torch.cuda.synchronize()
    # the graphs reference the contexts' events: release them before the contexts go
    graph = None
    for st in stacks:
        st.close()

    rec = {
        "workload": workload_config(cfg, world)["workload"],
        "tokens_per_s": round(value, 1), "ms_per_step": round(ms_per_step, 5),
        "step": graph_note, "tflops": round(tflops, 1),
        "grouped_gemm_tflops": round(gemm_tflops, 1),
        "frac_bf16_peak": round(gemm_tflops / peaks["bf16_tflops"], 4),
        "roofline": roof, "kernels": kernels, "e2e": e2e, "e2e_pipelined_graph": e2e_pipe,
        "gpu_launches": gpu_launches, "clocks": clocks.summary(),
    }

    # ---- router logits upstream of the top-k (its own kernel, not part of the step) ----
    if cfg.dtype == "bf16" and not args.no_router:
        rec["router"] = measure_router(cfg, X0, dev, stream, flush, peaks, args.steps)
    # ---- the same layer with 4-bit experts ----
    if cfg.dtype == "bf16" and not args.no_q4:
        rec["q4"] = measure_q4(args, cfg, wl, dev, stream, flush, peaks)
    # ---- arena-paged run of the same config (host-link bound) ----
    if not args.no_paged:
        paged = measure_paged(args, cfg, wl, dev, stream, flush, peaks)
        if args.pipeline_study and cfg.layers == 1:
            paged["pipeline_study"] = pipeline_study(cfg, wl, dev, flush)
        if args.pipeline_study and cfg.layers > 1:
            paged["layer_granular_study"] = layer_granular_study(cfg, wl, dev, flush)
        rec["paged"] = paged
    del X0, logits, Xbuf, Y
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args, rank, world, local_rank):
    """The headline config's line, with every config of the set measured the
    same way under "configs"."""
    import torch

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    # host threads (and so the pinned pools and staging buffers they allocate)
    # on the CPU NUMA node attached to this GPU, when the host has several
    host = bind_to_gpu_numa_node(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > L2
    keys = [args.config] if args.no_configs else \
        [k for k in args.configs.split(",") if k != args.config] + [args.config]
    recs = {}
    cpu_baseline = None
    for key in keys:
        cfg = W.CONFIGS[key]
        wl = W.make_workload(cfg, seed=W.CONFIG_SEEDS[cfg.key] + 100 * rank)
        recs[key] = measure_config(args, cfg, wl, dev, flush, peaks, world, rank)
        if key == args.config and rank == 0 and not args.no_cpu_baseline:
            # the oracle as it stands, on the host's cores, on a bounded sample
            if host.get("restore") is not None:
                os.sched_setaffinity(0, host["restore"])
            tps, n, dt, cores = oracle_tokens_per_s(cfg, wl, target_s=10.0)
            cpu_baseline = {"value": round(tps, 3), "unit": "tokens/s", "cores": cores,
                            "kind": "oracle",
                            "sample": f"routing of all {cfg.T} tokens + Eq.2 for {n} sampled "
                                      f"tokens of layer 0 ({dt:.1f} s)"}
        del wl
    head = recs[args.config]
    cfg = W.CONFIGS[args.config]
    line = {
        "metric": METRIC, "value": head["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 gate/up, fp16 down (fp32 accumulate)" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; random-init weights)",
        "config": {**workload_config(cfg, world), "step": head["step"]},
        "tflops": head["tflops"], "grouped_gemm_tflops": head["grouped_gemm_tflops"],
        "frac_bf16_peak": head["frac_bf16_peak"],
        "roofline": head["roofline"], "kernels": head["kernels"],
        "e2e": head["e2e"], "e2e_pipelined_graph": head["e2e_pipelined_graph"],
        "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
        "router": head.get("router"), "q4": head.get("q4"), "paged": head.get("paged"),
        "h2d_link": h2d_link_by_numa_node(dev) if not args.no_paged else None,
        "host_numa": {k: v for k, v in host.items() if k != "restore"},
    }
    if cpu_baseline is not None:
        line["cpu_baseline"] = cpu_baseline
    if not args.no_configs:
        line["configs"] = {k: recs[k] for k in sorted(recs)}
    return line


def _numa_cpus():
    """CPU NUMA nodes of this host: {node: set of CPUs} (nodes without CPUs,
    such as a GPU's own memory exposed as a node, are left out)."""
    import glob
    out = {}
    for d in sorted(glob.glob("/sys/devices/system/node/node[0-9]*")):
        try:
            with open(os.path.join(d, "cpulist")) as f:
                spec = f.read().strip()
        except OSError:
            continue
        cpus = set()
        for part in filter(None, spec.split(",")):
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
        if cpus:
            out[int(os.path.basename(d)[4:])] = cpus
    return out


def _gpu_numa_node(index: int):
    """The CPU NUMA node nvidia-smi reports as the GPU's affinity, or None."""
    try:
        r = subprocess.run(["nvidia-smi", "topo", "-m"], capture_output=True, text=True, timeout=20)
    except Exception:
        return None
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    if not lines:
        return None
    head = lines[0].split("\t")
    col = next((i for i, h in enumerate(head) if "NUMA Affinity" in h), None)
    for ln in lines[1:]:
        cells = ln.split("\t")
        if cells and cells[0].strip() == f"GPU{index}" and col is not None and col < len(cells):
            try:
                return int(cells[col].strip().split(",")[0].split("-")[0])
            except ValueError:
                return None
    return None


def bind_to_gpu_numa_node(dev):
    """Restrict this thread (and the threads it starts later) to the CPUs of
    the NUMA node nvidia-smi names as the GPU's affinity, so that pinned host
    buffers are placed there. Returns what was done, and the previous CPU set
    under "restore"."""
    nodes = _numa_cpus()
    node = _gpu_numa_node(dev.index)
    info = {"cpu_numa_nodes": sorted(nodes), "gpu_numa_node": node, "bound": False, "restore": None}
    if node in nodes and len(nodes) > 1 and hasattr(os, "sched_setaffinity"):
        info["restore"] = os.sched_getaffinity(0)
        os.sched_setaffinity(0, nodes[node])
        info["bound"] = True
    return info


def h2d_link_by_numa_node(dev, nbytes=1 << 30, reps=8):
    """Host-to-device copy bandwidth of a 1 GiB pinned buffer allocated while
    this thread runs on each CPU NUMA node in turn (pages are placed on the
    allocating thread's node), best of `reps` cudaMemcpyAsync calls timed with
    CUDA events: shows whether the pinned pools sit on the node attached to
    the GPU and what the link gives from there."""
    import ctypes

    import torch

    from routed_expert_ffn_topk_gb300 import estream as es
    es.lib()                                     # loads the CUDA runtime it links
    rt = ctypes.CDLL("libcudart.so.13")
    rt.cudaHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
    rt.cudaFreeHost.argtypes = [ctypes.c_void_p]
    rt.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                                   ctypes.c_void_p]
    nodes = _numa_cpus()
    gpu_node = _gpu_numa_node(dev.index)
    out = {"gpu_numa_node": gpu_node, "cpu_numa_nodes": sorted(nodes), "by_node": {}}
    if not hasattr(os, "sched_setaffinity") or not nodes:
        return out
    stream = torch.cuda.current_stream(dev)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    orig = os.sched_getaffinity(0)
    try:
        for n, cpus in sorted(nodes.items()):
            os.sched_setaffinity(0, cpus)
            p = ctypes.c_void_p()
            if rt.cudaHostAlloc(ctypes.byref(p), nbytes, 0) != 0 or not p.value:
                continue
            try:
                ctypes.memset(p, 1, nbytes)
                best = None
                for _ in range(reps):
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    rc = rt.cudaMemcpyAsync(dst.data_ptr(), p, nbytes, 1, stream.cuda_stream)
                    b.record(stream)
                    b.synchronize()
                    if rc != 0:
                        break
                    ms = a.elapsed_time(b)
                    best = ms if best is None else min(best, ms)
            finally:
                torch.cuda.synchronize()
                rt.cudaFreeHost(p)
            if best:
                out["by_node"][str(n)] = round(nbytes / (best / 1e3) / 1e9, 1)
    finally:
        os.sched_setaffinity(0, orig)
    return out


def capture_graph(fn):
    """Capture fn() (launches on torch's current stream) into a CUDA graph,
    after two warm runs on the capture side stream."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def measure_router(cfg, X0, dev, stream, flush, peaks, steps):
    """estream_router_logits on the config's X and a seeded W_r [E, H]: CUDA
    events around each call on the launching stream, L2 flushed before each."""
    import torch

    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300 import workloads as W
    _, W_r = W.make_router(1, cfg.H, cfg.E, seed=W.CONFIG_SEEDS[cfg.key] + 500)
    W_r = W_r.to(dev)
    T, H, E = cfg.T, cfg.H, cfg.E
    logits = torch.empty(T, E, dtype=torch.float32, device=dev)
    ws = torch.empty(max(es.router_workspace_bytes(T, H, E), 256), dtype=torch.uint8, device=dev)
    for _ in range(3):
        es.router_logits(X0, W_r, logits=logits, workspace=ws)
    ms = []
    for _ in range(max(steps, 5)):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        es.router_logits(X0, W_r, logits=logits, workspace=ws)
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
    assert es.workspace_error(ws) == es.OK
    t = sorted(ms)[len(ms) // 2]
    nbytes = T * H * 2 + E * H * 2 + T * E * 4
    gbs = nbytes / (t / 1e3) / 1e9

    # routing from the layer input: router logits + top-k + route map, as one
    # fused launch, against the router kernel followed by the route build
    k = cfg.k
    rws = torch.empty(es.route_workspace_bytes(T, E, k, E), dtype=torch.uint8, device=dev)
    out = es.route_build_from_x(X0, W_r, k, cfg.renorm, workspace=rws)

    def timed(fn, n):
        for _ in range(3):
            fn()
        res = []
        for _ in range(n):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            res.append(a.elapsed_time(b))
        return sorted(res)[len(res) // 2]

    t_fused = timed(lambda: es.route_build_from_x(X0, W_r, k, cfg.renorm, out=out, workspace=rws),
                    max(steps, 5))
    assert es.workspace_error(rws) == es.OK
    lg = out["logits"]

    def two():
        es.router_logits(X0, W_r, logits=lg, workspace=ws)
        es.route_build(lg, k, cfg.renorm, out=out, workspace=rws)

    t_two = timed(two, max(steps, 5))
    assert es.workspace_error(rws) == es.OK
    return {"kernel": "k_router_partial (tcgen05, K split over a CTA cluster, fixed-order DSMEM sum)",
            "ms": round(t, 4), "algorithmic_bytes": nbytes, "GBps": round(gbs, 1),
            "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "TFLOPs": round(2.0 * T * H * E / (t / 1e3) / 1e12, 1),
            "workspace_bytes": int(ws.numel()),
            "routing_from_x": {
                "fused_single_launch": es.route_build_from_x_fused(T, H, E),
                "kernel": "k_route_from_x (router tile per cluster, top-k from shared memory, route map)",
                "ms": round(t_fused, 4),
                "two_launches_ms": round(t_two, 4),
                "note": "router logits + top-k + route map (no residual rows); two launches = "
                        "k_router_partial then the route build's memset + k_route_fused"}}


def measure_q4(args, cfg, wl, dev, stream, flush, peaks):
    """The same layer (layer 0) with 4-bit experts (ESTREAM_Q4): resident,
    timed like the main step, with the fused kernel's roofline from the
    packed weight bytes (3*H*F*9/16 per active expert) + X + Y; and paged,
    every group streamed (arena invalidated), through an arena of the config's
    group size G and as many banks as fit in the bytes of the config's bf16
    arena (the paper's fixed memory budget: 4-bit slots are 3.56x smaller)."""
    import torch

    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300 import workloads as W
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl1 = W.Workload(cfg.__class__(**{**cfg.__dict__, "layers": 1}), [wl.logits[0]], wl.X, [wl.layers[0]])
    X = wl.X.to(dev)
    lg = wl.logits[0].to(dev)
    Y = torch.empty(cfg.T, cfg.H, dtype=torch.float32, device=dev)
    out = {"format": "4-bit codes, one scale per 32 weights along the reduction (Q4_0-style)"}
    for mode in ("resident", "paged"):
        # paged: banks free before routing are filled in storage order (the
        # pages' prefetch schedule); with 28 MB groups the route-and-decide
        # time at the start of a call is a larger share than with bf16
        form = {"auto": es.FFN_AUTO, "single": es.FFN_SINGLE, "pair": es.FFN_PAIR}[args.q4_form]
        kw = {}
        if mode == "paged":
            budget = es.arena_bytes(cfg.E, cfg.H, cfg.F, cfg.G, cfg.B, es.BF16)
            bank = es.arena_bytes(cfg.E, cfg.H, cfg.F, cfg.G, 1, es.Q4)
            kw = {"B": max(1, min(-(-cfg.E // cfg.G), budget // bank))}
        st = BoundLayerStack(wl1, mode=mode, wdtype=es.Q4, ffn_form=form,
                             schedule=es.SCHED_PREFETCH if mode == "paged" else es.SCHED_AFTER_ROUTING,
                             **kw)
        arena = f"P={st.G * st.B} (G={st.G}, B={st.B})"
        try:
            def one():
                if mode == "paged":
                    es.arena_invalidate(st.ctx)
                Y.copy_(X)
                st.prefill(0, X, lg, Y)
            for _ in range(3):
                one()
            torch.cuda.synchronize()
            es.reset_stats(st.ctx)
            es.set_timing(st.ctx, True)
            ms = []
            n = max(3, args.steps if mode == "resident" else min(args.steps, args.paged_steps))
            for _ in range(n):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                one()
                b.record(stream)
                b.synchronize()
                ms.append(a.elapsed_time(b))
            stats = es.last_stats(st.ctx)
            es.set_timing(st.ctx, False)
            assert es.get_device_error(st.ctx) == es.OK
        finally:
            st.close()
        t = sum(ms) / len(ms)
        rec = {"ms_per_layer": round(t, 4), "tokens_per_s": round(cfg.T / (t / 1e3), 1)}
        if mode == "resident":
            n_act = active_experts(cfg, [wl.logits[0]])[0]
            ffn_ms = stats["ms_ffn"] / max(1, stats["n_ffn"])
            nbytes = n_act * 3 * cfg.H * cfg.F * 9 // 16 + cfg.T * cfg.H * 2 + 2 * cfg.T * cfg.H * 4
            flops = 6.0 * cfg.H * cfg.F * cfg.T * cfg.k
            gbs = nbytes / (ffn_ms / 1e3) / 1e9
            tfs = flops / (ffn_ms / 1e3) / 1e12
            # the 4-bit weights move 3.56x fewer bytes for the same FLOPs: the
            # roof is the tensor one whenever the intensity is above the ridge
            ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
            sus = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
            tensor = flops / nbytes >= ridge
            # the library's automatic form choice, the same rule as for bf16
            q4_pair = cfg.T * cfg.k >= es.PAIR_MIN_ROWS * cfg.E
            rec.update({"kernel": "k_expert_ffn_pair<4-bit> (CTA pairs)" if q4_pair else "k_expert_ffn_q4",
                        "ffn_ms": round(ffn_ms, 4),
                        "algorithmic_bytes_per_launch": int(nbytes),
                        "algorithmic_flops_per_launch": int(flops),
                        "arithmetic_intensity": round(flops / nbytes, 1),
                        "GBps": round(gbs, 1), "TFLOPs": round(tfs, 1),
                        "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
                        "frac_tensor_sustained": round(tfs / sus, 4),
                        "bound": "tensor" if tensor else "hbm",
                        "frac": round(tfs / sus if tensor else gbs / peaks["hbm_gbs"], 4)})
        else:
            h2d = stats["h2d_bytes"] / len(ms)
            rec.update({"schedule": "prefetch before routing",
                        "arena": arena + ", within the bytes of the bf16 arena",
                        "h2d_bytes_per_layer": int(h2d),
                        "h2d_GBps": round(h2d / (t / 1e3) / 1e9, 1)})
        out[mode] = rec
    return out


def measure_paged(args, cfg, wl, dev, stream, flush, peaks):
    import torch

    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    L = cfg.layers
    st = BoundLayerStack(wl, mode="paged")
    X = wl.X.to(dev)
    logits = [lg.to(dev) for lg in wl.logits]
    Y = torch.zeros(cfg.T, cfg.H, dtype=torch.float32, device=dev)
    steps = max(3, min(args.steps, args.paged_steps))

    def one(l):
        es.arena_invalidate(st.ctx)    # every group really streams
        st.prefill(l, X, logits[l], Y)

    for _ in range(2):
        one(0)
    torch.cuda.synchronize()
    es.reset_stats(st.ctx)
    es.set_timing(st.ctx, True)
    times = []
    for i in range(steps):
        for l in range(L):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            es.arena_invalidate(st.ctx)
            a.record(stream)
            st.prefill(l, X, logits[l], Y)
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
    stats = es.last_stats(st.ctx)
    adsf, t_ne = es.pipeline_trace(st.ctx)       # the last call's groups
    es.set_timing(st.ctx, False)
    st.close()
    t_paged = sum(times) / len(times)
    model = None
    if len(adsf):
        L_k, X_k = adsf[:, 1] - adsf[:, 0], adsf[:, 3] - adsf[:, 2]
        t_model, _ = es.maxplus_pipeline(L_k, X_k, 1, cfg.B, t_ne)
        model = {"eq5_predicted_ms": round(t_model, 4), "measured_ms": round(float(adsf[-1, 3]), 4),
                 "groups": int(len(adsf)), "q": 1, "b": cfg.B, "T_ne_ms": round(t_ne, 4)}
    bytes_per_call = stats["h2d_bytes"] / len(times)

    def time_schedule(B, schedule):
        """The same layers through another schedule of EStream Fig. 6: mean
        ms per layer call, every group streamed."""
        sts = BoundLayerStack(wl, mode="paged", B=B, schedule=schedule)
        try:
            for _ in range(2):
                es.arena_invalidate(sts.ctx)
                sts.prefill(0, X, logits[0], Y)
            torch.cuda.synchronize()
            ts = []
            for i in range(steps):
                for l in range(L):
                    flush.zero_()
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    es.arena_invalidate(sts.ctx)
                    a.record(stream)
                    sts.prefill(l, X, logits[l], Y)
                    b.record(stream)
                    b.synchronize()
                    ts.append(a.elapsed_time(b))
            assert es.get_device_error(sts.ctx) == es.OK
        finally:
            sts.close()
        return sum(ts) / len(ts)

    t_pf = time_schedule(cfg.B, es.SCHED_PREFETCH)     # prefetch before routing
    t_od = time_schedule(1, es.SCHED_AFTER_ROUTING)    # on demand: one bank

    # the same bytes, copy only (host link alone), and the link's own peak
    pool = st.pools[0]
    dst = torch.empty(int(bytes_per_call) if bytes_per_call else 1, dtype=torch.uint8, device=dev)
    src = pool[: dst.numel()]
    for _ in range(2):
        dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    io = []
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src, non_blocking=True)
        b.record(stream)
        b.synchronize()
        io.append(a.elapsed_time(b))
    t_io = min(io)
    big = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    bigd = torch.empty(1 << 30, dtype=torch.uint8, device=dev)
    best = None
    for _ in range(10):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        bigd.copy_(big, non_blocking=True)
        b.record(stream)
        b.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    h2d_peak = (1 << 30) / (best / 1e3) / 1e9
    del big, bigd, dst
    t_exec = (stats["ms_route"] + stats["ms_ffn"] + stats["ms_shared"]) / len(times)
    h2d_gbs = bytes_per_call / (t_paged / 1e3) / 1e9
    return {
        "arena": f"P={cfg.P} (G={cfg.G}, B={cfg.B})", "schedule": "after routing",
        "tokens_per_s": round(cfg.T / (t_paged / 1e3), 1),
        "prefetch_before_routing": {"ms_per_layer": round(t_pf, 4),
                                    "tokens_per_s": round(cfg.T / (t_pf / 1e3), 1),
                                    "bubble_rate": round(1 - max(t_io, t_exec) / t_pf, 4)},
        "on_demand": {"arena": f"P={cfg.G} (G={cfg.G}, B=1)", "ms_per_layer": round(t_od, 4),
                      "tokens_per_s": round(cfg.T / (t_od / 1e3), 1),
                      "bubble_rate": round(1 - max(t_io, t_exec) / t_od, 4)},
        "ms_per_layer": round(t_paged, 4), "h2d_bytes_per_layer": int(bytes_per_call),
        "h2d_GBps": round(h2d_gbs, 1), "h2d_peak_GBps": round(h2d_peak, 1),
        "frac_h2d_peak": round(h2d_gbs / h2d_peak, 4),
        "t_io_alone_ms": round(t_io, 4), "t_exec_ms": round(t_exec, 4),
        "hidden_fraction": round((t_io + t_exec - t_paged) / t_io, 4) if t_io > 0 else None,
        "compute_hidden_fraction": round((t_io + t_exec - t_paged) / t_exec, 4) if t_exec > 0 else None,
        "bubble_rate": round(1 - max(t_io, t_exec) / t_paged, 4),
        "library_stats_overlap": {"hidden_fraction": round(stats["hidden_fraction"], 4),
                                  "bubble_rate": round(stats["bubble_rate"], 4),
                                  "from": "estream_last_stats over the timed calls (copy-stream "
                                          "busy time vs execution and call time)"},
        "groups_loaded_per_layer": stats["groups_loaded"] / len(times),
        "groups_skipped_per_layer": stats["groups_skipped"] / len(times),
        "max_plus_model": model,
    }


def pipeline_study(cfg, wl, dev, flush, reps=5):
    """Section 3.4 on this GPU: the three loading schedules of Fig. 6
    (on-demand = one bank, after routing, prefetch before routing) with their
    bubble rates, and the auto-configurator of Eqs. 8-10 profiled with one
    call per candidate group size and checked against a measured sweep of
    (G, B) under the same memory budget (the Fig. 10 analogue)."""
    import torch

    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    stream = torch.cuda.current_stream()
    X = wl.X.to(dev)
    lg = wl.logits[0].to(dev)
    Y = torch.zeros(cfg.T, cfg.H, dtype=torch.float32, device=dev)
    W_e = cfg.expert_bytes()

    def timed(st, n):
        ms, last = [], None
        for _ in range(n):
            flush.zero_()
            es.arena_invalidate(st.ctx)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            st.prefill(0, X, lg, Y)
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return sorted(ms)[len(ms) // 2]

    def profile(G, B, sched=es.SCHED_AFTER_ROUTING):
        st = BoundLayerStack(wl, mode="paged", G=G, B=B, schedule=sched)
        try:
            timed(st, 2)
            es.set_timing(st.ctx, True)
            t = timed(st, reps)
            adsf, t_ne = es.pipeline_trace(st.ctx)
            es.set_timing(st.ctx, False)
        finally:
            st.close()
        return t, adsf, t_ne

    out = {"schedules": {}, "autoconfig": {}}
    t_io = None
    for name, B, sched in (("on_demand", 1, es.SCHED_AFTER_ROUTING),
                           ("after_routing", cfg.B, es.SCHED_AFTER_ROUTING),
                           ("prefetch_before_routing", cfg.B, es.SCHED_PREFETCH)):
        t, adsf, t_ne = profile(cfg.G, B, sched)
        io = float((adsf[:, 1] - adsf[:, 0]).sum()) if len(adsf) else 0.0
        ex = float((adsf[:, 3] - adsf[:, 2]).sum()) if len(adsf) else 0.0
        out["schedules"][name] = {"G": cfg.G, "B": B, "ms": round(t, 4),
                                  "bubble_rate": round(1 - max(io, ex) / t, 4)}
    budget = cfg.P * W_e                      # the config's arena budget
    profiles, measured = {}, {}
    for g in (1, 2, 4, 8, 16):
        if g > cfg.E:
            continue
        t, adsf, t_ne = profile(g, 2 if budget >= 2 * g * W_e else 1)
        profiles[g] = (adsf[:, 1] - adsf[:, 0], adsf[:, 3] - adsf[:, 2])
        bmax = es.bank_bound(g, budget, 0.0, W_e, cfg.E)
        for b in range(1, min(bmax, 4) + 1):
            tm, _, _ = profile(g, b)
            measured[(g, b)] = tm
    G, B, T = es.autoconfig(profiles, t_ne, 1, budget, W_e, cfg.E)
    best = min(measured, key=measured.get)
    out["autoconfig"] = {"budget_bytes": budget, "chosen": [G, B], "predicted_ms": round(T, 4),
                         "chosen_measured_ms": round(measured.get((G, B), float("nan")), 4),
                         "sweep_best": list(best), "sweep_best_ms": round(measured[best], 4),
                         "regret": round(measured.get((G, B), float("nan")) / measured[best] - 1, 4),
                         "sweep": {f"G{g}_B{b}": round(v, 4) for (g, b), v in sorted(measured.items())}}
    return out


def layer_granular_study(cfg, wl, dev, flush, reps=3):
    """Section 4 (layer-granular baselines): a whole L-layer step streamed
    through the config's group-granular arena (P = B*G slots reused across
    layers), against banks that each hold one whole layer (G = E) with two
    banks (Layer-B=2) or L banks (Layer-B=L, every layer's experts held at
    once). Every step starts from an empty arena, so each layer's experts
    stream once; reported: ms per step and arena bytes."""
    import torch

    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    stream = torch.cuda.current_stream()
    L = cfg.layers
    X0 = wl.X.to(dev)
    logits = [lg.to(dev) for lg in wl.logits]
    out = {}
    variants = (("group_granular", cfg.G, cfg.B, es.SCHED_AFTER_ROUTING),
                ("group_granular_prefetch", cfg.G, cfg.B, es.SCHED_PREFETCH),
                ("layer_B2", cfg.E, 2, es.SCHED_PREFETCH),
                ("layer_BL", cfg.E, L, es.SCHED_PREFETCH))
    for name, G, B, sched in variants:
        st = BoundLayerStack(wl, mode="paged", G=G, B=B, schedule=sched)
        try:
            def step():
                es.arena_invalidate(st.ctx)
                X = X0
                for l in range(L):
                    Y = X.float()
                    st.prefill(l, X, logits[l], Y)
                    if l + 1 < L:
                        Xn = torch.empty_like(X)
                        es.cast_f32_bf16(Y, Xn)
                        X = Xn
            step()
            torch.cuda.synchronize()
            ms = []
            for _ in range(reps):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                step()
                b.record(stream)
                b.synchronize()
                ms.append(a.elapsed_time(b))
            assert es.get_device_error(st.ctx) == es.OK
        finally:
            arena = st.arena.numel()
            st.close()
        out[name] = {"G": G, "B": B, "schedule": "prefetch" if sched == es.SCHED_PREFETCH else "after_routing",
                     "arena_bytes": int(arena), "ms_per_step": round(sorted(ms)[len(ms) // 2], 4)}
    return out


# --------------------------------------------------------------------------
# reference arm: the CPU oracle
# --------------------------------------------------------------------------

def workload_config(cfg, world, mode="resident"):
    L = cfg.layers
    return {"workload": f"{cfg.key} {cfg.name}: T={cfg.T} H={cfg.H} E={cfg.E} k={cfg.k} "
                        f"F={cfg.F}" + (f" shared={cfg.n_shared}x{cfg.F_shared}" if cfg.n_shared else "")
                        + (f" layers={L}" if L > 1 else "") + f", experts {mode}",
            "tokens_per_step_per_gpu": cfg.T, "l2": "flushed (256 MiB write) before every step",
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    from routed_expert_ffn_topk_gb300 import workloads as W
    cfg = W.CONFIGS[args.config]
    if rank != 0:
        return None
    wl = W.make_workload(cfg)
    target = max(2.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    rates = []
    for i in range(args.warmup + args.steps):
        tps, n, dt, cores = oracle_tokens_per_s(cfg, wl, target_s=target)
        if i >= args.warmup:
            rates.append((tps, n, dt))
    tps = sum(r[0] for r in rates) / len(rates)
    n = rates[-1][1]
    ms = 1e3 * cfg.T / tps
    return {"impl": "reference", "metric": METRIC, "value": round(tps, 3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
            "config": workload_config(cfg, world),
            "cpu_baseline": {"value": round(tps, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"routing of all {cfg.T} tokens + Eq.2 for {n} sampled tokens per step"},
            "e2e": {"value": round(tps, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="c5", choices=["c1", "c2", "c3", "c4", "c5"],
                    help="the headline workload (default: the Mixtral-shaped layer)")
    ap.add_argument("--configs", default="c2,c3,c4,c5",
                    help="workloads measured the same way under \"configs\"")
    ap.add_argument("--no-configs", action="store_true", help="measure the headline workload only")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--paged-steps", type=int, default=10)
    ap.add_argument("--no-paged", action="store_true")
    ap.add_argument("--no-q4", action="store_true", help="skip the 4-bit-expert measurement")
    ap.add_argument("--no-router", action="store_true", help="skip the router-logits measurement")
    ap.add_argument("--no-graph", action="store_true", help="time eager launches, not a CUDA-graph replay")
    ap.add_argument("--q4-form", default="auto", choices=["auto", "single", "pair"],
                    help="form of the 4-bit fused expert kernel (default: the library's choice)")
    ap.add_argument("--ffn-form", default="auto", choices=["auto", "single", "pair"],
                    help="form of the fused expert kernel in the resident step (default: the library's choice)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pipeline-study", action="store_true",
                    help="also measure the loading schedules and the (G, B) auto-configuration")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    bad = [k for k in args.configs.split(",") if k not in W.CONFIGS]
    if bad:
        ap.error(f"unknown configs {bad}")
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return 0
        else:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, rank, 1)
        print(json.dumps(line))
        return 0
    line = run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
