#!/usr/bin/env python
"""Benchmark of the fused-dequantization linear layer on one GB300 (or N
replicas under torchrun).

Headline (``value``): decode qGEMV weight throughput at M = 1 over the
70B-shaped stack -- 80 layers x (q, k, v, o, gate, up, down), INT4 group 128
with 0.1 % FP16 outliers, 36 GB of quantized weights resident in HBM.  One
token = the 560 products of the stack (q/k/v and gate/up as fused calls: 320
launches), captured once in a CUDA graph; a step is ``tokens_per_step``
consecutive tokens (graph replays), chosen so that the timed region lasts at
least two seconds.  The unit is GB/s of packed-weight bytes (codes only); the
all-bytes figure (codes + scales + zero-points + outlier CSR + x + y) is the
roofline's ``achieved``.

Secondary objects in the same JSON line, each with the clock record of its
own timed region: the same stack at M = 16 and 64; prefill qGEMM TFLOP/s at
M = 2048 on one layer of the stack and on 11008 x 4096 products at widths
2/3/4/5/6; the MoE layer (16 experts, 256 tokens, top-2 Zipf routing); the
single 4096 x 4096 INT4 layer and the mixed-width sweep (2/3/5/6 bits,
groups 64/128) at M = 1, 8, 32; the 7B-shaped mixed-width stack at M = 1, 8,
32; the device quantizer; and two CPU figures: the oracle (``cpu_baseline``)
and the fused multi-threaded CPU qGEMV (``cpu_fused_baseline``).

``--impl reference`` times the CPU oracle (plain C, fp64) on the host cores
on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "qGEMV weight GB/s (% of HBM peak) at M=1; qGEMM TFLOP/s at M=2048"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--layers", type=int, default=80, help="layers of the 70B-shaped stack")
    ap.add_argument("--no-secondary", action="store_true", help="skip the prefill and MoE lines")
    ap.add_argument("--mode", choices=("all", "decode", "prefill", "moe", "widths", "variants", "case"), default="all",
                    help="run only that measurement and print its object (profiling runs): 'decode' = the "
                         "headline alone; 'prefill' = the 70B layer and the width sweep at M=2048; 'widths' = "
                         "the single layer, the mixed-width sweep and the 7B-shaped stack at M=1, 8, 32")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-oracle sample")
    ap.add_argument("--case", default="gateup1",
                    help="--mode case: one small case, three calls, for a profiler: gateup<M> (fused 28672x8192 "
                         "gate/up decode at M), decode<bits>g<group> (11008x4096 at M=1), tiles<bits>[m<M>] / planar<bits>[m<M>] "
                         "(8192x8192 at M=2048 or M), moe (gate/up of "
                         "the MoE layer), w8a8 (28672x8192 at M=1), diag / repack (28672x8192 INT4)")
    return ap.parse_args()


# DRAM bytes (read + written) per 70B-shaped layer of the decode step, from one
# ncu capture (dram__bytes_read.sum + dram__bytes_write.sum over the launches
# of a layer, captured on a 2-layer stack), valid only for the kernel source
# it was taken on.
DECODE_TRAFFIC = {"kernel_sha256": "00273f39ac9c098db419e953c18c78228479fd93816f5a6eb2d8d6bafcfd8424",
                  "bytes_per_layer": 454.925e6}


def decode_traffic(n_layers):
    src = os.path.join(ROOT, "bit_weight_only_group_gb300", "csrc", "gemv_impl.cuh")
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != DECODE_TRAFFIC["kernel_sha256"]:
            return None
    return DECODE_TRAFFIC["bytes_per_layer"] * n_layers


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d.get("hbm_gbs", 6800.0), bf16=d.get("bf16_tflops", 1900.0),
                    bf16_sust=d.get("bf16_tflops_sustained", 1700.0), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


# ---------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class Clocks:
    """nvidia-smi sampled every 200 ms for the whole run; each timed region
    reads the samples whose timestamp falls inside it (window)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.rows = None
        try:
            self.dev = "GPU-" + str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        except Exception:
            self.dev = str(torch.cuda.current_device())

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", self.dev], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        import datetime
        rows = []
        self.fh.flush()
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm = float(f[1])
            except ValueError:
                continue
            rows.append((ts, sm, f))
        return rows

    def window(self, t0: float, t1: float):
        """Clock record of the timed region [t0, t1] (wall-clock seconds)."""
        if self.proc is None:
            return None
        time.sleep(0.25)   # the sample that closes the region
        rows = [(sm, f) for ts, sm, f in self._read() if t0 <= ts <= t1]
        if not rows:
            return {"sm_mhz": None, "samples": 0, "reasons": [], "note": "no nvidia-smi sample inside the timed region"}
        reasons = set()
        for _, f in rows:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        pw = [float(f[3]) for _, f in rows if f[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm for sm, _ in rows), "sm_max_mhz": float(rows[0][1][2]),
                "samples": len(rows), "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons)}

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        os.unlink(self.path)
        self.proc = None


CLK = None   # the run's sampler (rank 0 of each process: every process samples its own GPU)


def region_clocks(t0, t1):
    return CLK.window(t0, t1) if CLK is not None else None


# ---------------------------------------------------------------- our arm
def build_stack(qg, layers, device):
    """Quantize every matrix of the stack on the device from seeded fp16 W."""
    ws_bytes = max(qg.qpack_workspace_size(L.N, L.K) for L in layers)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    qws = []
    for i, L in enumerate(layers):
        W = wl.gen_weight(L.N, L.K, seed=wl.SEED_W + i, outlier_frac=L.frac, outlier_seed=wl.SEED_OUTLIER + i,
                          device=device, distinct_positions=False)
        qws.append(qg.qpack_quantize(W, L.bits, L.group, L.frac, workspace=ws))
        del W
    torch.cuda.synchronize()
    return qws


def layer_bytes(qg, L, M):
    s = qg.qpack_query_sizes(L.N, L.K, L.bits, L.group, L.frac)
    packed = s["packed"]
    rest = s["scale"] + s["zp"] + s["codebook"] + (L.N + 1) * 4 + s["nnz"] * 6
    io = M * L.K * 2 + M * L.N * 4
    return packed, packed + rest + io


def decode_config(n_layers, world):
    """The headline workload's config object (both arms report this one)."""
    weights = 0
    for L in wl.stack_70b(n_layers):
        ng = L.K // L.group
        nnz = int(L.frac * L.N * L.K)
        weights += L.N * L.K * L.bits // 8 + L.N * ng * 3 + (L.N + 1) * 4 + nnz * 6
    return {"workload": f"70B-shaped stack decode: {n_layers} layers x q/k/v/o/gate/up/down, INT4 group 128, "
                        "0.1% FP16 outliers, M=1, y fp32",
            "layers": n_layers, "M": 1, "weights_GB_per_gpu": round(weights / 1e9, 3),
            "l2": "inputs larger than L2 (weights per step far above 129 MB)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def check_graph_covers(g, ys, what):
    """Replay the captured step once over outputs filled with NaN: every
    product must have written its output, or work escaped the capture."""
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    missing = [i for i, y in enumerate(ys) if not torch.isfinite(y).all()]
    if missing:
        raise RuntimeError(f"{what}: the captured step did not compute products {missing[:10]}")


def capture(step):
    """Run step once eagerly (lazy loading outside capture), then capture it."""
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    torch.cuda.synchronize()
    return g


def time_replays(g, n, warmup=3, world=1, flush=None):
    """Device time (ms) of n replays of g on the current stream, bracketed by
    a barrier and a synchronize on both sides, and the wall-clock window of
    the timed region.  flush: a buffer larger than L2, rewritten before each
    replay (inside the timed region: its time is measured separately and
    subtracted by the caller)."""
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record(s)
    for _ in range(n):
        if flush is not None:
            flush.fill_(1.0)
        g.replay()
    e1.record(s)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    return e0.elapsed_time(e1), (t0, t1)


def reps_for(g, seconds, cap=100000):
    """Replays of g that take about `seconds` (one timed probe of 3 replays)."""
    ms, _ = time_replays(g, 3, warmup=1)
    return int(max(3, min(cap, math.ceil(seconds * 1e3 / max(ms / 3, 1e-3)))))


def timed_object(g, seconds=0.5, flush=None):
    """(ms per replay, replays, clock record) of a secondary measurement whose
    timed region lasts about `seconds`."""
    n = reps_for(g, seconds)
    ms, (t0, t1) = time_replays(g, n, flush=flush)
    return ms / n, n, region_clocks(t0, t1)


def decode_stack_step(qg, layers, qws, xs, ys):
    """One token (or M tokens) through the stack on one stream: the fused
    q/k/v projection (one call, one launch), o, the fused gate/up projection,
    down -- four decode launches per layer; consecutive launches overlap
    through programmatic dependent launch."""
    def step():
        for li in range(0, len(layers), 7):
            qg.qgemm_forward_multi(xs[li], qws[li:li + 3], outs=ys[li:li + 3])
            qg.qgemm_forward(xs[li + 3], qws[li + 3], out=ys[li + 3])
            qg.qgemm_forward_multi(xs[li + 4], qws[li + 4:li + 6], outs=ys[li + 4:li + 6])
            qg.qgemm_forward(xs[li + 6], qws[li + 6], out=ys[li + 6])
    return step


def stack_inputs(layers, M, dev, seed_off=0):
    x_hid = wl.gen_x(M, 8192, seed=wl.SEED_X + seed_off, device=dev)
    x_ffn = wl.gen_x(M, 28672, seed=wl.SEED_X + 1 + seed_off, device=dev)
    xs = [x_ffn if L.K == 28672 else x_hid for L in layers]
    ys = [torch.empty((M, L.N), dtype=torch.float32, device=dev) for L in layers]
    return x_hid, x_ffn, xs, ys


def run_decode(qg, args, world, rank, P):
    layers = wl.stack_70b(args.layers)
    dev = torch.device("cuda")
    t0 = time.time()
    qws = build_stack(qg, layers, dev)
    setup_s = time.time() - t0
    M = 1
    x_hid, x_ffn, xs, ys = stack_inputs(layers, M, dev)
    g = capture(decode_stack_step(qg, layers, qws, xs, ys))
    check_graph_covers(g, ys, "decode step")

    # tokens per step: enough that the timed region (steps x tokens) lasts >= 2 s
    tok_ms, _ = time_replays(g, 3, warmup=2)
    tok_ms /= 3
    R = max(1, math.ceil(2000.0 / (args.steps * tok_ms)))
    R = int(max_over_ranks(float(R), world))
    ms, (c0, c1) = time_replays(g, args.steps * R, warmup=args.warmup * R, world=world)
    clocks = region_clocks(c0, c1)
    ms_max = max_over_ranks(ms, world)
    packed = sum(layer_bytes(qg, L, M)[0] for L in layers)
    allb = sum(layer_bytes(qg, L, M)[1] for L in layers)
    per_token_s = ms_max / 1e3 / (args.steps * R)
    value = sum_over_ranks(packed, world) / per_token_s / 1e9

    # end to end: per token, pinned host x -> device, the captured token, y -> host
    xh_pin = x_hid.cpu().pin_memory()
    xf_pin = x_ffn.cpu().pin_memory()
    y_pin = torch.empty_like(ys[-1], device="cpu").pin_memory()
    s = torch.cuda.current_stream()

    def e2e_token():
        x_hid.copy_(xh_pin, non_blocking=True)
        x_ffn.copy_(xf_pin, non_blocking=True)
        g.replay()
        y_pin.copy_(ys[-1], non_blocking=True)
    for _ in range(args.warmup * R):
        e2e_token()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(args.steps * R):
        e2e_token()
    e1.record(s)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e = {"value": sum_over_ranks(packed, world) / (e2e_ms / 1e3 / (args.steps * R)) / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": R * (xh_pin.numel() * 2 + xf_pin.numel() * 2),
           "d2h_bytes_per_step": R * y_pin.numel() * 4,
           "note": f"per token: x copied from pinned host memory, the token's 320 C-ABI calls (captured once in "
                   f"a CUDA graph on one stream), y read back; {R} tokens per step"}

    achieved = allb / per_token_s / 1e9
    traffic = decode_traffic(len(layers) // 7)
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": P["hbm"], "unit": "GB/s",
            "frac": round(achieved / P["hbm"], 4), "traffic": None if traffic is None else traffic * R,
            "traffic_unit": "bytes per step (R tokens; the achieved figure is per step as well: every launch "
                            "of the step is this kernel)",
            "kernel": "k_gemv<4,128,1> / k_gemv_multi<4,128,1> (decode qGEMV, the only kernel of the step)",
            "peak_source": P["src"] + " hbm_gbs"}
    out = dict(value=value, ms_per_step=ms_max / args.steps, tokens_per_step=R, ms_per_token=ms_max / (args.steps * R),
               roofline=roof, e2e=e2e, clocks=clocks, gpu_launches=(len(layers) // 7) * 4 * args.steps * R,
               setup_s=round(setup_s, 1), weights_GB=round(sum(q.nbytes() for q in qws) / 1e9, 3),
               all_bytes_GBps=round(achieved, 1), frac_of_nominal_8TBs=round(value / 8000.0, 4),
               bytes_per_token=allb, packed_bytes_per_token=packed)
    del g
    return out, qws


def run_decode_m(qg, qws, layers, M, P):
    """The 70B-shaped stack at M tokens per product (the decode configs at
    M = 16 and 64): weights already resident, one graph of the 320 launches."""
    dev = torch.device("cuda")
    _, _, xs, ys = stack_inputs(layers, M, dev, seed_off=10 + M)
    g = capture(decode_stack_step(qg, layers, qws, xs, ys))
    check_graph_covers(g, ys, f"decode step M={M}")
    ms, n, clocks = timed_object(g, 0.6)
    packed = sum(layer_bytes(qg, L, M)[0] for L in layers)
    allb = sum(layer_bytes(qg, L, M)[1] for L in layers)
    del g
    return {"metric": f"decode qGEMV weight GB/s at M={M}", "value": round(packed / ms / 1e6, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "all_GBps": round(allb / ms / 1e6, 1),
            "frac_of_hbm_peak": round(allb / ms / 1e6 / P["hbm"], 4), "replays": n, "clocks": clocks,
            "config": f"70B-shaped stack, {len(layers) // 7} layers, INT4 g128, 0.1% outliers, M={M}; 320 launches "
                      "per step (fused q/k/v, o, fused gate/up, down)"}


def run_prefill(qg, args, P):
    """One layer of the 70B stack at M = 2048 (7 products), TFLOP/s."""
    layers = wl.stack_70b(1)
    dev = torch.device("cuda")
    qws = build_stack(qg, layers, dev)
    M = wl.STACK_70B_PREFILL_M
    x_hid, x_ffn, xs, ys = stack_inputs(layers, M, dev)
    wsb = max(qg.qgemm_workspace_size(M, q) for q in qws)
    # one workspace per concurrent product (each holds its fp16 copy of x)
    wss = [torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev) for _ in range(3)]
    side = [torch.cuda.Stream(), torch.cuda.Stream()]

    run = lambda j, w, s=None: qg.qgemm_forward(xs[j], qws[j], out=ys[j], workspace=w, stream=s)

    def step():
        # the layer's dependency structure, as in the decode step: {q, k, v} -> o -> {gate, up} -> down,
        # products that share an input as parallel graph branches (fork and join on the stream current
        # at call time, the capture stream under graph capture)
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        done = []
        for sj, j, w in zip(side, (1, 2), wss[1:]):
            sj.wait_event(fork)
            with torch.cuda.stream(sj):
                run(j, w, sj)
                e = torch.cuda.Event()
                e.record(sj)
                done.append(e)
        run(0, wss[0])
        for e in done:
            main.wait_event(e)
        run(3, wss[0])
        fork = torch.cuda.Event()
        fork.record(main)
        side[0].wait_event(fork)
        with torch.cuda.stream(side[0]):
            run(5, wss[1], side[0])
            e = torch.cuda.Event()
            e.record(side[0])
        run(4, wss[0])
        main.wait_event(e)
        run(6, wss[0])

    g = capture(step)
    check_graph_covers(g, ys, "prefill step")
    ms, n, clocks = timed_object(g, 0.6)
    flops = sum(2.0 * M * L.N * L.K for L in layers)
    tflops = flops / (ms / 1e3) / 1e12
    # the same layer from the tile-ordered copies (repacked once, outside the timed region)
    tiles = [qg.qrepack_tiles(q) for q in qws]
    run = lambda j, w, s=None: qg.qgemm_forward_tiles(xs[j], qws[j], tiles[j], out=ys[j], workspace=w, stream=s)
    gt = capture(step)
    check_graph_covers(gt, ys, "prefill step (tile-ordered)")
    mst, nt, clocks_t = timed_object(gt, 0.6)
    tflops_t = flops / (mst / 1e3) / 1e12
    del qws, g, gt, tiles
    torch.cuda.empty_cache()
    return {"metric": "qGEMM TFLOP/s at M=2048", "value": round(tflops_t, 1), "unit": "TFLOP/s",
            "ms_per_step": round(mst, 4), "replays": nt, "clocks": clocks_t,
            "config": "one 70B-shaped layer (7 products; q/k/v and gate/up as parallel graph branches), INT4 g128, "
                      "0.1% outliers, M=2048; weights in the tile-ordered copy (qrepack_tiles once, at load; "
                      "qgemm_forward_tiles per product)",
            "frac_of_bf16_peak": round(tflops_t / P["bf16"], 4),
            "frac_of_bf16_sustained": round(tflops_t / P["bf16_sust"], 4),
            "planar": {"value": round(tflops, 1), "frac_of_bf16_peak": round(tflops / P["bf16"], 4),
                       "ms_per_step": round(ms, 4), "replays": n, "clocks": clocks,
                       "config": "the same layer from the planar layout (qgemm_forward per product)"},
            # the layer's products run back to back for the whole timed region
            # (power cap active): the sustained measured peak is the denominator
            "roofline": {"bound": "tensor", "achieved": round(tflops_t, 1), "peak": P["bf16_sust"], "unit": "TFLOP/s",
                         "frac": round(tflops_t / P["bf16_sust"], 4), "traffic": None,
                         "kernel": "k_gemm_tc<4,128,tiles> (tcgen05, TMEM accumulators)",
                         "peak_source": P["src"] + " bf16_tflops_sustained (kernels timed inside a long step; "
                                        "fp16 and bf16 share the tensor rate)"}}


def run_prefill_widths(qg, P):
    """11008 x 4096 products at M = 2048 for every width (group 128, 0.1 %
    outliers): the tensor-core kernel, TFLOP/s."""
    dev = torch.device("cuda")
    M, N, K = wl.STACK_70B_PREFILL_M, 11008, 4096
    W = wl.gen_weight(N, K, outlier_frac=0.001, device=dev, distinct_positions=False)
    x = wl.gen_x(M, K, device=dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    out = {}
    t_all0 = time.time()
    for bits in (2, 3, 4, 5, 6, 8):
        q = qg.qpack_quantize(W, bits, 128, 0.001)
        ws = torch.empty(qg.qgemm_workspace_size(M, q), dtype=torch.uint8, device=dev)
        g = capture(lambda: qg.qgemm_forward(x, q, out=y, workspace=ws))
        ms, n, clocks = timed_object(g, 0.4)
        tf = 2.0 * M * N * K / (ms / 1e3) / 1e12
        # the same product from the tile-ordered copy (one-time repack, timed once)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t = qg.qrepack_tiles(q)
        e0.record()
        qg.qrepack_tiles(q, out=t)
        e1.record()
        torch.cuda.synchronize()
        rp_us = e0.elapsed_time(e1) * 1e3
        gt = capture(lambda: qg.qgemm_forward_tiles(x, q, t, out=y, workspace=ws))
        mst, nt, clocks_t = timed_object(gt, 0.4)
        tft = 2.0 * M * N * K / (mst / 1e3) / 1e12
        out[f"w{bits}"] = {"TFLOP_s": round(tf, 1), "frac_of_bf16_peak": round(tf / P["bf16"], 4),
                           "us": round(ms * 1e3, 1), "replays": n, "clocks": clocks,
                           "tiles_TFLOP_s": round(tft, 1), "tiles_frac_of_bf16_peak": round(tft / P["bf16"], 4),
                           "tiles_us": round(mst * 1e3, 1), "tiles_clocks": clocks_t, "repack_us": round(rp_us, 1)}
        del g, gt, q, ws, t
    del W
    torch.cuda.empty_cache()
    return {"metric": "qGEMM TFLOP/s at M=2048 by width", "unit": "TFLOP/s", "by_width": out,
            "config": "W 11008x4096 ~N(0,0.02) + 0.1% outliers, group 128, x bf16 [2048, 4096], y fp32; "
                      "one product per replay (k_x_to_f16 + k_gemm_tc<bits,128,planar>); tiles_*: the same product "
                      "from the tile-ordered copy (k_gemm_tc<bits,128,tiles>), repack_us: the one-time repack",
            "seconds": round(time.time() - t_all0, 1)}


def run_moe(qg, args):
    cfg = wl.MoE()
    dev = torch.device("cuda")
    projs = cfg.projections()
    experts = {}
    for pi, (name, N, K) in enumerate(projs):
        lay = [wl.Linear(f"{name}{e}", N, K, cfg.bits, cfg.group, cfg.frac) for e in range(cfg.n_experts)]
        qs = []
        for e, L in enumerate(lay):
            W = wl.gen_weight(N, K, seed=wl.SEED_W + 1000 * pi + e, device=dev)
            qs.append(qg.qpack_quantize(W, L.bits, L.group, L.frac))
        experts[name] = qs
    x = wl.gen_x(cfg.tokens, cfg.hidden, device=dev)
    xd = wl.gen_x(cfg.tokens, cfg.ffn, seed=wl.SEED_X + 2, device=dev)
    topk = wl.gen_topk(cfg.tokens, cfg.top_k, cfg.n_experts).to(dev)
    ys = {n: torch.empty((cfg.tokens, cfg.top_k, N), dtype=torch.float32, device=dev) for n, N, _ in projs}
    wsb = max(qg.qgemm_moe_workspace_size(cfg.tokens, cfg.top_k, experts[n]) for n, _, _ in projs)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)

    def step():
        # gate and up read the same routed x: one call over one routing; down alone
        qg.qgemm_moe_grouped_multi(x, topk, [experts["gate"], experts["up"]], outs=[ys["gate"], ys["up"]],
                                   workspace=ws)
        qg.qgemm_moe_grouped(xd, topk, experts["down"], out=ys["down"], workspace=ws)

    g = capture(step)
    check_graph_covers(g, list(ys.values()), "MoE step")
    # the layer's weights fit in L2: a buffer larger than L2 is rewritten before
    # each replay; its own time (measured alone) is subtracted
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    gf = capture(lambda: flush.fill_(1.0))
    n = reps_for(g, 0.5, cap=2000)
    ms_both, (t0, t1) = time_replays(g, n, flush=flush)
    ms_flush, _ = time_replays(gf, n)
    ms = (ms_both - ms_flush) / n
    clocks = region_clocks(t0, t1)
    touched = torch.unique(topk).numel()
    used = sorted(set(topk.flatten().tolist()))
    wbytes = sum(experts[n_][e].nbytes() for n_, _, _ in projs for e in used)
    flops = sum(2.0 * cfg.tokens * cfg.top_k * N * K for _, N, K in projs)
    return {"metric": "MoE grouped qGEMM", "value": round(wbytes / (ms / 1e3) / 1e9, 1), "unit": "GB/s",
            "tflops": round(flops / (ms / 1e3) / 1e12, 2), "ms_per_step": round(ms, 4), "experts_touched": touched,
            "replays": n, "clocks": clocks,
            "config": "16 experts gate/up 3072x4096 + down 4096x3072, INT4 g128, 256 tokens top-2 Zipf(1.1); "
                      "gate and up in one call over one routing",
            "l2": "a 512 MB buffer rewritten before each replay (L2 flushed); its time, measured alone, subtracted"}


def weight_copies(qg, q, min_bytes=600e6):
    """q and clones of it, together larger than L2 several times over."""
    copies = max(4, int(math.ceil(min_bytes / q.nbytes())))
    fields = {f.name: getattr(q, f.name) for f in dataclasses.fields(q)}
    clone = lambda: qg.QWeight(**{k: v.clone() if torch.is_tensor(v) else v for k, v in fields.items()})
    return [q] + [clone() for _ in range(copies - 1)]


def layer_rate(qg, cs, M, P, seconds=0.15):
    """One decode product per copy in one graph (the copies exceed L2)."""
    dev = torch.device("cuda")
    q = cs[0]
    x = wl.gen_x(M, q.K, seed=wl.SEED_X + M, device=dev)
    y = torch.empty((M, q.N), device=dev)
    g = capture(lambda: [qg.qgemm_forward(x, c, out=y) for c in cs])
    ms, n, clocks = timed_object(g, seconds)
    us = ms * 1e3 / len(cs)
    packed = q.N * q.K * q.bits // 8
    allb = q.nbytes() + M * q.K * 2 + M * q.N * 4
    del g
    return {"M": M, "us": round(us, 2), "packed_GBps": round(packed / us / 1e3, 1),
            "all_GBps": round(allb / us / 1e3, 1), "frac_of_hbm_peak": round(allb / us / 1e3 / P["hbm"], 4),
            "clocks": clocks}


def run_single_layer(qg, P):
    """The single 4096 x 4096 INT4 group-128 layer at M = 1 (no outliers): one
    product per weight copy, 64+ copies in one graph."""
    dev = torch.device("cuda")
    L = wl.single_layer()
    W = wl.gen_weight(L.N, L.K, device=dev)
    q = qg.qpack_quantize(W, L.bits, L.group, L.frac)
    cs = weight_copies(qg, q, min_bytes=64 * q.nbytes())
    r = layer_rate(qg, cs, 1, P, seconds=0.5)
    del cs, q, W
    torch.cuda.empty_cache()
    return {"metric": "decode qGEMV weight GB/s at M=1, single layer", "value": r["packed_GBps"], "unit": "GB/s",
            "us_per_call": r["us"], "all_GBps": r["all_GBps"], "clocks": r["clocks"],
            "roofline": {"bound": "hbm", "achieved": r["all_GBps"], "peak": P["hbm"], "unit": "GB/s",
                         "frac": r["frac_of_hbm_peak"], "traffic": None,
                         "kernel": "k_gemv<4,128,1>", "peak_source": P["src"] + " hbm_gbs"},
            "config": "W 4096x4096 ~N(0,0.02), INT4 g128, no outliers, x bf16 [1,4096], y fp32; 64 weight copies "
                      "(563 MB, above L2) in one graph, one product per copy"}


def run_sweep(qg, P):
    """The mixed-width sweep: 4096x4096 and 11008x4096, widths 2/3/5/6, groups
    64/128, 0.1 % outliers, M = 1, 8, 32; each product over weight copies
    larger than L2."""
    dev = torch.device("cuda")
    rows = []
    t0 = time.time()
    for L in wl.mixed_sweep():
        W = wl.gen_weight(L.N, L.K, outlier_frac=L.frac, device=dev, distinct_positions=False)
        q = qg.qpack_quantize(W, L.bits, L.group, L.frac)
        del W
        cs = weight_copies(qg, q)
        for M in (1, 8, 32):
            r = layer_rate(qg, cs, M, P)
            r["layer"] = L.name
            rows.append(r)
        del cs, q
        torch.cuda.empty_cache()
    return {"metric": "decode qGEMV GB/s over widths 2/3/5/6 at M = 1, 8, 32", "unit": "GB/s", "rows": rows,
            "config": "W 4096x4096 and 11008x4096 ~N(0,0.02) + 0.1% outliers, widths {2 (codebook),3,5,6} x groups "
                      "{64,128}; x bf16 [M, K]; weight copies above 600 MB per graph",
            "seconds": round(time.time() - t0, 1)}


VARIANTS = [  # (name, bits, group, mode, scale format)
    ("b4_g128", 4, 128, "asymmetric", "fp16"),
    ("b4_g128_fp8", 4, 128, "asymmetric", "fp8"),
    ("b3_g32", 3, 32, "asymmetric", "fp16"),
    ("b3_g32_fp8", 3, 32, "asymmetric", "fp8"),
    ("b3_g32_sym_fp8", 3, 32, "symmetric", "fp8"),
    ("b2_g32", 2, 32, "asymmetric", "fp16"),
    ("b2_g128_sym", 2, 128, "symmetric", "fp16"),
    ("b2_g128_linear", 2, 128, "linear2", "fp16"),
]


def run_variants(qg, P):
    """The format variants (group 32, E4M3 scales with the fp16 fallback,
    symmetric and linear 2-bit) on one 11008 x 4096 matrix with 0.1 %
    outliers: decode at M = 1 over weight copies above L2, and the
    tensor-core product at M = 2048 from the tile-ordered copy."""
    dev = torch.device("cuda")
    N, K, frac = 11008, 4096, 0.001
    W = wl.gen_weight(N, K, outlier_frac=frac, device=dev, distinct_positions=False)
    x = wl.gen_x(2048, K, device=dev)
    rows = {}
    for name, bits, group, mode, fmt in VARIANTS:
        q = qg.qpack_quantize(W, bits, group, frac, mode=mode, scale_fmt=fmt)
        cs = weight_copies(qg, q)
        r = layer_rate(qg, cs, 1, P)
        del cs
        t = qg.qrepack_tiles(q)
        y = torch.empty((2048, N), device=dev)
        g = capture(lambda: qg.qgemm_forward_tiles(x, q, t, out=y))
        ms, n, clocks = timed_object(g, 0.15)
        del g, t, y
        r.update(eff_bits=round(q.nbytes() * 8 / (N * K), 3),
                 prefill_TFLOP_s=round(2 * 2048 * N * K / ms / 1e9, 1), prefill_us=round(ms * 1e3, 1),
                 prefill_clocks=clocks)
        if fmt == "fp8":
            r["fallback_groups"] = int(q.fb_row_ptr[-1].item())
        rows[name] = r
        del q
        torch.cuda.empty_cache()
    del W, x
    return {"metric": "format variants: decode GB/s at M=1, tensor-core TFLOP/s at M=2048", "unit": "GB/s",
            "rows": rows,
            "config": "W 11008x4096 ~N(0,0.02) + 0.1% outliers; decode over weight copies above 600 MB per graph "
                      "(packed_GBps = codes only, all_GBps = every byte of the layer); prefill from the tile-ordered "
                      "copy, x bf16 [2048, 4096]"}


def run_quantize(qg, P):
    """The device quantizer (outlier selection, group statistics, codes,
    packing: offline, not on the decode path) on one 28672 x 8192 fp16
    matrix of the 70B stack, INT4 group 128, 0.1 % outliers, into preallocated
    buffers; GB/s of fp16 W read (each call makes five passes over W)."""
    dev = torch.device("cuda")
    N, K, bits, group, frac = 28672, 8192, 4, 128, 0.001
    W = wl.gen_weight(N, K, outlier_frac=frac, device=dev, distinct_positions=False)
    out = qg.QWeight.empty(N, K, bits, group, frac, dev)
    ws = torch.empty(qg.qpack_workspace_size(N, K), dtype=torch.uint8, device=dev)
    g = capture(lambda: qg.qpack_quantize(W, bits, group, frac, out=out, workspace=ws))
    ms, n, clocks = timed_object(g, 0.4)
    wbytes = N * K * 2
    del W, out, ws, g
    torch.cuda.empty_cache()
    return {"metric": "device quantizer (offline)", "value": round(wbytes / ms / 1e6, 1), "unit": "GB/s of fp16 W",
            "ms_per_matrix": round(ms, 4), "passes_over_W": 5, "replays": n, "clocks": clocks,
            "config": "28672x8192 fp16 W, INT4 group 128, 0.1% outliers, outputs and workspace preallocated"}


def build_stack7b(qg):
    dev = torch.device("cuda")
    layers = wl.stack_7b()
    qs = []
    for i, L in enumerate(layers):
        W = wl.gen_weight(L.N, L.K, seed=wl.SEED_W + i, outlier_frac=L.frac, device=dev, distinct_positions=False)
        qs.append(qg.qpack_quantize(W, L.bits, L.group, L.frac))
        del W
    return layers, qs


def run_stack7b(qg, P, layers, qs, M):
    """One decode step (M tokens) of the 32-layer 7B-shaped stack with
    per-layer widths 2 (codebook) / 3 / 5 / 6, group 128, 0.1 % outliers: 224
    products in a CUDA graph, those that share x, width and group (q/k,
    gate/up) fused into one call."""
    dev = torch.device("cuda")
    xh, xf = wl.gen_x(M, 4096, device=dev), wl.gen_x(M, 11008, device=dev)
    ys = [torch.empty((M, L.N), device=dev) for L in layers]
    # products that read the same x with the same width and group run as one
    # fused call: q/k(/v) and gate/up of a layer
    calls = []
    for li in range(0, len(layers), 7):
        for grp in ((0, 1, 2), (3,), (4, 5), (6,)):
            idx = [li + j for j in grp]
            run = [idx[0]]
            for i in idx[1:]:
                if layers[i].bits == layers[run[0]].bits:
                    run.append(i)
                else:
                    calls.append(run)
                    run = [i]
            calls.append(run)

    def step7():
        for run in calls:
            x = xf if layers[run[0]].K == 11008 else xh
            if len(run) == 1:
                qg.qgemm_forward(x, qs[run[0]], out=ys[run[0]])
            else:
                qg.qgemm_forward_multi(x, [qs[i] for i in run], outs=[ys[i] for i in run])
    g = capture(step7)
    check_graph_covers(g, ys, f"7B step M={M}")
    ms, n, clocks = timed_object(g, 0.5)
    packed = sum(L.N * L.K * L.bits // 8 for L in layers)
    allb = sum(q.nbytes() for q in qs) + sum(M * (L.K * 2 + L.N * 4) for L in layers)
    del g
    return {"metric": f"7B-shaped mixed-width stack decode, M={M}", "value": round(packed / ms / 1e6, 1),
            "unit": "GB/s", "ms_per_step": round(ms, 4), "all_GBps": round(allb / ms / 1e6, 1),
            "frac_of_hbm_peak": round(allb / ms / 1e6 / P["hbm"], 4), "weights_GB": round(allb / 1e9, 3),
            "launches": len(calls), "replays": n, "clocks": clocks,
            "config": "32 layers q/k/v/o 4096x4096, gate/up 11008x4096, down 4096x11008; widths 6 (layers 0, 1, "
                      "30, 31), else q/k/o 5, v 6, gate/up 2 (codebook), down 2/3/5; group 128, 0.1% outliers, "
                      f"M={M}; products sharing x and width fused per call (q/k, gate/up; q/k/v where all 6-bit)"}


def run_cpu_fused(qg, seconds, qs7=None, layers7=None):
    """The fused multi-threaded CPU qGEMV (every host core) at M = 1 on the
    single 4096 x 4096 layer, on one 4096 x 4096 and one 11008 x 4096 layer of
    each sweep width (group 128), and on the 7B-shaped stack; the quantized
    weights are the device quantizer's (bit-identical to the oracle's),
    copied to host memory."""
    import cpu_baseline as cb
    cb.build()
    dev = torch.device("cuda")
    cores = cb.cores()
    out = {}

    def rate(hws, budget):
        xs = {}
        for hw in hws:
            if hw.K not in xs:
                xs[hw.K] = wl.gen_x(1, hw.K, seed=wl.SEED_X + hw.K).float().numpy().ravel()
        ys = [np.empty(hw.N, np.float32) for hw in hws]
        for hw, y in zip(hws, ys):
            cb.gemv(xs[hw.K], hw, y)
        t0 = time.time()
        passes = 0
        while passes == 0 or time.time() - t0 < budget:
            for hw, y in zip(hws, ys):
                cb.gemv(xs[hw.K], hw, y)
            passes += 1
        dt = time.time() - t0
        return sum(hw.nbytes_packed() for hw in hws) * passes / dt / 1e9, passes

    per = seconds / 4
    L = wl.single_layer()
    q = qg.qpack_quantize(wl.gen_weight(L.N, L.K, device=dev), L.bits, L.group, L.frac)
    v, p = rate([cb.HostWeight.from_device(q)], per)
    out["single_4096_int4_g128"] = {"GBps": round(v, 3), "passes": p}
    for L in wl.mixed_sweep():
        if L.group != 128:
            continue
        W = wl.gen_weight(L.N, L.K, outlier_frac=L.frac, device=dev, distinct_positions=False)
        q = qg.qpack_quantize(W, L.bits, L.group, L.frac)
        v, p = rate([cb.HostWeight.from_device(q)], per / 8)
        out[f"sweep_{L.name}"] = {"GBps": round(v, 3), "passes": p}
    if qs7 is not None:
        hws = [cb.HostWeight.from_device(q) for q in qs7]
        v, p = rate(hws, per)
        out["stack_7b"] = {"GBps": round(v, 3), "passes": p}
    head = out["single_4096_int4_g128"]["GBps"]
    return {"value": head, "unit": "GB/s", "cores": cores,
            "kind": "fused CPU qGEMV: unpack + fp32 FMA with the group scale factored out, std::thread row blocks "
                    "over every hardware thread",
            "sample": f"M=1, packed-weight GB/s; value = the single 4096x4096 INT4 g128 layer; about {seconds:.0f} s "
                      "in all",
            "per_config": out}


# ---------------------------------------------------------------- CPU oracle
def oracle_sample():
    """A bounded sample of the 70B decode workload for the CPU oracle: 128
    rows of each of the 7 projection shapes of a layer, quantized by the
    oracle itself (INT4 g128, 0.1 % outliers), M = 1."""
    import oracle
    oracle.build()
    rows = 128
    qs, xs = [], {}
    for i, L in enumerate(wl.stack_70b(1)):
        W = wl.gen_weight(rows, L.K, seed=wl.SEED_W + i, outlier_frac=L.frac, outlier_seed=wl.SEED_OUTLIER + i)
        qs.append(oracle.quantize(W, L.bits, L.group, L.frac))
        if L.K not in xs:
            xs[L.K] = wl.gen_x(1, L.K, seed=wl.SEED_X + L.K)
    packed = sum(q.packed.nbytes for q in qs)
    return qs, xs, packed


def oracle_pass(sample):
    """One pass of the oracle's product (fp64, one core) over the sample."""
    import oracle
    qs, xs, _ = sample
    for q in qs:
        oracle.linear(xs[q.K], q)


def oracle_rate(seconds: float):
    sample = oracle_sample()
    oracle_pass(sample)                     # warm
    t0 = time.time()
    passes = 0
    while passes == 0 or time.time() - t0 < seconds:
        oracle_pass(sample)
        passes += 1
    dt = time.time() - t0
    txt = (f"{passes} passes over 128 rows of each of the 7 projection shapes of a 70B-shaped layer "
           f"(INT4 g128, 0.1% outliers, M=1; {sample[2] / 1e6:.2f} MB packed per pass) in {dt:.1f} s")
    return sample[2] * passes / dt / 1e9, 1, txt


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    sample = oracle_sample()
    for _ in range(args.warmup):
        oracle_pass(sample)
    t0 = time.time()
    for _ in range(args.steps):
        oracle_pass(sample)
    dt = time.time() - t0
    value = sample[2] * args.steps / dt / 1e9
    txt = (f"each step: one pass of the oracle over 128 rows of each of the 7 projection shapes of a "
           f"70B-shaped layer (INT4 g128, 0.1% outliers, M=1; {sample[2] / 1e6:.2f} MB packed)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": decode_config(args.layers, world),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": txt},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_case(qg, name):
    """One small case of a single kernel family, called three times (for ncu
    captures: a few hundred MB on the device, one kernel per call)."""
    dev = torch.device("cuda")
    if name.startswith("gateup"):
        M = int(name[6:])
        qs = [qg.qpack_quantize(wl.gen_weight(28672, 8192, seed=s, device=dev), 4, 128, 0.001) for s in (1, 2)]
        x = wl.gen_x(M, 8192, device=dev)
        call = lambda: qg.qgemm_forward_multi(x, qs)
    elif name.startswith("tiles") or name.startswith("planar"):
        spec = name[5:] if name.startswith("tiles") else name[6:]   # <bits> or <bits>m<M>
        bits, M = (int(spec.split("m")[0]), int(spec.split("m")[1])) if "m" in spec else (int(spec), 2048)
        q = qg.qpack_quantize(wl.gen_weight(8192, 8192, seed=1, device=dev, outlier_frac=0.001), bits, 128, 0.001)
        x = wl.gen_x(M, 8192, device=dev)
        if name.startswith("tiles"):
            t = qg.qrepack_tiles(q)
            call = lambda: qg.qgemm_forward_tiles(x, q, t)
        else:
            call = lambda: qg.qgemm_forward(x, q)
    elif name.startswith("decode"):   # decode<bits>g<group>: 11008 x 4096 at M = 1
        bits, group = (int(v) for v in name[6:].split("g"))
        q = qg.qpack_quantize(wl.gen_weight(11008, 4096, seed=1, device=dev, outlier_frac=0.001), bits, group, 0.001)
        x = wl.gen_x(1, 4096, device=dev)
        call = lambda: qg.qgemm_forward(x, q)
    elif name == "moe":
        cfg = wl.MoE()
        ex = [[qg.qpack_quantize(wl.gen_weight(cfg.ffn, cfg.hidden, seed=10 * p + e, device=dev), 4, 128, 0.0)
               for e in range(cfg.n_experts)] for p in range(2)]
        x = wl.gen_x(cfg.tokens, cfg.hidden, device=dev)
        topk = wl.gen_topk(cfg.tokens, cfg.top_k, cfg.n_experts).to(dev)
        call = lambda: qg.qgemm_moe_grouped_multi(x, topk, ex)
    elif name == "w8a8":
        q = qg.qpack_quantize(wl.gen_weight(28672, 8192, seed=1, device=dev), 8, 128, 0.0)
        x = wl.gen_x(1, 8192, device=dev)
        call = lambda: qg.qgemm_forward_w8a8(x, q)
    elif name in ("diag", "repack"):
        W = wl.gen_weight(28672, 8192, seed=1, device=dev, outlier_frac=0.001, distinct_positions=False)
        q = qg.qpack_quantize(W, 4, 128, 0.001)
        t = qg.qrepack_tiles(q) if name == "repack" else None
        call = (lambda: qg.qdiag_layer(W, q)) if name == "diag" else (lambda: qg.qrepack_tiles(q, out=t))
    else:
        raise SystemExit(f"unknown case {name}")
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    return {"case": name, "calls": 3}


def secondary(line, key, fn, *a):
    try:
        line[key] = fn(*a)
    except Exception as e:  # report, do not hide
        line[key] = {"error": repr(e)}


def main():
    global CLK
    args = parse()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    import bit_weight_only_group_gb300 as qg
    qg.lib()
    P = peaks()
    CLK = Clocks().start()
    try:
        if args.mode != "all":
            out = {}
            if args.mode == "prefill":
                out = run_prefill(qg, args, P)
                out["widths"] = run_prefill_widths(qg, P)
            elif args.mode == "moe":
                out = run_moe(qg, args)
            elif args.mode == "widths":
                layers7, qs7 = build_stack7b(qg)
                out = {"single": run_single_layer(qg, P), "sweep": run_sweep(qg, P),
                       "stack_7b": [run_stack7b(qg, P, layers7, qs7, M) for M in (1, 8, 32)]}
            elif args.mode == "variants":
                out = run_variants(qg, P)
            elif args.mode == "case":
                out = run_case(qg, args.case)
            elif args.mode == "decode":
                dec, qws = run_decode(qg, args, world, rank, P)
                out = {k: v for k, v in dec.items()}
                for M in (16, 64):
                    out[f"m{M}"] = run_decode_m(qg, qws, wl.stack_70b(args.layers), M, P)
            if rank == 0:
                print(json.dumps(out))
            return 0
        dec, qws = run_decode(qg, args, world, rank, P)
        line = {"metric": METRIC, "value": round(dec["value"], 1), "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dec["ms_per_step"], 4),
                "tokens_per_step": dec["tokens_per_step"], "ms_per_token": round(dec["ms_per_token"], 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "int4 weights, fp16 x fp16 MMA, fp32 accumulate", "data": "synthetic",
                "config": dict(decode_config(args.layers, world), tokens_per_step=dec["tokens_per_step"]),
                "frac_of_hbm_peak": round(dec["value"] / P["hbm"], 4),
                "frac_of_nominal_8TBs": dec["frac_of_nominal_8TBs"],
                "roofline": dec["roofline"], "e2e": dec["e2e"], "clocks": dec["clocks"],
                "gpu_launches": dec["gpu_launches"], "setup_s": dec["setup_s"]}
        if not args.no_secondary and rank == 0:
            layers = wl.stack_70b(args.layers)
            for M in (16, 64):
                secondary(line, f"decode_70b_m{M}", run_decode_m, qg, qws, layers, M, P)
            del qws
            torch.cuda.empty_cache()
            secondary(line, "prefill", run_prefill, qg, args, P)
            secondary(line, "prefill_widths", run_prefill_widths, qg, P)
            secondary(line, "moe", run_moe, qg, args)
            layers7, qs7 = build_stack7b(qg)
            for M, key in ((1, "decode_7b_mixed"), (8, "decode_7b_mixed_m8"), (32, "decode_7b_mixed_m32")):
                secondary(line, key, run_stack7b, qg, P, layers7, qs7, M)
            secondary(line, "single_layer", run_single_layer, qg, P)
            secondary(line, "mixed_sweep", run_sweep, qg, P)
            secondary(line, "format_variants", run_variants, qg, P)
            secondary(line, "quantize", run_quantize, qg, P)
            secondary(line, "cpu_fused_baseline", run_cpu_fused, qg, args.cpu_seconds, qs7, layers7)
            del qs7
        else:
            del qws
        if rank == 0:
            v, cores, txt = oracle_rate(args.cpu_seconds)
            line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                    "sample": txt}
            print(json.dumps(line))
    finally:
        CLK.stop()
    barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
