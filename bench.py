#!/usr/bin/env python3
"""Benchmark of the GB300 MoE FFN layer (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one whole layer (router logits, top-k, grouping, activation
quantisation, gate/up GEMM + SiLU*up, down GEMM, combine) over the
workload's T tokens, on seeded synthetic inputs of the workload's shapes.
Default workload: the DeepSeek-V3-shaped decode layer with T = 16 tokens
(metric: microseconds per layer, lower is better).  Prefill workloads report
tokens per second.

Device timing: CUDA events around every step on the launching stream, after
W warm-up steps; L2 is flushed between steps, outside the timed events (a
512 MiB write, then a 512 MiB read of another buffer, so that L2 holds
clean lines unrelated to the layer).  The dominant kernel's duration comes from the library's
stage events around that kernel alone, inside each timed step (an event
between two kernels costs their programmatic-launch overlap, so the other
stage boundaries carry none); the split over all stages is reported from
separate untimed steps.  e2e: the same layer through
moe_forward_host from pinned host buffers (copies included).  cpu_baseline:
the CPU oracle on the host cores, on a bounded sample of the workload.

With a DeepSeek-V3 decode workload (the default), the same run also times
the 8K-token DeepSeek-V3 prefill layer on the same weights and reports it
under "prefill_8k" (tokens per second, the tensor-core roofline of the
dominant expert GEMM, the whole-layer roofline, e2e and its own oracle
baseline); --no-prefill-beside skips it.

--impl reference times the CPU oracle itself (there is no other reference
implementation of this layer) on the same workload and prints the same line
with "impl": "reference".
"""
from __future__ import annotations

import argparse
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

import synth  # noqa: E402
from moe_expert_ffn_02_gb300 import roofline  # noqa: E402

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.json")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP8_OVER_BF16 = 2.0          # nominal dense ratio (4.5 / 2.25 PFLOP/s)
L2_FLUSH_BYTES = 512 << 20
L2_NOTE = "flushed between steps (512 MiB written, then 512 MiB of another buffer read; outside the timed events)"


class L2Flush:
    """Evicts L2 between timed steps: writes a buffer four times the size of
    L2, then reads another one of the same size.  After the write alone L2
    is full of dirty lines, and the next step would pay for writing them
    back to HBM as it allocates its own lines (about 130 MB, a third of a
    one-token decode layer's own traffic); after the read the resident
    lines are clean and belong to no input of the step."""

    def __init__(self):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None, help="timed steps (default 300 decode, 20 prefill)")
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="ds_decode_t16", choices=sorted(synth.WORKLOADS))
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-prefill-beside", action="store_true",
                   help="decode workloads: skip the 8K-token prefill record timed in the same run")
    p.add_argument("--no-graph", action="store_true", help="decode: time plain launches instead of a graph replay")
    p.add_argument("--layers", type=int, default=1,
                   help="> 1: time a stack of this many layers (distinct weight copies in HBM, distinct routers), "
                        "captured as one CUDA graph; the metric is then per layer")
    p.add_argument("--host-tiles", action="store_true",
                   help="with --layers: keep every layer's expert tiles in pinned host memory and stream them "
                        "through a two-slot device ring while the previous layer computes")
    a = p.parse_args()
    a.warmup = max(a.warmup, 3)
    if a.steps is None:
        a.steps = 300 if synth.WORKLOADS[a.workload].T <= 64 else 20
    return a


def peaks():
    try:
        d = json.load(open(MEASURED_PEAKS))
        return {"hbm": float(d["hbm_gbs"]), "bf16": float(d["bf16_tflops"]),
                "bf16_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "src": "measured"}
    except Exception:
        return {"hbm": FALLBACK_HBM_GBS, "bf16": FALLBACK_BF16_TFLOPS, "bf16_sustained": 1700.0, "src": "fallback"}


def is_decode(wl) -> bool:
    return wl.T <= 64


def metric_of(wl):
    if is_decode(wl):
        return "moe_layer_decode_us_per_layer", "us/layer", False
    return "moe_layer_prefill_tokens_per_s", "tokens/s", True


def value_of(wl, seconds_per_step: float, n_ranks: int = 1):
    """Whole-job figure of a step timed as the max over n_ranks replicas, each
    running the workload's layer: decode, microseconds per layer over all the
    layers the job ran (n_ranks per step); prefill, tokens per second over all
    ranks."""
    if is_decode(wl):
        return seconds_per_step * 1e6 / n_ranks
    return wl.T * n_ranks / seconds_per_step


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if len(r) > 4 + i and r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


# the source file of each timed GEMM; its traffic record is tied to that file and the shared headers
KERNEL_SOURCES = {"decode": "expert_dec.cu", "prefill": "expert_tc.cu"}
SHARED_HEADERS = ("moe_internal.cuh", "tcgen05.cuh")


def kernel_source_hash(path_kind: str) -> str:
    """Hash of the sources one GEMM kernel is compiled from (its file and the
    shared headers): a committed DRAM-traffic figure stays valid while they
    are unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_expert_ffn_02_gb300", "csrc")
    for f in (KERNEL_SOURCES[path_kind],) + SHARED_HEADERS:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str, path_kind: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current sources of that kernel; else None."""
    try:
        d = json.load(open(TRAFFIC_FILE))
    except Exception:
        return None
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash(path_kind):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------- CPU oracle timing

def oracle_sample_plan(wl, target_s: float = 15.0):
    """Tokens per oracle call and number of calls for ~target_s of CPU work."""
    import oracle
    per_token_macs = 3 * wl.hidden * wl.inter * (wl.top_k + wl.n_shared) + wl.hidden * wl.n_experts
    rate = 0.6e9 * oracle.threads()          # rough fp64 MAC/s of the oracle per core
    tokens = max(1, min(wl.T, int(target_s * rate / per_token_macs)))
    return tokens


def time_oracle(wl, inp, rows, repeats=1):
    """Wall time of the oracle layer (logits + routing + experts + combine) on `rows`."""
    import oracle
    sub = dict(inp, x=inp["x"][rows])
    best = None
    for _ in range(repeats):
        t0 = time.perf_counter()
        L = oracle.logits(sub["x"], inp["router_w"], inp["router_b"])
        r = oracle.route_from_logits(L, wl.top_k)
        oracle.forward(sub, wl.top_k, r["ids"], r["w"])
        dt = time.perf_counter() - t0
        best = dt if best is None else min(best, dt)
    return best


def cpu_value(wl, seconds: float, n_tokens: int):
    """Oracle throughput in the workload's unit (decode: us for a T-token layer)."""
    if is_decode(wl):
        return seconds / n_tokens * wl.T * 1e6
    return n_tokens / seconds


# ---------------------------------------------------------------------------- reference arm

def run_reference(a, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    metric, unit, hib = metric_of(wl)
    inp = synth.make_inputs(wl, seed=a.seed)
    # at least one token per oracle thread: the oracle runs tokens in parallel, so a sample
    # smaller than its thread count takes as long as a full one and would scale up wrongly
    n_tok = min(wl.T, max(oracle.threads(), oracle_sample_plan(wl, target_s=60.0 / max(1, a.steps + a.warmup))))
    rows = np.arange(n_tok)
    for _ in range(a.warmup):
        time_oracle(wl, inp, rows[: max(1, n_tok // 4)])
    times = [time_oracle(wl, inp, rows) for _ in range(a.steps)]
    sec = sum(times) / len(times)
    v = cpu_value(wl, sec, n_tok)
    line = {
        "impl": "reference", "metric": metric, "value": v, "unit": unit, "n_gpus": a.gpus, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": sec * 1e3, "higher_is_better": hib, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "T": wl.T, "hidden": wl.hidden, "inter": wl.inter,
                   "n_experts": wl.n_experts, "top_k": wl.top_k, "n_shared": wl.n_shared},
        "cpu_baseline": {"value": v, "unit": unit, "cores": oracle.threads(), "kind": "oracle",
                         "sample": f"first {n_tok} of {wl.T} tokens per step, scaled to the workload"},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- our arm

def time_layer(a, layer, wl, x_np, steps, world, local):
    """Warm-up, diagnostic and timed steps of one workload on `layer`; returns
    the fields of a bench line (value, roofline of the dominant kernel, whole
    layer roofline, end-to-end figure, clocks, stage split)."""
    import torch
    import torch.distributed as dist

    import moe_expert_ffn_02_gb300 as moe
    metric, unit, hib = metric_of(wl)
    T, H = wl.T, wl.hidden
    mode = moe.MODE_DECODE if is_decode(wl) else moe.MODE_PREFILL
    stream = torch.cuda.current_stream()
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    y = torch.empty_like(x)
    ws, nbytes = layer.workspace(T, mode)
    fwd = moe.moe_forward_decode if mode == moe.MODE_DECODE else moe.moe_forward_prefill
    flush = L2Flush()

    def step():
        fwd(layer.handle, x.data_ptr(), T, y.data_ptr(), None, ws, nbytes, stream.cuda_stream)

    # routing of this workload (for the algorithmic-byte count)
    ids = torch.empty((T, wl.top_k), dtype=torch.int32, device="cuda")
    moe.moe_forward_prefill(layer.handle, x.data_ptr(), T, y.data_ptr(), {"topk_ids": ids.data_ptr()}, ws, nbytes,
                            stream.cuda_stream)
    ids_np = ids.cpu().numpy()
    st, flags = moe.moe_get_device_status(layer.handle, stream.cuda_stream)
    if st != 0:
        raise RuntimeError(f"device status {st} flags {flags:#x}")

    for _ in range(a.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    use_graph = mode == moe.MODE_DECODE and not a.no_graph

    # untimed diagnostic steps with every stage's events: the stage split, and which expert GEMM dominates
    moe.moe_profile_enable(layer.handle, True)
    g_diag = moe.LayerStackGraph([layer.handle], mode, x, y) if use_graph else None
    diag = []
    for _ in range(max(3, a.warmup)):
        flush()
        g_diag.replay() if g_diag is not None else step()
        diag.append(moe.moe_profile_read(layer.handle))
    torch.cuda.synchronize()
    del g_diag
    moe.moe_profile_enable(layer.handle, False)
    mean_stage = {k: statistics.mean(d[k] for d in diag) for k in diag[0]}
    dom = "gate_up" if mean_stage["gate_up"] >= mean_stage["down"] else "down"

    # timed steps: only the dominant kernel's two events are recorded (for its roofline); an event
    # between two kernels removes their programmatic-launch overlap, so the other boundaries carry none
    moe.moe_profile_enable(layer.handle, True, stages=(dom,))
    # decode: the step is one CUDA graph replay (the layer's kernels, and the events, captured once),
    # as a decode loop runs it
    graph = None
    if use_graph:
        graph = moe.LayerStackGraph([layer.handle], mode, x, y)
        for _ in range(a.warmup):
            flush()
            graph.replay()
        torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    stage_ms = []
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(steps):
            flush()
            starts[i].record(stream)
            graph.replay() if graph is not None else step()
            ends[i].record(stream)
            stage_ms.append(moe.moe_profile_read(layer.handle)[dom])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    moe.moe_profile_enable(layer.handle, False)
    del graph
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_s = sum(step_ms) / 1e3
    if world > 1:
        t = torch.tensor([total_s], device="cuda", dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_s = float(t.item())
        dist.barrier()
    sec_per_step = total_s / steps
    value = value_of(wl, sec_per_step, world)
    # kernels per step: decode-sized batches (T <= 64) route in 2 (logits GEMV, one-CTA top-k and grouping),
    # larger ones in 5 (logits GEMM, top-k, count, scan, scatter); then quantise, gate/up, down, combine
    n_launches = (6 if T <= 64 else 9) * steps

    # ---------------------------------------------- roofline of the dominant kernel
    pk = peaks()
    dom_s = statistics.mean(stage_ms) / 1e3
    n_touched = roofline.touched_experts(ids_np, wl.n_experts) + wl.n_shared
    rows = T * wl.top_k + T * wl.n_shared
    if is_decode(wl):
        if dom == "gate_up":
            alg = roofline.decode_gate_up_bytes(ids_np, H, wl.inter, wl.n_experts, wl.n_shared) + rows * (H + wl.inter)
        else:
            alg = n_touched * (H * wl.inter + (H // 128) * (wl.inter // 128) * 4) + rows * (wl.inter + 4 * H)
        achieved = alg / dom_s / 1e9
        roof = {"bound": "hbm", "kernel": f"moe::dec::expert_dec_kernel<{1 if dom == 'gate_up' else 0}> ({dom})",
                "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s", "frac": achieved / pk["hbm"],
                "algorithmic_bytes_per_launch": alg, "peak_source": pk["src"],
                "traffic": traffic_for(dom, wl.name, "decode")}
    else:
        flops_all = roofline.layer_flops(T, H, wl.inter, wl.top_k, wl.n_shared)
        alg = flops_all * (2 / 3 if dom == "gate_up" else 1 / 3)
        achieved = alg / dom_s / 1e12
        peak = pk["bf16"] * FP8_OVER_BF16
        roof = {"bound": "tensor", "kernel": f"tc::expert_tc_kernel<{1 if dom == 'gate_up' else 0}> ({dom})",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "algorithmic_flops_per_launch": alg,
                "peak_source": f"{pk['src']} bf16 burst x {FP8_OVER_BF16} (nominal fp8/bf16 dense ratio)",
                "traffic": traffic_for(dom, wl.name, "prefill")}

    # ---------------------------------------------- the whole layer against the same peak (the targets are
    # stated per layer: touched-expert bytes / layer time for decode, expert FLOP / layer time for prefill)
    if is_decode(wl):
        lb = roofline.decode_weight_bytes(ids_np, H, wl.inter, wl.n_experts, wl.n_shared)
        layer_roof = {"bound": "hbm", "algorithmic_bytes": lb, "achieved": lb / sec_per_step / 1e9,
                      "peak": pk["hbm"], "unit": "GB/s", "frac": lb / sec_per_step / 1e9 / pk["hbm"]}
    else:
        lf = roofline.layer_flops(T, H, wl.inter, wl.top_k, wl.n_shared)
        layer_roof = {"bound": "tensor", "algorithmic_flops": lf, "achieved": lf / sec_per_step / 1e12,
                      "peak": pk["bf16"] * FP8_OVER_BF16, "unit": "TFLOP/s",
                      "frac": lf / sec_per_step / 1e12 / (pk["bf16"] * FP8_OVER_BF16)}

    # ---------------------------------------------- end to end through the host entry
    e2e = None
    if not a.no_e2e:
        xh = torch.from_numpy(x_np.view(np.int16)).pin_memory()
        yh = torch.empty_like(xh).pin_memory()
        ws_h, nb_h = layer.workspace(T, mode)
        for _ in range(2):
            moe.moe_forward_host(layer.handle, mode, xh.data_ptr(), T, yh.data_ptr(), ws_h, nb_h, stream.cuda_stream)
        e_ms = []
        for _ in range(steps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            moe.moe_forward_host(layer.handle, mode, xh.data_ptr(), T, yh.data_ptr(), ws_h, nb_h, stream.cuda_stream)
            e1.record(stream)
            e1.synchronize()
            e_ms.append(e0.elapsed_time(e1))
        e2e = {"value": value_of(wl, statistics.mean(e_ms) / 1e3, world), "unit": unit,
               "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2}
    del x, y, flush
    torch.cuda.empty_cache()
    return {
        "metric": metric, "value": value, "unit": unit, "steps": steps, "ms_per_step": sec_per_step * 1e3,
        "higher_is_better": hib, "roofline": roof, "layer_roofline": layer_roof, "e2e": e2e,
        "gpu_launches": n_launches * world, "clocks": clk.summary(), "stage_ms": mean_stage,
        "touched_experts": n_touched, "wall_s_timed_region": t_wall, "tokens_per_s": T * world / sec_per_step,
        "graph": use_graph,
    }


def cpu_baseline_of(wl, inp_x, router_inp, target_s):
    """The oracle on the host cores on the first tokens of the workload, scaled to its unit."""
    import oracle
    oracle.build()
    n_tok = min(wl.T, max(oracle.threads(), oracle_sample_plan(wl, target_s=target_s)))
    sec = time_oracle(wl, dict(router_inp, x=inp_x), np.arange(n_tok))
    return {"value": cpu_value(wl, sec, n_tok), "unit": metric_of(wl)[1], "cores": oracle.threads(), "kind": "oracle",
            "sample": f"first {n_tok} of {wl.T} tokens (logits, routing, experts, combine), scaled to the workload"}


def config_of(wl, world, graph):
    return {"workload": wl.name, "T": wl.T, "hidden": wl.hidden, "inter": wl.inter, "n_experts": wl.n_experts,
            "top_k": wl.top_k, "n_shared": wl.n_shared, "parallelism": f"replicas{world}", "graph": graph,
            "l2": L2_NOTE}


# The prefill workload timed beside a decode workload of the same layer
# shapes (DeepSeek-V3: the decode layers' weights are the 8K prefill layer's).
PREFILL_BESIDE = {"ds_decode_t1": "ds_prefill_8k", "ds_decode_t4": "ds_prefill_8k", "ds_decode_t16": "ds_prefill_8k"}


def run_ours(a, wl):
    import torch
    import torch.distributed as dist

    import moe_expert_ffn_02_gb300 as moe

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    moe.load()
    inp = synth.make_inputs(wl, seed=a.seed)
    dev = {k: (torch.from_numpy(np.ascontiguousarray(v)).cuda() if v is not None else None)
           for k, v in inp.items() if k != "x"}
    layer = moe.Layer(wl.hidden, wl.inter, wl.n_experts, wl.top_k, dev, n_shared=wl.n_shared)
    del dev
    torch.cuda.empty_cache()
    rec = time_layer(a, layer, wl, inp["x"], a.steps, world, local)

    # the 8K-token prefill layer on the same weights, timed in the same run
    sub = None
    pname = None if a.no_prefill_beside else PREFILL_BESIDE.get(wl.name)
    if pname:
        pw = synth.WORKLOADS[pname]
        px = synth.bf16_normal(a.seed, synth.STREAM_X, (pw.T, pw.hidden))
        sub = time_layer(a, layer, pw, px, min(a.steps, 20), world, local)
        sub["config"] = config_of(pw, world, sub.pop("graph"))
        sub["dtype"] = "fp8_e4m3"
        if not a.no_cpu_baseline and rank == 0 and world == 1:
            sub["cpu_baseline"] = cpu_baseline_of(pw, px, inp, 8.0)

    cpu = None
    if not a.no_cpu_baseline and rank == 0 and world == 1:
        cpu = cpu_baseline_of(wl, inp["x"], inp, 12.0)

    layer.close()
    if rank == 0:
        line = {
            "metric": rec["metric"], "value": rec["value"], "unit": rec["unit"], "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": rec["higher_is_better"],
            "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic",
            "config": config_of(wl, world, rec["graph"]),
            "roofline": rec["roofline"], "layer_roofline": rec["layer_roofline"], "cpu_baseline": cpu,
            "e2e": rec["e2e"], "gpu_launches": rec["gpu_launches"] + (sub["gpu_launches"] if sub else 0),
            "clocks": rec["clocks"], "stage_ms": rec["stage_ms"],
            "stage_ms_note": "every stage timed in separate untimed steps; the timed steps carry only the "
                             "dominant kernel's events", "touched_experts": rec["touched_experts"],
            "wall_s_timed_region": rec["wall_s_timed_region"], "tokens_per_s": rec["tokens_per_s"],
        }
        if sub is not None:
            line["prefill_8k"] = sub
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def host_copy_peak_gbps(nbytes: int = 2 << 30, reps: int = 3) -> float:
    """The machine's host -> device copy rate: one copy from pinned host memory,
    best of `reps` (the reference for the host-tile ring's streaming rate)."""
    import torch
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        e1.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del src, dst
    return best


def run_layers(a, wl):
    """A stack of a.layers layers run as one CUDA graph replay per step
    (moe_forward_layers inside LayerStackGraph).  Every layer is its own copy
    of the expert weights in HBM with its own router (seed + l), so each
    layer routes its input differently; the input of layer l + 1 is the
    output of layer l."""
    import torch
    import moe_expert_ffn_02_gb300 as moe
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    moe.load()
    metric, unit, hib = metric_of(wl)
    inp = synth.make_inputs(wl, seed=a.seed)
    dev = {k: (torch.from_numpy(np.ascontiguousarray(v)).cuda() if v is not None else None)
           for k, v in inp.items() if k != "x"}
    layers = []
    for l in range(a.layers):
        if l:
            rstd = wl.router_std if wl.router_std is not None else 1.0 / np.sqrt(wl.hidden)
            dev["router_w"] = torch.from_numpy(
                synth.f32_normal(a.seed + l, synth.STREAM_ROUTER_W, (wl.n_experts, wl.hidden), float(rstd))).cuda()
        layers.append(moe.Layer(wl.hidden, wl.inter, wl.n_experts, wl.top_k, dev, n_shared=wl.n_shared,
                                host_tiles=a.host_tiles))
    del dev
    torch.cuda.empty_cache()
    T, H = wl.T, wl.hidden
    mode = moe.MODE_DECODE if is_decode(wl) else moe.MODE_PREFILL
    x = torch.from_numpy(inp["x"].view(np.int16)).cuda()
    y = torch.empty_like(x)

    # per-layer routing of the chained inputs, for the touched-byte count
    touched_bytes, xi = 0, x.clone()
    for ly in (layers if not a.host_tiles else []):
        ids = torch.empty((T, wl.top_k), dtype=torch.int32, device="cuda")
        ws, nb = ly.workspace(T, mode)
        yi = torch.empty_like(xi)
        moe.moe_forward_prefill(ly.handle, xi.data_ptr(), T, yi.data_ptr(), {"topk_ids": ids.data_ptr()}, ws, nb,
                                torch.cuda.current_stream().cuda_stream)
        touched_bytes += roofline.decode_weight_bytes(ids.cpu().numpy(), H, wl.inter, wl.n_experts, wl.n_shared)
        xi = yi
    if a.host_tiles:
        g = moe.StreamedStack(layers, mode, x, y)
        g.replay = g.run
        tiles_bytes = moe.moe_tiles_bytes(layers[0].handle)
    else:
        g = moe.LayerStackGraph([ly.handle for ly in layers], mode, x, y)
    flush = L2Flush()
    for _ in range(a.warmup):
        flush()
        g.replay()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps)]
    cur = torch.cuda.current_stream()          # the graph replays on the current stream
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        for i in range(a.steps):
            flush()
            starts[i].record(cur)
            g.replay()
            ends[i].record(cur)
        torch.cuda.synchronize()
    sec_per_step = sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / a.steps / 1e3
    for ly in layers:
        st, flags = moe.moe_get_device_status(ly.handle, 0)
        if st != 0:
            raise RuntimeError(f"device status {st} flags {flags:#x}")
    pk = peaks()
    per_layer = sec_per_step / a.layers
    if is_decode(wl) and not a.host_tiles:
        achieved = touched_bytes / sec_per_step / 1e9
        roof = {"bound": "hbm", "kernel": f"stack of {a.layers} layers (one CUDA graph)", "achieved": achieved,
                "peak": pk["hbm"], "unit": "GB/s", "frac": achieved / pk["hbm"],
                "algorithmic_bytes_per_launch": touched_bytes, "peak_source": pk["src"], "traffic": None}
    else:
        lf = roofline.layer_flops(T, H, wl.inter, wl.top_k, wl.n_shared) * a.layers
        achieved = lf / sec_per_step / 1e12
        peak = pk["bf16"] * FP8_OVER_BF16
        roof = {"bound": "tensor", "achieved": achieved,
                "kernel": f"stack of {a.layers} layers " + ("(two-slot host-tile ring)" if a.host_tiles else
                                                            "(one CUDA graph)"),
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "algorithmic_flops_per_launch": lf,
                "peak_source": f"{pk['src']} bf16 burst x {FP8_OVER_BF16} (nominal fp8/bf16 dense ratio)",
                "traffic": None}
    line = {
        "metric": metric, "value": value_of(wl, per_layer, 1), "unit": unit, "n_gpus": 1, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": sec_per_step * 1e3, "higher_is_better": hib, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic",
        "config": {"workload": wl.name, "T": T, "hidden": H, "inter": wl.inter, "n_experts": wl.n_experts,
                   "top_k": wl.top_k, "n_shared": wl.n_shared, "parallelism": "replicas1", "layers": a.layers,
                   "graph": True, "l2": L2_NOTE},
        "roofline": roof, "cpu_baseline": None, "e2e": None, "gpu_launches": (6 if T <= 64 else 9) * a.layers * a.steps,
        "clocks": clk.summary(),
    }
    if a.host_tiles:
        line["config"]["graph"] = False
        line["config"]["weights"] = "expert tiles in pinned host memory, streamed host->device per layer"
        achieved = tiles_bytes * a.layers / sec_per_step / 1e9
        peak = host_copy_peak_gbps()
        line["host_stream"] = {"tiles_bytes_per_layer": tiles_bytes, "achieved_GBps": achieved,
                               "host_copy_peak_GBps": peak, "frac": achieved / peak,
                               "peak_how": "one 2 GiB pinned host -> device copy, best of 3, CUDA events"}
    print(json.dumps(line), flush=True)
    for ly in layers:
        ly.close()
    return 0


def main():
    a = parse()
    wl = synth.WORKLOADS[a.workload]
    if a.impl == "reference":
        return run_reference(a, wl)
    if a.layers > 1:
        return run_layers(a, wl)
    return run_ours(a, wl)


if __name__ == "__main__":
    sys.exit(main())
