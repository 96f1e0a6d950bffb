#!/usr/bin/env python
"""Benchmark of the SiTU-GLU expert feed-forward on GB300.

One step = one dense SiTU-GLU FFN forward over 16384 tokens (M=2048, I=3072,
bf16): the tcgen05 gate_up GEMM with the activation fused into its epilogue,
then the tcgen05 down GEMM.  ``value`` is tokens/s of that step, device-timed
with CUDA events, L2 flushed between steps.  The same JSON line also carries:
  * ``act``: the standalone activation on [65536, 2x3072] bf16 (GB/s, HBM roofline);
  * ``moe``: the routed layer (index build + grouped FFN + combine) on the Zipf
    top-8 64-expert workload and on the Kimi-K3-shaped layer (896 routed + 2
    shared experts) at 512 and 32768 tokens;
  * ``mxfp8``: the same FFN and routed layers with MX experts (MXFP8 activations,
    MXFP8 or MXFP4 weights, block-scaled tensor cores);
  * ``train``: a training step of the dense FFN (forward keeping gu and h, backward),
    and (``train.grouped``) of the grouped experts on the Zipf top-8 64-expert workload;
  * ``roofline`` of the dominant kernel (the fused gate_up GEMM);
  * ``e2e``: the public ``situ_ffn_forward`` call with host (pinned) buffers,
    host->device copy of x and device->host copy of y inside the timed region;
  * ``cpu_baseline``: the FP64 CPU oracle on a bounded sample of the same rows.

``--impl reference`` times the FP64 CPU oracle itself (the reference arm) on the
same workload, a bounded sample of rows per step.

Multi-GPU (torchrun): every rank runs the same per-GPU workload (replicas, weak
scaling, no collective on the data path); the step time is the max over ranks
and value the tokens of all ranks over that time.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "expert-FFN tokens/s + TFLOP/s (% bf16 TC peak); SiTU act GB/s (% HBM)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20
FLOP_PER_ROW = 6  # x (2*M*2I + 2*I*M) = 6*M*I per row
E2E_CHUNK_ROWS = 4096


# ---------------------------------------------------------------------------
# distributed helpers (replicas; the only collectives are the timing barrier
# and the max/sum reductions of the result)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_ms: float, local_units: float, world: int):
    """Max of the step time and sum of the work over ranks (identity at world 1)."""
    if world <= 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist

    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else None
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------------------
# peaks, clocks, L2
# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None or self.tmp is None:
            return None
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r for r in csv.reader(f) if len(r) >= 9]
        os.unlink(self.tmp.name)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, smax, reasons = [], 0.0, set()
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax = max(smax, float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_digest(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "situ_glu_activation_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, digest: str, units: float):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.txt), if it was captured on the current kernel source;
    else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split("#", 1)[0].split()
                if len(parts) >= 3 and parts[0] == kernel and parts[1] == digest:
                    return float(parts[2]) * units
    except (OSError, ValueError):
        return None
    return None


# ---------------------------------------------------------------------------
# timing
# ---------------------------------------------------------------------------
def timed_steps(step, K: int, W: int, flush, world: int, inner: int = 0):
    """W untimed warm-up steps, then K device-timed steps (CUDA events on the
    current stream, L2 flushed before each).  `step(marks)` may record `inner`
    extra events between its launches.  Returns (per-step ms, per-segment ms)."""
    import torch

    for _ in range(W):
        flush()
        step(None)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    per_step, segs = [], [[] for _ in range(inner + 1)]
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(inner + 2)] for _ in range(K)]
    for i in range(K):
        ev = events[i]
        flush()
        ev[0].record()
        step(ev[1:-1] if inner else None)
        ev[-1].record()
        ev[-1].synchronize()
        per_step.append(ev[0].elapsed_time(ev[-1]))
        for i in range(inner + 1):
            segs[i].append(ev[i].elapsed_time(ev[i + 1]))
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return per_step, segs


def mean(v):
    return sum(v) / len(v)


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def bench_dense(args, dev, peaks, world, flush):
    import torch

    import situ_glu_activation_gb300 as situ
    from situ_glu_activation_gb300 import workloads as wl

    w = wl.WORKLOADS["dense"]
    x, wgu, wd = wl.ffn_inputs(w.M, w.I, w.rows, seed=0, device=dev)
    h = torch.empty(w.rows, w.I, dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(x)
    ws = torch.empty(situ.ffn_workspace_bytes(w.rows, w.M, w.I), dtype=torch.uint8, device=dev)

    # The step: the public dense call, one persistent launch for both projections.
    def step(_):
        situ.situ_ffn_forward(x, wgu, wd, wl.BETA, wl.LINEAR_BETA, y=y, workspace=ws)

    per_step, _ = timed_steps(step, args.steps, args.warmup, flush, world)
    ms = mean(per_step)
    path = situ.ffn_last_path()
    if path != (situ.FFN_PATH_TWO_LAUNCHES if args.ffn_two_launches else situ.FFN_PATH_FUSED):
        raise RuntimeError(f"the dense forward took path {path}")

    # The same projections as two launches, timed apart: the per-GEMM figures.
    def step2(marks):
        situ.situ_ffn_gate_up(x, wgu, wl.BETA, wl.LINEAR_BETA, h=h)
        if marks:
            marks[0].record()
        situ.situ_ffn_down(h, wd, y=y)

    per_step2, (t_gu, t_down) = timed_steps(step2, args.steps, args.warmup, flush, world,
                                            inner=1)
    # The same fused GEMM with both caps removed (SwiGLU): the cost of the caps.
    inf = float("inf")
    sw_ms, _ = timed_steps(lambda m: situ.situ_ffn_gate_up(x, wgu, inf, inf, h=h), args.steps,
                           args.warmup, flush, world)
    flop_gu = 2.0 * w.rows * w.M * 2 * w.I
    flop_down = 2.0 * w.rows * w.I * w.M
    out = {
        "ms": ms, "ms_median": statistics.median(per_step), "tokens": w.rows,
        "launches_per_step": 2 if args.ffn_two_launches else 1,
        "path": "two launches" if args.ffn_two_launches else "one persistent launch",
        "two_launch_ms": mean(per_step2),
        "gate_up_ms": mean(t_gu), "down_ms": mean(t_down),
        "tflops": (flop_gu + flop_down) / (ms * 1e-3) / 1e12,
        "gate_up_tflops": flop_gu / (mean(t_gu) * 1e-3) / 1e12,
        "down_tflops": flop_down / (mean(t_down) * 1e-3) / 1e12,
        "flop_gate_up": flop_gu,
        "swiglu_gate_up_ms": mean(sw_ms),
    }

    # End to end through the public host-buffer call: x is copied in from pinned host
    # memory and y copied back every step, pipelined in row chunks by the library.
    x_h = x.cpu().pin_memory()
    y_h = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    ws = torch.empty(situ.ffn_host_workspace_bytes(w.rows, w.M, w.I, E2E_CHUNK_ROWS),
                     dtype=torch.uint8, device=dev)

    def e2e_step(_):
        situ.situ_ffn_forward_host(x_h, wgu, wd, wl.BETA, wl.LINEAR_BETA, y_host=y_h,
                                   chunk_rows=E2E_CHUNK_ROWS, workspace=ws)

    e2e_ms, _ = timed_steps(e2e_step, args.steps, args.warmup, flush, world)
    out["e2e_ms"] = mean(e2e_ms)
    # The timed step's inputs and output, for the oracle's baseline and accuracy check.
    out["inputs"] = (x.cpu(), wgu.cpu(), wd.cpu())
    out["y"] = y.cpu()
    out["h2d_bytes"] = x.numel() * x.element_size()
    out["d2h_bytes"] = y.numel() * y.element_size()
    return out, w


def bench_act(args, dev, peaks, world, flush, check_rows: int = 0):
    """check_rows > 0: the first check_rows output rows against the FP64 oracle, in bf16
    ulps (the oracle on the host cores)."""
    import numpy as np
    import torch

    import situ_glu_activation_gb300 as situ
    from situ_glu_activation_gb300 import workloads as wl

    w = wl.WORKLOADS["act"]
    g = wl.gate_up_input(w, seed=0, device=dev)
    o = torch.empty(w.rows, w.I, dtype=torch.bfloat16, device=dev)
    per_step, _ = timed_steps(lambda m: situ.situ_glu_act(g, wl.BETA, wl.LINEAR_BETA, out=o),
                              args.steps, args.warmup, flush, world)
    ms = mean(per_step)
    accuracy = None
    if check_rows > 0:
        from oracle import Oracle

        gin = g[:check_rows].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        ref = Oracle().situ_glu_act(gin, wl.BETA, wl.LINEAR_BETA)
        accuracy = ulp_stats(o[:check_rows].cpu(), ref)
    inf = float("inf")
    sw_ms, _ = timed_steps(lambda m: situ.situ_glu_act(g, inf, inf, out=o), args.steps,
                           args.warmup, flush, world)
    nbytes = 3 * w.rows * w.I * 2  # read 2I, write I per row, bf16
    gbs = nbytes / (ms * 1e-3) / 1e9
    digest = source_digest("act.cu", "situ_math.cuh")
    res = {"workload": w.name, "ms": ms, "bytes": nbytes, "gbs": gbs, "swiglu_ms": mean(sw_ms),
           "roofline": {"bound": "hbm", "kernel": "act_bf16_vec_kernel", "achieved": gbs,
                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / peaks["hbm_gbs"],
                        "traffic": profiled_traffic("situ_act", digest, w.rows * w.I)}}
    if accuracy is not None:
        res["accuracy"] = accuracy
    return res


def bench_moe(args, dev, peaks, world, flush, names, cpu=False):
    """Grouped workloads; cpu: also time the FP64 oracle on a sample of each one's
    routes (host copies of the expert weights, made once per weight set)."""
    import torch

    import situ_glu_activation_gb300 as situ
    from situ_glu_activation_gb300 import workloads as wl

    results = {}
    weights = {}
    host_weights = {}
    for name in names:
        w = wl.WORKLOADS[name]
        E = w.num_experts
        key = (E, w.M, w.I)
        if key not in weights:
            weights.clear()
            host_weights.clear()
            torch.cuda.empty_cache()
            weights[key] = wl.expert_weights(E, w.M, w.I, seed=0, device=dev)
        wgu, wd = weights[key]
        ids_cpu = wl.routes(w, seed=0)
        ids = ids_cpu.to(dev)
        x = wl.normal((w.T, w.M), 1.0, seed=0, device=dev)
        R = w.T * w.k_eff
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        tix = torch.empty(R, dtype=torch.int32, device=dev)
        y = torch.empty(w.T, w.k_eff, w.M, dtype=torch.bfloat16, device=dev)
        cw = wl.combine_weights(w.T, w.k, len(w.shared), seed=0).to(dev)
        layer_out = torch.empty(w.T, w.M, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(situ.moe_workspace_bytes(R, E, w.M, w.I), dtype=torch.uint8, device=dev)

        def step(marks):
            situ.situ_moe_build_index(ids, E, expert_offsets=off, token_index=tix)
            if marks:
                marks[0].record()
            situ.situ_moe_grouped_forward(x, off, tix, wgu, wd, w.k_eff, wl.BETA, wl.LINEAR_BETA,
                                          y=y, workspace=ws)
            if marks:
                marks[1].record()
            situ.situ_moe_combine(y, cw, out=layer_out)

        per_step, (t_idx, t_ffn, t_comb) = timed_steps(step, args.steps, args.warmup, flush,
                                                       world, inner=2)
        ms = mean(per_step)
        # The same layer with the combine fused into the down projection (scatter-add).
        ws_c = torch.empty(situ.moe_combined_workspace_bytes(w.T, w.k_eff, E, w.M, w.I),
                           dtype=torch.uint8, device=dev)

        def fused_step(marks):
            situ.situ_moe_build_index(ids, E, expert_offsets=off, token_index=tix)
            situ.situ_moe_grouped_forward_combined(x, off, tix, wgu, wd, cw, wl.BETA,
                                                   wl.LINEAR_BETA, out=layer_out, workspace=ws_c)

        fused_ms, _ = timed_steps(fused_step, args.steps, args.warmup, flush, world)
        del ws_c
        counts = torch.bincount(ids_cpu.view(-1).long(), minlength=E)
        touched = int((counts > 0).sum())
        wbytes = touched * 3 * w.M * w.I * 2
        flop = FLOP_PER_ROW * R * w.M * w.I
        tflops = flop / (ms * 1e-3) / 1e12
        weight_gbs = wbytes / (ms * 1e-3) / 1e9
        results[name] = {
            "workload": w.name, "ms": ms, "index_ms": mean(t_idx), "ffn_ms": mean(t_ffn),
            "combine_ms": mean(t_comb),
            "fused_combine_layer_ms": mean(fused_ms),
            "tokens": w.T, "routes": R, "experts_touched": touched,
            "tokens_per_s": w.T / (ms * 1e-3), "tflops": tflops,
            "tc_frac": tflops / peaks["bf16_tflops"],
            "weight_gbs": weight_gbs, "hbm_frac": weight_gbs / peaks["hbm_gbs"],
            "launches_per_step": 4 + 4 + 1,
            "step": "expert index, grouped SiTU-GLU experts, router-weighted combine",
        }
        if cpu:
            wbytes_all = (wgu.numel() + wd.numel()) * 2
            if key not in host_weights and host_bytes_available() > 2 * wbytes_all:
                host_weights[key] = (wgu.cpu(), wd.cpu())
            if key in host_weights:
                base, sample, ref = cpu_baseline_routes(w, x, ids_cpu, *host_weights[key])
                results[name]["cpu_baseline"] = base
                # The GPU's outputs of the sampled routes against the oracle's.
                got = y.view(-1, w.M).index_select(0, torch.from_numpy(sample).to(dev)).cpu()
                results[name]["accuracy"] = accuracy_stats(got, ref.reshape(-1, w.M))
            else:
                results[name]["cpu_baseline"] = {
                    "unavailable": f"host memory below twice the {wbytes_all / 1e9:.1f} GB of "
                                   "expert weights the oracle needs"}
        del x, y, ws, off, tix, ids
    weights.clear()
    host_weights.clear()
    torch.cuda.empty_cache()
    return results


def bench_train(args, dev, peaks, world, flush):
    """Training step of the dense FFN: forward that keeps gu and h, then the
    backward for a seeded upstream gradient (dx, dW_gate_up, dW_down)."""
    import torch

    import situ_glu_activation_gb300 as situ
    from situ_glu_activation_gb300 import workloads as wl

    w = wl.WORKLOADS["dense"]
    x, wgu, wd = wl.ffn_inputs(w.M, w.I, w.rows, seed=0, device=dev)
    dy = wl.normal((w.rows, w.M), 1.0, seed=7, device=dev)
    ws = torch.empty(situ.ffn_backward_workspace_bytes(w.rows, w.M, w.I), dtype=torch.uint8,
                     device=dev)
    state = {}

    def step(marks):
        y, gu, h = situ.situ_ffn_forward_train(x, wgu, wd, wl.BETA, wl.LINEAR_BETA)
        if marks:
            marks[0].record()
        state["g"] = situ.situ_ffn_backward(x, wgu, wd, gu, h, dy, wl.BETA, wl.LINEAR_BETA,
                                            workspace=ws)

    per_step, (t_fwd, t_bwd) = timed_steps(step, args.steps, args.warmup, flush, world, inner=1)
    ms = mean(per_step)
    flop_f = 6.0 * w.rows * w.M * w.I
    flop_b = 12.0 * w.rows * w.M * w.I
    return {"workload": w.name + ", training step (forward keeping gu and h, backward)",
            "ms": ms, "forward_ms": mean(t_fwd), "backward_ms": mean(t_bwd),
            "tokens_per_s": w.rows / (ms * 1e-3),
            "tflops": (flop_f + flop_b) / (ms * 1e-3) / 1e12,
            "backward_tflops": flop_b / (mean(t_bwd) * 1e-3) / 1e12,
            "tc_frac": (flop_f + flop_b) / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "launches_per_step": 2 + 4}


def bench_mx(args, dev, peaks, world, flush, names=("grouped", "k3_decode", "k3_prefill")):
    """MX experts: the dense FFN (quantize x, block-scaled gate_up with the activation
    and h's MX quantization in its epilogue, block-scaled down) and the routed layers,
    each with MXFP8 and with MXFP4 expert weights (quantized once, outside the
    timing); activations are MXFP8 throughout."""
    import torch

    import situ_glu_activation_gb300 as situ
    from situ_glu_activation_gb300 import workloads as wl

    fp8_peak = 2.0 * peaks["bf16_tflops"]  # nominal dense fp8 / bf16 ratio 4.5 / 2.25
    out = {"peak_fp8_tflops": fp8_peak,
           "peak_note": "measured bf16 burst x 2 (nominal dense fp8/bf16 ratio); the "
                        "E4M3 x E2M1 MMA runs at the fp8 rate"}
    fmts = (("mxfp8", situ.MX_E4M3, 1.0), ("mxfp4", situ.MX_E2M1, 0.5))
    w = wl.WORKLOADS["dense"]
    x, wgu, wd = wl.ffn_inputs(w.M, w.I, w.rows, seed=0, device=dev)
    y = torch.empty_like(x)
    ws = torch.empty(situ.ffn_mxfp8_workspace_bytes(w.rows, w.M, w.I), dtype=torch.uint8,
                     device=dev)
    xq = situ.mx_quantize_act(x)
    flop = FLOP_PER_ROW * w.rows * w.M * w.I
    flop_gu = 4.0 * w.rows * w.M * w.I
    for tag, fmt, _ in fmts:
        wguq = situ.mx_quantize_weights(wgu, situ.MX_GATE_UP, fmt)
        wdq = situ.mx_quantize_weights(wd, situ.MX_DOWN, fmt)
        per_step, _ = timed_steps(
            lambda m: situ.situ_ffn_forward_mxfp8(x, wguq, wdq, wl.BETA, wl.LINEAR_BETA, y=y,
                                                  workspace=ws),
            args.steps, args.warmup, flush, world)
        gu_ms, _ = timed_steps(lambda m: situ.situ_ffn_gate_up_mxfp8(xq, wguq, wl.BETA,
                                                                     wl.LINEAR_BETA),
                               args.steps, args.warmup, flush, world)
        ms = mean(per_step)
        out["dense_" + tag] = {
            "workload": w.name + f", MXFP8 activations, {tag.upper()} weights", "ms": ms,
            "tokens_per_s": w.rows / (ms * 1e-3), "tflops": flop / (ms * 1e-3) / 1e12,
            "tc_frac_fp8": flop / (ms * 1e-3) / 1e12 / fp8_peak,
            "gate_up_ms": mean(gu_ms),
            "gate_up_tflops": flop_gu / (mean(gu_ms) * 1e-3) / 1e12,
            "gate_up_tc_frac_fp8": flop_gu / (mean(gu_ms) * 1e-3) / 1e12 / fp8_peak,
            "launches_per_step": 3}
        del wguq, wdq
    del x, y, ws, xq, wgu, wd
    torch.cuda.empty_cache()
    for name in names:
        wk = wl.WORKLOADS[name]
        E = wk.num_experts
        R = wk.T * wk.k_eff
        ids_cpu = wl.routes(wk, seed=0)
        ids = ids_cpu.to(dev)
        x = wl.normal((wk.T, wk.M), 1.0, seed=0, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        tix = torch.empty(R, dtype=torch.int32, device=dev)
        y = torch.empty(wk.T, wk.k_eff, wk.M, dtype=torch.bfloat16, device=dev)
        cw = wl.combine_weights(wk.T, wk.k, len(wk.shared), seed=0).to(dev)
        layer_out = torch.empty(wk.T, wk.M, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(situ.moe_mxfp8_workspace_bytes(R, E, wk.M, wk.I), dtype=torch.uint8,
                         device=dev)
        counts = torch.bincount(ids_cpu.view(-1).long(), minlength=E)
        touched = int((counts > 0).sum())
        flop = FLOP_PER_ROW * R * wk.M * wk.I
        for tag, fmt, code_bytes in fmts:
            wgu, wd = wl.expert_weights(E, wk.M, wk.I, seed=0, device=dev)
            wguq = situ.mx_quantize_weights(wgu, situ.MX_GATE_UP, fmt)
            del wgu
            wdq = situ.mx_quantize_weights(wd, situ.MX_DOWN, fmt)
            del wd
            torch.cuda.empty_cache()

            def step(marks):
                situ.situ_moe_build_index(ids, E, expert_offsets=off, token_index=tix)
                situ.situ_moe_grouped_forward_mxfp8(x, off, tix, wguq, wdq, wk.k_eff, wl.BETA,
                                                    wl.LINEAR_BETA, y=y, workspace=ws)
                situ.situ_moe_combine(y, cw, out=layer_out)

            per_step, _ = timed_steps(step, args.steps, args.warmup, flush, world)
            ms = mean(per_step)
            # weight bytes streamed: codes + scales (1 byte per 32 elements)
            wbytes = touched * 3 * wk.M * wk.I * (code_bytes + 1 / 32)
            out[name + "_" + tag] = {
                "workload": wk.name + f", MXFP8 activations, {tag.upper()} expert weights",
                "ms": ms, "tokens_per_s": wk.T / (ms * 1e-3),
                "tflops": flop / (ms * 1e-3) / 1e12,
                "tc_frac_fp8": flop / (ms * 1e-3) / 1e12 / fp8_peak,
                "weight_gbs": wbytes / (ms * 1e-3) / 1e9,
                "hbm_frac": wbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "launches_per_step": 4 + 4 + 1}
            del wguq, wdq
            torch.cuda.empty_cache()
        del x, y, ws, off, tix, ids
        torch.cuda.empty_cache()
    return out


def bench_moe_train(args, dev, peaks, world, flush, name="grouped"):
    """Training step of the grouped experts (E=64, 16384 tokens top-8 Zipf; or the
    16-expert slice for profiling): expert index, forward that keeps gu and h in
    expert order, backward for a seeded upstream gradient of the per-route outputs
    (dx, per-expert dW)."""
    import torch

    import situ_glu_activation_gb300 as situ
    from situ_glu_activation_gb300 import workloads as wl

    w = wl.WORKLOADS[name]
    E = w.num_experts
    R = w.T * w.k_eff
    wgu, wd = wl.expert_weights(E, w.M, w.I, seed=0, device=dev)
    ids = wl.routes(w, seed=0).to(dev)
    x = wl.normal((w.T, w.M), 1.0, seed=0, device=dev)
    dy = wl.normal((w.T, w.k_eff, w.M), 1.0, seed=7, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    tix = torch.empty(R, dtype=torch.int32, device=dev)
    ws_f = torch.empty(situ.moe_workspace_bytes(R, E, w.M, w.I), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(situ.moe_backward_workspace_bytes(R, E, w.M, w.I), dtype=torch.uint8,
                       device=dev)
    state = {}

    def step(marks):
        situ.situ_moe_build_index(ids, E, expert_offsets=off, token_index=tix)
        y, gu, h = situ.situ_moe_grouped_forward_train(x, off, tix, wgu, wd, w.k_eff, wl.BETA,
                                                       wl.LINEAR_BETA, workspace=ws_f)
        if marks:
            marks[0].record()
        state["g"] = situ.situ_moe_grouped_backward(x, off, tix, wgu, wd, gu, h, dy, wl.BETA,
                                                    wl.LINEAR_BETA, workspace=ws_b)

    per_step, (t_fwd, t_bwd) = timed_steps(step, args.steps, args.warmup, flush, world, inner=1)
    state.clear()
    ms = mean(per_step)
    flop_f = 6.0 * R * w.M * w.I
    flop_b = 12.0 * R * w.M * w.I
    out = {"workload": w.name + ", training step (index, forward keeping gu and h, backward)",
           "ms": ms, "forward_ms": mean(t_fwd), "backward_ms": mean(t_bwd),
           "tokens_per_s": w.T / (ms * 1e-3), "routes": R,
           "tflops": (flop_f + flop_b) / (ms * 1e-3) / 1e12,
           "backward_tflops": flop_b / (mean(t_bwd) * 1e-3) / 1e12,
           "tc_frac": (flop_f + flop_b) / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
           "launches_per_step": 4 + 4 + 10}
    del wgu, wd, ws_f, ws_b, dy, x
    torch.cuda.empty_cache()
    return out


def accuracy_stats(got, ref):
    """Error of GPU outputs `got` (a bf16 or float tensor) against the FP64 oracle's `ref`
    (same shape): the largest error over the FFN bound 2e-2 (1 + |ref|) the parity tests
    use, the largest absolute error and the relative RMS error."""
    import numpy as np

    g = got.float().numpy().astype(np.float64).reshape(ref.shape)
    err = np.abs(g - ref)
    return {"reference": "FP64 oracle", "values": int(ref.size),
            "max_err_over_bound": float((err / (2e-2 * (1.0 + np.abs(ref)))).max()),
            "bound": "2e-2 (1 + |ref|)", "max_abs_err": float(err.max()),
            "rms_rel_err": float(np.sqrt((err ** 2).sum() / max(float((ref ** 2).sum()), 1e-300)))}


def ulp_stats(got, ref):
    """Error of bf16 outputs against the FP64 oracle in bf16 ulps of the oracle's value:
    2^(floor(log2 |ref|) - 7) for |ref| >= 2^-126, else 2^-133 (zero included)."""
    import numpy as np

    g = got.float().numpy().astype(np.float64).reshape(ref.shape)
    a = np.abs(ref)
    ulp = np.where(a >= 2.0 ** -126, np.exp2(np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 7),
                   2.0 ** -133)
    e = np.abs(g - ref) / ulp
    return {"reference": "FP64 oracle", "values": int(ref.size), "max_ulp_err": float(e.max()),
            "frac_within_half_ulp": float((e <= 0.5).mean()), "bound": "1 bf16 ulp"}


def cpu_baseline(seconds: float, rows_hint: int = 0, inputs=None):
    """The FP64 oracle (as it stands) on a bounded sample of the dense workload's
    rows: rows/s = tokens/s on the host cores.  inputs: the GPU run's (x, W_gate_up,
    W_down) on the host (generated on the CPU otherwise; the device generator's values
    differ).  Returns the baseline and the oracle's outputs of the sampled rows."""
    import numpy as np
    import torch

    from oracle import Oracle
    from situ_glu_activation_gb300 import workloads as wl

    o = Oracle()
    w = wl.WORKLOADS["dense"]
    x, wgu, wd = inputs if inputs is not None else wl.ffn_inputs(w.M, w.I, w.rows, seed=0)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    xb, wgb, wdb = bits(x), bits(wgu), bits(wd)
    threads = o.num_threads()
    n = rows_hint or max(threads, 8)
    t0 = time.perf_counter()
    ref = o.ffn_forward(xb[:n], wgb, wdb)
    dt = time.perf_counter() - t0
    if not rows_hint and dt < seconds:
        n2 = min(w.rows, max(n, int(n * seconds / max(dt, 1e-3))))
        t0 = time.perf_counter()
        ref = o.ffn_forward(xb[:n2], wgb, wdb)
        dt = time.perf_counter() - t0
        n = n2
    return {"value": n / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"first {n} of the 16384 token rows of the dense workload "
                      f"(FP64 gate_up, SiTU-GLU, down), {dt:.1f} s"}, ref


def route_sample(ids_cpu, n: int, seed: int = 0):
    """A seeded sample of n flat routes (token * k_eff + slot) of ids [T, k_eff] that
    covers every non-empty expert with the first and the last row of its group (in
    expert order, ties by flat index: the expert's smallest and largest flat route),
    then takes a seeded permutation's next routes up to n."""
    import numpy as np

    flat = ids_cpu.contiguous().view(-1).numpy()
    experts, first = np.unique(flat, return_index=True)
    _, last_rev = np.unique(flat[::-1], return_index=True)
    last = flat.size - 1 - last_rev
    chosen = np.unique(np.concatenate([first, last]))
    order = np.random.default_rng(seed).permutation(flat.size)
    rest = order[~np.isin(order, chosen)][: max(0, n - chosen.size)]
    return np.sort(np.concatenate([chosen, rest]))


def host_bytes_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def cpu_baseline_routes(w, x, ids_cpu, wgu_host, wd_host, n_routes: int = 4096):
    """The FP64 oracle's grouped experts (as it stands) on a seeded sample of n_routes
    routes of a grouped workload holding the first and last row of every non-empty
    expert's group, each route with its own expert's weights: the sampled routes run as a grouped call of one slot per
    sampled route.  routes/s is measured; tokens/s = routes/s / k_eff is extrapolated."""
    import numpy as np
    import torch

    from oracle import Oracle

    o = Oracle()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    sample = route_sample(ids_cpu, n_routes, seed=0)
    tokens = torch.from_numpy(sample // w.k_eff)
    ids_s = ids_cpu.contiguous().view(-1)[torch.from_numpy(sample)].view(-1, 1).numpy()
    xs = bits(x.index_select(0, tokens.to(x.device)).cpu())
    t0 = time.perf_counter()
    ref = o.moe_grouped_forward(xs, ids_s, bits(wgu_host), bits(wd_host))
    dt = time.perf_counter() - t0
    experts = int(np.unique(ids_s).size)
    return {"value": sample.size / dt / w.k_eff, "unit": "tokens/s",
            "routes_per_s": sample.size / dt, "cores": o.num_threads(), "kind": "oracle",
            "sample": f"{sample.size} seeded routes of the workload holding the first and last "
                      f"row of all {experts} non-empty experts' groups, each route with its "
                      f"expert's own weights (FP64 grouped experts, "
                      f"per-route loop), {dt:.1f} s; tokens/s = routes/s / {w.k_eff}, "
                      "extrapolated to the workload"}, sample, ref


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import torch

    from oracle import Oracle
    from situ_glu_activation_gb300 import workloads as wl

    o = Oracle()
    w = wl.WORKLOADS["dense"]
    x, wgu, wd = wl.ffn_inputs(w.M, w.I, w.rows, seed=0)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    xb, wgb, wdb = bits(x), bits(wgu), bits(wd)
    rows = args.ref_rows or max(o.num_threads(), 4)
    for i in range(args.warmup):
        o.ffn_forward(xb[i * rows:(i + 1) * rows], wgb, wdb)
    t0 = time.perf_counter()
    for i in range(args.steps):
        r0 = (i * rows) % (w.rows - rows)
        o.ffn_forward(xb[r0:r0 + rows], wgb, wdb)
    dt = time.perf_counter() - t0
    value = args.steps * rows / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.rows, "M": w.M, "I": w.I,
                   "beta": wl.BETA, "linear_beta": wl.LINEAR_BETA,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": o.num_threads(),
                         "kind": "oracle",
                         "sample": f"{rows} token rows per step of the dense workload"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_situ(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import situ_glu_activation_gb300 as situ
    from situ_glu_activation_gb300 import workloads as wl
    from situ_glu_activation_gb300.build import build

    build()
    if args.ffn_two_launches:
        situ.ffn_set_single_launch(False)
    peaks, peak_src = load_peaks()
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush = lambda: flush_buf.fill_(1)
    if args.suite not in ("full", "dense"):
        # One workload alone (profiling runs): a reduced line with that result.
        if args.suite == "act":
            res = bench_act(args, dev, peaks, world, flush)
        elif args.suite == "train":
            res = bench_train(args, dev, peaks, world, flush)
        elif args.suite == "grouped_train":
            res = bench_moe_train(args, dev, peaks, world, flush)
        elif args.suite == "grouped_train_slice":
            res = bench_moe_train(args, dev, peaks, world, flush, "grouped_slice")
        elif args.suite == "mx":
            res = bench_mx(args, dev, peaks, world, flush)
        elif args.suite == "mx_dense":
            res = bench_mx(args, dev, peaks, world, flush, names=())
        else:
            res = bench_moe(args, dev, peaks, world, flush, [args.suite],
                            cpu=rank == 0 and world == 1 and not args.no_cpu_baseline)[args.suite]
        if rank == 0:
            print(json.dumps({"suite": args.suite, "steps": args.steps, "warmup": args.warmup,
                              "result": res, "device_status": situ.device_status(clear=True)}),
                  flush=True)
        return 0

    with ClockSampler(dev.index or 0) as clk:
        dense, w = bench_dense(args, dev, peaks, world, flush)
    clocks = clk.summary()
    ms_max, tokens_all = aggregate(dense["ms"], float(dense["tokens"]), world)
    value = tokens_all / (ms_max * 1e-3)
    e2e_ms, _ = aggregate(dense["e2e_ms"], 0.0, world)

    def with_clocks(fn):
        """A sub-suite's result with the clock record taken while it ran."""
        with ClockSampler(dev.index or 0) as suite_clk:
            res = fn()
        res["clocks"] = suite_clk.summary()
        return res

    act = moe = mx = train = None
    if args.suite == "full":
        check = 64 if rank == 0 and not args.no_cpu_baseline else 0
        act = with_clocks(lambda: bench_act(args, dev, peaks, world, flush, check_rows=check))
        # The oracle's CPU baseline of the grouped workloads: rank 0 of a 1-GPU run.
        cpu_moe = rank == 0 and world == 1 and not args.no_cpu_baseline
        moe = with_clocks(lambda: bench_moe(args, dev, peaks, world, flush,
                                            ["grouped", "k3_decode", "k3_prefill"], cpu=cpu_moe))
        mx = with_clocks(lambda: bench_mx(args, dev, peaks, world, flush))
        train = with_clocks(lambda: bench_train(args, dev, peaks, world, flush))
        train["grouped"] = with_clocks(lambda: bench_moe_train(args, dev, peaks, world, flush))
    status = situ.device_status(clear=True)

    achieved = dense["tflops"]
    digest = source_digest("gemm_kernel.cuh", "gemm.cu", "situ_math.cuh", "situ_ptx.cuh")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max,
        "ms_per_step_median": dense["ms_median"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded x ~ N(0,1), weights ~ N(0, 1/fan_in); no dataset",
        "config": {"workload": w.name, "tokens": w.rows, "M": w.M, "I": w.I,
                   "beta": wl.BETA, "linear_beta": wl.LINEAR_BETA,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write)"},
        "tflops": dense["tflops"],
        "tc_frac": dense["tflops"] / peaks["bf16_tflops"],
        "kernels": {"ffn_fused": {"ms": dense["ms"], "tflops": dense["tflops"]},
                    "two_launches": {"ms": dense["two_launch_ms"],
                                     "ffn_gate_up_situ": {
                                         "ms": dense["gate_up_ms"],
                                         "tflops": dense["gate_up_tflops"],
                                         "frac": dense["gate_up_tflops"] / peaks["bf16_tflops"],
                                         "traffic": profiled_traffic("ffn_gate_up_situ", digest,
                                                                     w.rows)},
                                     "ffn_down": {
                                         "ms": dense["down_ms"],
                                         "tflops": dense["down_tflops"],
                                         "frac": dense["down_tflops"] / peaks["bf16_tflops"],
                                         "traffic": profiled_traffic("ffn_down", digest,
                                                                     w.rows)}}},
        "roofline": {"bound": "tensor",
                     "kernel": ("ffn_gate_up_situ + ffn_down (two launches)"
                                if args.ffn_two_launches else
                                "ffn_fused (gate_up GEMM + SiTU-GLU epilogue + down GEMM, one "
                                "persistent launch)"), "achieved": achieved,
                     "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "peak_source": f"{peak_src} (bf16 dense, burst)",
                     "timing": "CUDA events around the call (its counter reset included)",
                     "traffic": profiled_traffic("ffn_fused", digest, w.rows)},
        "e2e": {"value": tokens_all / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": dense["h2d_bytes"],
                "d2h_bytes_per_step": dense["d2h_bytes"],
                "call": f"situ_ffn_forward_host, pinned host x and y, {E2E_CHUNK_ROWS}-row "
                        "chunks (copies overlap the GEMMs)"},
        "gpu_launches": dense["launches_per_step"] * args.steps,
        "clocks": clocks,
        "device_status": status,
    }
    cost = {"page_remark": "two extra tanh per element, on the order of a percent of the FFN "
                           "(unmeasured remark on the SiTU-GLU chapter page)",
            "fused_gate_up_situ_ms": dense["gate_up_ms"],
            "fused_gate_up_swiglu_ms": dense["swiglu_gate_up_ms"],
            "fused_gate_up_overhead_pct": 100.0 * (dense["gate_up_ms"] / dense["swiglu_gate_up_ms"]
                                                   - 1.0)}
    if act:
        line["act"] = act
        cost["act_situ_ms"] = act["ms"]
        cost["act_swiglu_ms"] = act["swiglu_ms"]
        cost["act_overhead_pct"] = 100.0 * (act["ms"] / act["swiglu_ms"] - 1.0)
    line["situ_cost_vs_swiglu"] = cost
    if moe:
        line["moe"] = moe
    if mx:
        line["mxfp8"] = mx
    if train:
        line["train"] = train
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"], ref = cpu_baseline(args.cpu_seconds, inputs=dense["inputs"])
        # The timed dense call's outputs of the oracle's rows against the oracle's.
        line["accuracy"] = accuracy_stats(dense["y"][: ref.shape[0]], ref)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["situ", "reference"], default="situ")
    ap.add_argument("--suite", default="full",
                    choices=["full", "dense", "act", "grouped", "k3_decode", "k3_prefill",
                             "k3_prefill_slice", "k3_decode_slice", "train", "grouped_train",
                             "grouped_train_slice",
                             "mx", "mx_dense"],
                    help="full: the headline line with every sub-result; dense: the headline "
                         "only; any other name: that workload alone (for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ffn-two-launches", action="store_true",
                    help="run the bf16 dense forward as two launches (for kernel profilers, "
                         "which do not replay its cooperative cluster launch)")
    ap.add_argument("--ref-rows", type=int, default=0, help="oracle rows per reference step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = dist_env()[0]
    if args.gpus != world:
        # One process per GPU: N GPUs are N ranks (torchrun --nproc-per-node N).
        ap.error(f"--gpus {args.gpus} with {world} rank(s): run one rank per GPU, e.g. "
                 f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py "
                 f"--gpus {args.gpus}")
    if args.impl == "reference":
        return run_reference(args)
    return run_situ(args)


if __name__ == "__main__":
    sys.exit(main())
