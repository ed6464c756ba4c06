#!/usr/bin/env python3
"""Benchmark of the W8A8 INT8 projection Linear on one GB300 (or N replicas).

Workload (the attention projection of the MiniMax-H3 DiT at native width):
X BF16 [8192, 5376] ~ N(0,1) with 0.5% of entries x30; four Linears Q, K, V, O
with weights [5376, 5376] ~ N(0, 0.02) quantised per output channel to INT8
with FP32 scales (untimed, offline), BF16 biases ~ N(0, 0.1); seed 1.

One step = the whole hot path over that batch: the per-token activation
quantisation of X, then the four INT8 GEMMs with the fused dequant + bias +
BF16 epilogue.  The metric is INT8 tera-operations per second, 2*M*N*K per
Linear (multiply and add counted separately), whole-job over all ranks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs an independent replica (the projection shards
by token rows with no exchange, so no collective touches the data path), and
rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W8A8 Linear INT8 TOPS at K=5376 and % of GB300 dense INT8 peak"
M, N, K, LINEARS = 8192, 5376, 5376, ("q", "k", "v", "o")
OPS_PER_STEP = 2 * M * N * K * len(LINEARS)
WORKLOAD = ("attn projection: X BF16 [8192,5376] N(0,1)+0.5% x30 outliers; Q,K,V,O W [5376,5376] "
            "N(0,0.02)->per-channel INT8 + FP32 scales; BF16 bias N(0,0.1); seed 1")
L2_FLUSH_BYTES = 512 << 20
# The GB300 datasheet INT8 figure: NVIDIA's GB300 NVL72 specification table
# gives "INT8 Tensor Core" as 23 POPS for the 72-GPU rack, under the table's
# sparsity footnote; per GPU that is about 319 TOPS with 2:4 sparsity and 160
# TOPS dense.  (From the public product page; there is no network here to
# re-check it, so the line also carries the rate measured on the part itself:
# sm_103a has no INT8 tcgen05 MMA, and h3q_probe_mma_s8_tops times its one
# INT8 tensor instruction, mma.sync m16n8k32 s8.)
DATASHEET_INT8 = {"rack_pops": 23.0, "gpus": 72, "sparse_tops_per_gpu": 23e3 / 72,
                  "dense_tops_per_gpu": 23e3 / 72 / 2,
                  "source": "NVIDIA GB300 NVL72 specifications table (public product page): "
                            "INT8 Tensor Core 23 POPS per 72 GPUs, with sparsity; dense = half"}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # the raw samples (the JSON line carries their summary)
        self.path = os.path.join(tempfile.gettempdir(), f"h3q_clocks_rank{index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --- cross-rank aggregation (replicas) ---------------------------------------------

def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time (ms); every rank gets the same value."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tops(total_ms: float, steps: int, world: int) -> float:
    """All ranks' operations over the slowest rank's time: each replica runs
    the full workload, so the job does world x steps x OPS_PER_STEP."""
    return OPS_PER_STEP * steps * world / (total_ms * 1e-3) / 1e12


# --- CPU baseline: the oracle, as it stands, on a bounded sample -------------------

def cpu_oracle_sample(case, qws, target_s: float = 12.0):
    """Time the CPU oracle on token-row chunks of the workload for ~target_s.

    Each chunk runs A2 + A3 + A4 for all four Linears on 256 token rows (the
    weights are quantised once beforehand, as on the GPU side).  Returns
    (TOPS, rows processed, seconds, threads).
    """
    import numpy as np
    from oracle import h3q_oracle as orc
    rows_done, t_total, chunk, start = 0, 0.0, 256, 0
    while t_total < target_s and start < M:
        xb = case.x_bits[start:start + chunk]
        t0 = time.perf_counter()
        for (qw, sw), bb in zip(qws, case.bias_bits):
            orc.linear(xb, qw, sw, bb)
        t_total += time.perf_counter() - t0
        rows_done += xb.shape[0]
        start += chunk
    ops = 2 * rows_done * N * K * len(LINEARS)
    return ops / t_total / 1e12, rows_done, t_total, _cpu_threads()


def _cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def _cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import numpy as np
    import synth
    from oracle import h3q_oracle as orc
    case = synth.attn()
    qws = [orc.quantize_weights(w) for w in case.w]
    times = []
    rows = 0
    chunk = 128
    for i in range(args.warmup + args.steps):
        start = (i * chunk) % M
        xb = case.x_bits[start:start + chunk]
        t0 = time.perf_counter()
        for (qw, sw), bb in zip(qws, case.bias_bits):
            orc.linear(xb, qw, sw, bb)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            rows += xb.shape[0]
    t = sum(times)
    tops = 2 * rows * N * K * len(LINEARS) / t / 1e12
    sample = (f"{chunk} token rows of the workload per step (all four Linears: A2+A3+A4), "
              f"{args.steps} steps")
    line = {"impl": "reference", "metric": METRIC, "value": tops, "unit": "TOPS",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t / len(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "s8", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "linears": 4,
                       "step_rows": chunk},
            "cpu_baseline": {"value": tops, "unit": "TOPS", "cores": _cpu_threads(),
                             "nproc": os.cpu_count(), "cpu_model": _cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": tops, "unit": "TOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --- the GPU arm -------------------------------------------------------------------

def run_gpu(args):
    import numpy as np
    import torch

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    import w8a8_int8_linear_h3q_gb300 as h3q
    import synth
    h3q.load()

    case = synth.attn()
    x_host = torch.from_numpy(case.x_bits.view(np.int16)).view(torch.bfloat16)
    x = x_host.to(dev)
    wq, wsc, bias = [], [], []
    for w, b in zip(case.w, case.bias_bits):
        q, s = h3q.h3q_quantize_weights(torch.from_numpy(w).to(dev))   # offline A1 (untimed)
        wq.append(q)
        wsc.append(s)
        bias.append(torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev))
    xs = torch.empty((M,), dtype=torch.float32, device=dev)
    ys_all = torch.empty((len(LINEARS), M, N), dtype=torch.bfloat16, device=dev)
    ys = [ys_all[i] for i in range(len(LINEARS))]
    workspace = torch.empty((h3q.h3q_linear_workspace_bytes(M, N, K),), dtype=torch.uint8,
                            device=dev)
    flush = torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    gws = torch.empty((h3q.h3q_linear_grouped_workspace_bytes(len(LINEARS), M, N, K),),
                      dtype=torch.uint8, device=dev)

    # events on the launching stream (the library's kernels run there)
    def step(ev=None):
        """One pass of the hot path: the four Linears share X, so one grouped
        call quantises X once (A2) and computes all four outputs in one GEMM
        launch."""
        if ev is not None:
            ev[0].record(stream)
        h3q.h3q_linear_w8a8_grouped(x, wq, wsc, bias, xs=xs, ys=ys, workspace=gws,
                                    stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def step_per_linear(ev=None):
        """The same pass as four calls: Q quantises X into the workspace and runs
        its GEMM; K, V and O reuse the coded activations.  Events between the
        calls time each reuse-mode GEMM call on its own."""
        if ev is not None:
            ev[0].record(stream)
        for i in range(len(LINEARS)):
            h3q.h3q_linear_w8a8(x if i == 0 else None, wq[i], wsc[i], bias[i], xs=xs, y=ys[i],
                                workspace=workspace, stream=stream)
            if ev is not None:
                ev[1 + i].record(stream)

    # A2, the weight-norm pre-pass (which returns at once when the activations
    # alone settle exactness), one single-accumulator GEMM launch for all four
    # Linears and one chunked GEMM launch for all four (which exits at once
    # when no tile needs it), after a memset of the workspace's status words
    launches_per_step = 4

    for _ in range(args.warmup):
        flush.zero_()
        step()
        flush.zero_()
        step_per_linear()
    torch.cuda.synchronize()

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
              for _ in range(args.steps)]
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.5)                             # let the sampler take its first reading
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for s in range(args.steps):
        flush.zero_()                           # L2 flush between timed steps (not timed)
        step(events[s])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()

    step_ms = [e[0].elapsed_time(e[-1]) for e in events]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = whole_job_tops(total_ms, args.steps, world)

    # the per-Linear form of the step (untimed for the headline): its calls
    # give the single GEMM call's time for the roofline
    pl_steps = min(args.steps, 50)
    pl_events = [[torch.cuda.Event(enable_timing=True) for _ in range(1 + len(LINEARS))]
                 for _ in range(pl_steps)]
    for s in range(pl_steps):
        flush.zero_()
        step_per_linear(pl_events[s])
    torch.cuda.synchronize()
    pl_ms = max_over_ranks(sum(e[0].elapsed_time(e[-1]) for e in pl_events), world, dev)
    per_linear_tops = whole_job_tops(pl_ms, pl_steps, world)
    gemm_ms = [e[i].elapsed_time(e[i + 1]) for e in pl_events for i in range(1, len(LINEARS))]
    # A2 inside the call: the Q call (A2 + GEMM) less a reuse-mode call (GEMM)
    q_call_ms = [e[0].elapsed_time(e[1]) for e in pl_events]

    # the grouped call on the activations the timed steps left coded in the
    # workspace: the step's own GEMM launch (all four Linears), with only the
    # small launches around it (a secondary roofline figure)
    gr_ms = []
    for _ in range(pl_steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h3q.h3q_linear_w8a8_grouped(None, wq, wsc, bias, xs=xs, ys=ys, workspace=gws,
                                    stream=stream)
        b.record(stream)
        gr_ms.append((a, b))
    torch.cuda.synchronize()
    grouped_call_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in gr_ms),
                                     world, dev)

    # the same grouped step captured once in a CUDA graph and replayed (a
    # secondary figure; the headline times the eager call)
    graph_ms, graph_note = float("inf"), None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            h3q.h3q_linear_w8a8_grouped(x, wq, wsc, bias, xs=xs, ys=ys, workspace=gws,
                                        stream=side)
            side.synchronize()
            with torch.cuda.graph(graph, stream=side):
                h3q.h3q_linear_w8a8_grouped(x, wq, wsc, bias, xs=xs, ys=ys, workspace=gws,
                                            stream=side)
        torch.cuda.synchronize()
        g_ms = []
        for _ in range(min(args.steps, 20)):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize()
            g_ms.append(a.elapsed_time(b))
        graph_ms = statistics.median(g_ms)
        del graph
    except RuntimeError as e:                      # reported, not fatal
        graph_note = f"capture failed: {e}"
    # every rank takes part in the reduction, whether or not its capture worked
    # (a failed rank sends infinity, so the slowest-rank figure reports it)
    graph_ms = max_over_ranks(graph_ms if graph_note is None else float("inf"), world, dev)
    if graph_ms == float("inf"):
        graph_ms = graph_note or "capture failed on another rank"

    # end to end through the public API with host buffers: one call of
    # h3q_linear_w8a8_grouped_host per step uploads X from pinned host memory,
    # runs the grouped hot path and downloads the four outputs into pinned host
    # memory, all inside the timed region.  The host link is the bound (the
    # outputs are four times the input): the library pipelines row chunks on
    # three streams, the first chunks small so that the downloads start early.
    x_pin = x_host.pin_memory()
    # the four outputs as one [4, M, N] buffer on each side: a chunk's
    # downloads are then one copy
    y_pin_all = torch.empty((len(LINEARS), M, N), dtype=torch.bfloat16).pin_memory()
    y_pin = [y_pin_all[i] for i in range(len(LINEARS))]
    e2e_steps = 0 if args.no_e2e else max(2, min(args.steps, 5))
    E2E_CHUNK = 2048
    h2d_stream, d2h_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    hws = torch.empty((h3q.h3q_linear_w8a8_grouped_host_workspace_bytes(len(LINEARS), M, N, K,
                                                                        E2E_CHUNK),),
                      dtype=torch.uint8, device=dev)

    # the call a user repeats step after step: checked and marshalled once,
    # then each call uploads X, runs the step and downloads the outputs
    e2e_step = h3q.GroupedHostCall(x_pin, wq, wsc, bias, ys_host=y_pin, x_dev=x, xs=xs,
                                   ys_dev=ys, chunk_rows=E2E_CHUNK, workspace=hws,
                                   stream=stream, h2d_stream=h2d_stream, d2h_stream=d2h_stream)

    if e2e_steps:
        e2e_step()
        torch.cuda.synchronize()
    e_ms = 0.0
    for _ in range(e2e_steps):
        flush.zero_()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e_ms += a.elapsed_time(b)
    e_ms = max_over_ranks(e_ms, world, dev)
    e2e_value = whole_job_tops(e_ms, e2e_steps, world) if e2e_steps else None
    h2d_gbs, d2h_gbs = (copy_bandwidth(x, x_pin, ys[0], y_pin[0], stream)
                        if e2e_steps else (None, None))

    # how many tiles of each Linear needed the chunked path (untimed)
    chunked = []
    for i in range(len(LINEARS)):
        h3q.h3q_linear_w8a8(x if i == 0 else None, wq[i], wsc[i], bias[i], xs=xs, y=ys[i],
                            workspace=workspace, stream=stream)
        chunked.append(h3q.h3q_linear_chunked_tiles(workspace, M, K, stream=stream))

    peaks, peak_kind = _peaks()
    int8_probe = h3q.h3q_probe_mma_s8_tops()
    f16_pair_probe = h3q.h3q_probe_mma_f16_pair_tflops(False)
    f16_pair_probe_ss = h3q.h3q_probe_mma_f16_pair_tflops(True)
    gemm_avg_s = statistics.mean(gemm_ms) * 1e-3
    gemm_tflops = 2 * M * N * K / gemm_avg_s / 1e12
    quant_avg_s = time_quantize_act(h3q, x, flush)
    quant_bytes = 2 * M * K + M * K + 4 * M       # BF16 in, INT8 out, FP32 scales
    copy_s = time_same_size_copy(quant_bytes, dev)
    a2_call_s = (statistics.median(q_call_ms) - statistics.median(gemm_ms)) * 1e-3
    a2_call_bytes = 2 * M * K + 2 * M * K + 4 * M  # BF16 in, FP16-coded out, FP32 scales
    traffic, traffic_note = profiled_traffic()
    roofline = {"bound": "tensor", "achieved": gemm_tflops, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": gemm_tflops / peaks["bf16_tflops"],
                "traffic": traffic, "traffic_source": traffic_note,
                # INT8 activations and weights, BF16 output, FP32 scales, BF16 bias
                "algorithmic_bytes_per_launch": M * K + N * K + 2 * M * N + 4 * M + 6 * N,
                # what this design must move at least: the tensor cores read the
                # activations FP16-coded (2 bytes each), as A2 wrote them
                "traffic_design": 2 * M * K + N * K + 2 * M * N + 4 * M + 6 * N,
                "kernel": gemm_kernel_name(h3q),
                "timed_as": "whole reuse-mode Linear call: status memset + weight-norm "
                            "pre-pass + gemm_wide_kernel + the chunked kernel's launch",
                "peak_source": f"{peak_kind} cuBLAS bf16 burst (MEASURED_PEAKS.json)"
                               if peak_kind == "measured" else "fallback 1.9 PFLOP/s bf16",
                "ops_per_launch": 2 * M * N * K,
                # the step's own launch: all four Linears in one gemm_wide_kernel
                "grouped_call": {
                    "achieved": OPS_PER_STEP / (grouped_call_ms * 1e-3) / 1e12,
                    "frac": OPS_PER_STEP / (grouped_call_ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                    "us": grouped_call_ms * 1e3,
                    "timed_as": "whole grouped reuse-mode call (Q, K, V, O): status memset + "
                                "weight-norm pre-pass + one gemm_wide_kernel launch + the "
                                "chunked kernel's launch"}}
    line = {"metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "linears": 4,
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "step": "h3q_linear_w8a8_grouped: A2 once, one GEMM launch for Q, K, V, O",
                       "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MB write)",
                       "chunked_tiles_per_linear": chunked,
                       "tiles_per_linear": -(-M // 128) * -(-N // 256)},
            "roofline": roofline,
            "pct_of_dense_int8_peak": 100.0 * value / int8_probe,
            "pct_of_datasheet_dense_int8": 100.0 * value / DATASHEET_INT8["dense_tops_per_gpu"],
            "dense_int8_peak": {"measured": int8_probe, "unit": "TOPS",
                                "measured_by": "h3q_probe_mma_s8_tops: mma.sync m16n8k32 s8, "
                                               "the one INT8 tensor instruction of sm_103a, 8 "
                                               "independent chains per warp, 32 warps per SM, "
                                               "CUDA events",
                                "datasheet": DATASHEET_INT8,
                                "note": "this path computes the exact INT8 products on the "
                                        "FP16 tensor pipe instead (no INT8 tcgen05 MMA on "
                                        "sm_103a); its roofline is the measured BF16 peak"},
            # the ceiling of the instruction the GEMM issues, measured alone: the
            # tensor-pipe share of the GEMM and of the step read against it
            "instruction_peak": {"instruction": "tcgen05.mma.cta_group::2.kind::f16, "
                                                "M = N = 256, K = 16, A in TMEM, B in shared "
                                                "memory (the hot GEMM's form)",
                                 "measured_tflops": f16_pair_probe,
                                 "a_in_smem_tflops": f16_pair_probe_ss,
                                 "measured_by": "h3q_probe_mma_f16_pair_tflops: one CTA pair "
                                                "per two SMs issuing MMAs back to back over "
                                                "resident operands, CUDA events",
                                 "gemm_frac": gemm_tflops / f16_pair_probe,
                                 "step_frac": value / f16_pair_probe},
            "kernels": {"legacy_mma_sync_s8_tops": legacy_tops(h3q, x, wq[0], wsc[0], bias[0], dev),
                        "quantize_act_us": quant_avg_s * 1e6,
                        "quantize_act_gbs": quant_bytes / quant_avg_s / 1e9,
                        "quantize_act_hbm_frac": quant_bytes / quant_avg_s / 1e9 / peaks["hbm_gbs"],
                        "quantize_act_timing": "steady state: back-to-back launches over "
                                               "rotating copies of X and outputs (> 4x L2); "
                                               "h3q_quantize_act launches with programmatic "
                                               "dependent launch, so each launch's ramp "
                                               "overlaps the previous one's tail (the "
                                               "same-size torch copy does not)",
                        "same_size_copy_us": copy_s * 1e6,
                        "same_size_copy_hbm_frac": quant_bytes / copy_s / 1e9 / peaks["hbm_gbs"],
                        "quantize_act_frac_of_same_size_copy": copy_s / quant_avg_s,
                        "quantize_act_in_call_us": a2_call_s * 1e6,
                        "quantize_act_in_call_hbm_frac":
                            a2_call_bytes / a2_call_s / 1e9 / peaks["hbm_gbs"] if a2_call_s > 0
                            else None,
                        "gemm_us_per_linear": gemm_avg_s * 1e6,
                        "per_linear_step_tops": per_linear_tops,
                        "step_graph_replay_ms": graph_ms,
                        "step_graph_replay_tops": OPS_PER_STEP / (graph_ms * 1e-3) / 1e12
                        if isinstance(graph_ms, float) else None,
                        "per_linear_step_ms": pl_ms / pl_steps,
                        "gemm_tops": gemm_tflops},
            "e2e": {"value": e2e_value, "unit": "TOPS", "ms_per_step":
                    e_ms / e2e_steps if e2e_steps else None,
                    "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
                    "api": "GroupedHostCall: h3q_linear_w8a8_grouped_host with its arguments "
                           "checked once (pinned host X in, pinned host outputs out; "
                           "synchronises)",
                    "overlap": f"row chunks ramping from {E2E_CHUNK // 4} to {E2E_CHUNK} rows: "
                               "H2D, grouped call and D2H pipelined on three streams",
                    "h2d_bytes_per_step": 2 * M * K,
                    "d2h_bytes_per_step": 2 * M * N * len(LINEARS)},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks}
    if not args.no_large:
        del gws, workspace
        torch.cuda.empty_cache()
        for name in ("fc1", "fc2"):
            for k, v in time_large_linear(h3q, synth, name, dev, flush, peaks).items():
                line["kernels"][f"{name}_{k}"] = v
            torch.cuda.empty_cache()
        line["kernels"].update(time_sweep(h3q, synth, dev, local, peaks))
        torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        qws = [(q.cpu().numpy(), s.cpu().numpy()) for q, s in zip(wq, wsc)]
        tops, rows, secs, thr = cpu_oracle_sample(case, qws)
        line["cpu_baseline"] = {"value": tops, "unit": "TOPS", "cores": thr,
                                "nproc": os.cpu_count(), "cpu_model": _cpu_model(),
                                "kind": "oracle",
                                "sample": f"{rows} token rows x 4 Linears (A2+A3+A4), {secs:.1f} s"}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def time_large_linear(h3q, synth, name, dev, flush, peaks, reps=5):
    """One fc1 or fc2 Linear at full size (device-drawn inputs of the
    workload's distributions): median of `reps` CUDA-event timings, L2
    flushed before each, of the whole call from BF16 X (A2 + A3 + A4) and of
    a reuse-mode call (the GEMM with its epilogue, on the coded activations
    the previous call left in the workspace)."""
    import torch
    x, w, b = synth.device_case(name, dev)
    qw, sw = h3q.h3q_quantize_weights(w)          # offline A1 (untimed)
    del w
    Mc, Kc = x.shape
    Nc = qw.shape[0]
    xs = torch.empty((Mc,), dtype=torch.float32, device=dev)
    y = torch.empty((Mc, Nc), dtype=torch.bfloat16, device=dev)
    ws = torch.empty((h3q.h3q_linear_workspace_bytes(Mc, Nc, Kc),), dtype=torch.uint8,
                     device=dev)

    def call(src):
        h3q.h3q_linear_w8a8(src, qw, sw, b, xs=xs, y=y, workspace=ws)

    def med_us(src):
        ts = []
        for _ in range(reps):
            flush.zero_()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call(src)
            e.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(e) * 1e3)
        return statistics.median(ts)

    for _ in range(2):
        call(x)
    torch.cuda.synchronize()
    t_call = med_us(x)
    call(x)
    t_gemm = med_us(None)
    ops = 2 * Mc * Nc * Kc
    out = {"shape": [Mc, Nc, Kc], "gemm_us": t_gemm, "gemm_tops": ops / t_gemm / 1e6,
           "gemm_frac": ops / t_gemm / 1e6 / peaks["bf16_tflops"],
           "call_us": t_call, "call_tops": ops / t_call / 1e6,
           "call_frac": ops / t_call / 1e6 / peaks["bf16_tflops"],
           "checkpointed_tiles": h3q.h3q_linear_checkpointed_tiles(ws, Mc, Kc),
           "chunked_tiles": h3q.h3q_linear_chunked_tiles(ws, Mc, Kc)}
    del x, qw, sw, b, xs, y, ws
    return out


def time_sweep(h3q, synth, dev, local, peaks, passes=2):
    """The full 300-Linear sweep: 50 blocks, each with its own seeded weights
    (17.3 GB of INT8 weights resident), M = 75647 tokens.  A block is Q, K, V,
    O as one grouped call on X5 [M, 5376], FC1 on X5 and FC2 on X21
    [M, 21504], each call quantising its BF16 input (A2 included); the blocks
    are not chained.  One untimed pass, then `passes` passes, each timed whole
    with CUDA events, clocks sampled meanwhile.  The inputs are far larger than
    L2, so no flush is needed between passes."""
    import torch
    M = synth.SWEEP_M
    W5, W21 = synth.H3_WIDTH, synth.H3_MLP_WIDTH
    xs_bf = {K: synth.sweep_x(K, dev) for K in (W5, W21)}
    t0 = time.perf_counter()
    blocks = []
    for blk in range(synth.H3_BLOCKS):
        lin = []
        for j in range(len(synth.SWEEP_LINEARS)):
            w, bias = synth.sweep_weight(blk, j, dev)
            q, sc = h3q.h3q_quantize_weights(w)     # offline A1 (untimed)
            del w
            lin.append((q, sc, bias))
        blocks.append(lin)
    setup_s = time.perf_counter() - t0
    weight_bytes = sum(q.numel() for lin in blocks for q, _, _ in lin)
    xs = torch.empty((M,), dtype=torch.float32, device=dev)
    ya = [torch.empty((M, W5), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    y1 = torch.empty((M, W21), dtype=torch.bfloat16, device=dev)
    y2 = torch.empty((M, W5), dtype=torch.bfloat16, device=dev)
    wsa = torch.empty((h3q.h3q_linear_grouped_workspace_bytes(4, M, W5, W5),), dtype=torch.uint8,
                      device=dev)
    ws1 = torch.empty((h3q.h3q_linear_workspace_bytes(M, W21, W5),), dtype=torch.uint8,
                      device=dev)
    ws2 = torch.empty((h3q.h3q_linear_workspace_bytes(M, W5, W21),), dtype=torch.uint8,
                      device=dev)

    def sweep_pass():
        for lin in blocks:
            att = lin[:4]
            h3q.h3q_linear_w8a8_grouped(xs_bf[W5], [a[0] for a in att], [a[1] for a in att],
                                        [a[2] for a in att], xs=xs, ys=ya, workspace=wsa)
            q, sc, bias = lin[4]
            h3q.h3q_linear_w8a8(xs_bf[W5], q, sc, bias, xs=xs, y=y1, workspace=ws1)
            q, sc, bias = lin[5]
            h3q.h3q_linear_w8a8(xs_bf[W21], q, sc, bias, xs=xs, y=y2, workspace=ws2)

    sweep_pass()
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    ms = []
    for _ in range(passes):
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        sweep_pass()
        e.record()
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(e))
    clocks = clk.stop()
    ops = synth.H3_BLOCKS * sum(2 * M * n * k for _, n, k in synth.SWEEP_LINEARS)
    t = statistics.median(ms)
    del blocks, xs_bf, ya, y1, y2, wsa, ws1, ws2
    return {"sweep_total_ms": t, "sweep_passes_ms": ms, "sweep_tops": ops / t / 1e9,
            "sweep_frac": ops / t / 1e9 / peaks["bf16_tflops"],
            "sweep_linears": synth.H3_BLOCKS * len(synth.SWEEP_LINEARS),
            "sweep_weight_bytes": weight_bytes, "sweep_setup_s": setup_s,
            "sweep_clocks": clocks,
            "sweep_note": "50 blocks x (Q,K,V,O grouped + FC1 + FC2), distinct weights per "
                          "block, M=75647, every call from BF16 X (A2 included); timed whole, "
                          "not extrapolated"}


def copy_bandwidth(x, x_pin, y, y_pin, stream, reps=5):
    """Pinned host<->device copy rates (GB/s) of the bench's own buffers, alone."""
    import torch
    out = []
    for dst, src in ((x, x_pin), (y_pin, y)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        out.append(reps * src.numel() * src.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9)
    return out[0], out[1]


def gemm_kernel_name(h3q) -> str:
    return "gemm_wide_kernel"


# The dominant kernel's DRAM traffic per launch (dram__bytes_read.sum +
# dram__bytes_write.sum) on the attn Linear, from one ncu capture (its summary
# is committed under profiles/, named for the kernel and workload), with the
# SHA-256 of the kernel's sources when it was taken.  It is reported only while
# those sources are unchanged: the files that compile into the kernel (the
# C-ABI header declares nothing it uses).
WIDE_SOURCES = ["w8a8_int8_linear_h3q_gb300/csrc/h3q_gemm_wide.cu",
                "w8a8_int8_linear_h3q_gb300/csrc/h3q_tc_ptx.cuh",
                "w8a8_int8_linear_h3q_gb300/csrc/h3q_epilogue.cuh",
                "w8a8_int8_linear_h3q_gb300/csrc/h3q_internal.cuh"]
WIDE_TRAFFIC = {"bytes_per_launch": 128485888 + 74615552,
                "source_sha256": "62e908619aed333261a4a233907ea825ceb8eb70a576b00d5e32bab187b1e980",
                "capture": "ncu --set full, one reuse-mode gemm_wide_kernel launch, attn Linear "
                           "8192x5376x5376 (python bench.py --kernel-case attn --steps 3 "
                           "--warmup 3; profiles/gemm_wide_attn_8192x5376x5376.md)"}


def wide_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in WIDE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic():
    """(bytes per launch, note) of the last ncu capture, or (None, why)."""
    if WIDE_TRAFFIC["source_sha256"] != wide_sources_sha256():
        return None, "kernel changed since the ncu capture"
    return WIDE_TRAFFIC["bytes_per_launch"], WIDE_TRAFFIC["capture"]


def time_quantize_act(h3q, x, flush, launches=36):
    """Average device time of A2 alone (BF16 -> INT8 + scales) in steady
    state: back-to-back launches between two CUDA events, rotating over copies
    of X (and of the outputs) that together exceed L2 by far, so every launch
    reads its X from DRAM and finds the previous launch's outputs dirty in L2,
    as in a stream of layers.  (A write flush before a single launch would
    instead leave L2 full of the flush buffer's dirty lines, whose write-back
    the short kernel would pay for; timing single launches from the host would
    add the launch latency.)"""
    import torch
    copies = max(2, -(-L2_FLUSH_BYTES // (3 * x.numel())))   # inputs + outputs: 4x L2 or more
    xs_in = [x.clone() for _ in range(copies)]
    outs = [(torch.empty((M, K), dtype=torch.int8, device=x.device),
             torch.empty((M,), dtype=torch.float32, device=x.device)) for _ in range(copies)]
    for i in range(copies):
        h3q.h3q_quantize_act(xs_in[i], *outs[i])
    flush.zero_()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(launches):
        h3q.h3q_quantize_act(xs_in[i % copies], *outs[i % copies])
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / launches * 1e-3


def time_same_size_copy(nbytes, dev, launches=36):
    """Steady-state time of a plain device copy moving `nbytes` (half read,
    half written), rotating over buffers that together exceed L2 by far, as
    time_quantize_act does: the rate a kernel of that size can reach, against
    which the whole-GPU copy peak (measured on gigabytes) overstates it."""
    import torch
    half = nbytes // 2
    copies = max(2, -(-L2_FLUSH_BYTES // nbytes))
    src = [torch.ones((half,), dtype=torch.uint8, device=dev) for _ in range(copies)]
    dst = [torch.empty((half,), dtype=torch.uint8, device=dev) for _ in range(copies)]
    for i in range(copies):
        dst[i].copy_(src[i])
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(launches):
        dst[i % copies].copy_(src[(i + 1) % copies])
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / launches * 1e-3


def legacy_tops(h3q, x, wq, wsc, bias, dev, reps=5):
    """The same GEMM + epilogue on the legacy mma.sync INT8 path (Q weights)."""
    import torch
    xq, xs = h3q.h3q_quantize_act(x)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    for _ in range(2):
        h3q.h3q_linear_w8a8_mma_sync(xq, xs, wq, wsc, bias, y=y)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        h3q.h3q_linear_w8a8_mma_sync(xq, xs, wq, wsc, bias, y=y)
    b.record()
    torch.cuda.synchronize()
    return 2 * M * N * K * reps / (a.elapsed_time(b) * 1e-3) / 1e12


CONFIG_TABLE = ("tiny", "attn", "fc1", "fc2", "image_qkv", "image_gate_up", "image_down",
                "sweep_block")


def run_sweep_block(h3q, synth, dev, flush, steps, warmup, peaks):
    """One block of the 300-Linear sweep at M = 75647 tokens (device-generated
    inputs, block 0): Q, K, V, O as one grouped call, then FC1 and FC2, each
    from BF16 X.  The 50 blocks differ only in their weights, so the sweep's
    time is 50 block times."""
    import statistics
    import torch
    xs_bf = {K: synth.sweep_x(K, dev) for K in (synth.H3_WIDTH, synth.H3_MLP_WIDTH)}
    lin = []
    for j, (_, N, K) in enumerate(synth.SWEEP_LINEARS):
        w, b = synth.sweep_weight(0, j, dev)
        q, sc = h3q.h3q_quantize_weights(w)
        del w
        lin.append((q, sc, b, N, K))
    M = synth.SWEEP_M
    attn = lin[:4]
    xs = torch.empty((M,), dtype=torch.float32, device=dev)
    ya = [torch.empty((M, attn[0][3]), dtype=torch.bfloat16, device=dev) for _ in attn]
    gws = torch.empty((h3q.h3q_linear_grouped_workspace_bytes(4, M, attn[0][3], attn[0][4]),),
                      dtype=torch.uint8, device=dev)
    mlp = []
    for q, sc, b, N, K in lin[4:]:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        ws = torch.empty((h3q.h3q_linear_workspace_bytes(M, N, K),), dtype=torch.uint8,
                         device=dev)
        mlp.append((q, sc, b, N, K, y, ws))

    def block():
        h3q.h3q_linear_w8a8_grouped(xs_bf[synth.H3_WIDTH], [a[0] for a in attn],
                                    [a[1] for a in attn], [a[2] for a in attn], xs=xs, ys=ya,
                                    workspace=gws)
        for q, sc, b, N, K, y, ws in mlp:
            h3q.h3q_linear_w8a8(xs_bf[K], q, sc, b, xs=xs, y=y, workspace=ws)

    for _ in range(warmup):
        block()
    torch.cuda.synchronize()
    ts = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        block()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    t = statistics.median(ts)
    ops = sum(2 * M * N * K for _, _, _, N, K in lin)
    return {"workload": "sweep_block", "M": M, "linears": 6, "reps": steps,
            "block_us": t, "block_tops": ops / t / 1e6,
            "block_frac_of_bf16_peak": ops / t / 1e6 / peaks["bf16_tflops"],
            "sweep_50_blocks_ms": 50 * t / 1e3,
            "note": "Q,K,V,O grouped + FC1 + FC2, each from BF16 X (A2 included); "
                    "50 blocks extrapolated from block 0"}


KERNEL_CASES = ("attn", "attn_grouped", "fc1", "fc2", "quantize_act", "image_down",
                "image_qkv_affine")


def run_kernel_case(args):
    """One kernel's workload run on its own, for profiling (ncu) and quick
    timing: `--warmup` untimed calls, then `--steps` calls, each timed with
    CUDA events after an L2 flush, and one line of medians.  attn: a
    reuse-mode attention Linear (8192 x 5376 x 5376); attn_grouped: the
    grouped Q, K, V, O call from BF16 X; fc1 / fc2: reuse-mode calls on
    device-drawn inputs of those workloads; quantize_act: A2 alone on the
    attention X (INT8 out); image_down: a reuse-mode call on the H3-Image down
    projection (4096 x 5376 x 14336, checkpointed tiles); image_qkv_affine: the
    group-wise affine comparison scheme's Linear on the H3-Image fused QKV
    shape (4096 x 21504 x 5376, Q8/g64)."""
    import numpy as np
    import torch
    import w8a8_int8_linear_h3q_gb300 as h3q
    import synth
    h3q.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=dev)
    name = args.kernel_case
    if name in ("fc1", "fc2"):
        x, w, b = synth.device_case(name, dev)
        lin = [(*h3q.h3q_quantize_weights(w), b)]
        del w
    elif name in ("image_down", "image_qkv_affine"):
        case = synth.WORKLOADS["image_down" if name == "image_down" else "image_qkv"]()
        x = torch.from_numpy(case.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        w = torch.from_numpy(case.w[0]).to(dev)
        b = torch.from_numpy(case.bias_bits[0].view(np.int16)).view(torch.bfloat16).to(dev)
        lin = [((*h3q.h3q_quantize_weights_affine(w),) if name == "image_qkv_affine"
                else (*h3q.h3q_quantize_weights(w),)) + (b,)]
        del w, case
    else:
        case = synth.attn()
        x = torch.from_numpy(case.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        n_lin = 4 if name == "attn_grouped" else 1
        lin = []
        for w, bb in list(zip(case.w, case.bias_bits))[:n_lin]:
            q, sc = h3q.h3q_quantize_weights(torch.from_numpy(w).to(dev))
            lin.append((q, sc, torch.from_numpy(bb.view(np.int16)).view(torch.bfloat16).to(dev)))
        del case
    Mc, Kc = x.shape
    Nc = lin[0][0].shape[0]
    xs = torch.empty((Mc,), dtype=torch.float32, device=dev)
    if name == "quantize_act":
        xq = torch.empty((Mc, Kc), dtype=torch.int8, device=dev)
        fn = lambda: h3q.h3q_quantize_act(x, xq, xs)
        ops = None
    elif name == "image_qkv_affine":
        qa, ab, b = lin[0]
        oa = h3q.h3q_linear_affine_w8(x, qa, ab, b)
        fn = lambda: h3q.h3q_linear_affine_w8(x, qa, ab, b, y=oa["y"], status=oa["status"])
        ops = 2 * Mc * Nc * Kc
    elif name == "attn_grouped":
        ys = [torch.empty((Mc, Nc), dtype=torch.bfloat16, device=dev) for _ in lin]
        ws = torch.empty((h3q.h3q_linear_grouped_workspace_bytes(len(lin), Mc, Nc, Kc),),
                         dtype=torch.uint8, device=dev)
        fn = lambda: h3q.h3q_linear_w8a8_grouped(x, [a[0] for a in lin], [a[1] for a in lin],
                                                 [a[2] for a in lin], xs=xs, ys=ys, workspace=ws)
        ops = 2 * Mc * Nc * Kc * len(lin)
    else:
        q, sc, b = lin[0]
        y = torch.empty((Mc, Nc), dtype=torch.bfloat16, device=dev)
        ws = torch.empty((h3q.h3q_linear_workspace_bytes(Mc, Nc, Kc),), dtype=torch.uint8,
                         device=dev)
        h3q.h3q_linear_w8a8(x, q, sc, b, xs=xs, y=y, workspace=ws)       # codes the activations
        fn = lambda: h3q.h3q_linear_w8a8(None, q, sc, b, xs=xs, y=y, workspace=ws)
        ops = 2 * Mc * Nc * Kc
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(args.steps):
        flush.zero_()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(e) * 1e3)
    t = statistics.median(ts)
    print(json.dumps({"kernel_case": name, "M": Mc, "N": Nc, "K": Kc, "median_us": t,
                      "tops": ops / t / 1e6 if ops else None, "calls": args.steps}), flush=True)
    return 0


def run_configs(args):
    """Per-workload table (not the contract line): for each seeded workload,
    one Linear timed with CUDA events, L2 flushed before each rep: GEMM +
    epilogue on activations already coded in the workspace (reuse mode), the
    whole call from BF16 X (A2 + A3 + A4), and the weight-only group-wise
    affine comparison scheme's call on the same X.  Prints one JSON object
    per workload."""
    import numpy as np
    import torch
    import w8a8_int8_linear_h3q_gb300 as h3q
    import synth
    h3q.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peaks, peak_kind = _peaks()
    flush = torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=dev)
    names = args.configs.split(",") if args.configs != "all" else CONFIG_TABLE
    for name in names:
        if name == "sweep_block":
            print(json.dumps(run_sweep_block(h3q, synth, dev, flush, min(args.steps, 10),
                                             args.warmup, peaks)), flush=True)
            torch.cuda.empty_cache()
            continue
        case = synth.WORKLOADS[name]()
        x = torch.from_numpy(case.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
        w_dev = torch.from_numpy(case.w[0]).to(dev)
        wq, wsc = h3q.h3q_quantize_weights(w_dev)
        bias = torch.from_numpy(case.bias_bits[0].view(np.int16)).view(torch.bfloat16).to(dev)
        del case
        Mc, Kc = x.shape
        Nc = wq.shape[0]
        xs = torch.empty((Mc,), dtype=torch.float32, device=dev)
        y = torch.empty((Mc, Nc), dtype=torch.bfloat16, device=dev)
        ws_buf = torch.empty((h3q.h3q_linear_workspace_bytes(Mc, Nc, Kc),), dtype=torch.uint8,
                             device=dev)

        def full():
            h3q.h3q_linear_w8a8(x, wq, wsc, bias, xs=xs, y=y, workspace=ws_buf)

        def reuse():
            h3q.h3q_linear_w8a8(None, wq, wsc, bias, xs=xs, y=y, workspace=ws_buf)

        def med_us(fn, reps):
            ts = []
            for _ in range(reps):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b) * 1e3)
            return statistics.median(ts)

        for _ in range(args.warmup):
            full()
        torch.cuda.synchronize()
        t_full = med_us(full, args.steps)
        full()
        t_gemm = med_us(reuse, args.steps)
        chunked = h3q.h3q_linear_chunked_tiles(ws_buf, Mc, Kc)
        ckpt = h3q.h3q_linear_checkpointed_tiles(ws_buf, Mc, Kc)
        ops = 2 * Mc * Nc * Kc
        # the group-wise affine comparison scheme (weight-only Q8/g64) on the
        # same Linear, from the same BF16 X
        t_aff = None
        if Kc % 64 == 0:
            qa, ab = h3q.h3q_quantize_weights_affine(w_dev)
            oa = h3q.h3q_linear_affine_w8(x, qa, ab, bias)

            def affine():
                h3q.h3q_linear_affine_w8(x, qa, ab, bias, y=oa["y"], status=oa["status"])

            for _ in range(args.warmup):
                affine()
            t_aff = med_us(affine, args.steps)
            del qa, ab, oa
        print(json.dumps({
            "workload": name, "M": Mc, "N": Nc, "K": Kc, "reps": args.steps,
            "gemm_us": t_gemm, "gemm_tops": ops / t_gemm / 1e6,
            "gemm_frac_of_bf16_peak": ops / t_gemm / 1e6 / peaks["bf16_tflops"],
            "call_us": t_full, "call_tops": ops / t_full / 1e6,
            "chunked_tiles": chunked, "tiles": -(-Mc // 128) * -(-Nc // 256),
            "checkpointed_tiles": ckpt,
            "affine_q8_call_us": t_aff,
            "affine_q8_call_tops": ops / t_aff / 1e6 if t_aff else None,
            "peak": f"{peaks['bf16_tflops']} TFLOP/s bf16 burst ({peak_kind})"}), flush=True)
        del x, w_dev, wq, wsc, bias, xs, y, ws_buf
        torch.cuda.empty_cache()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-large", action="store_true",
                    help="skip the fc1 / fc2 Linears and the full 300-Linear sweep")
    ap.add_argument("--configs", default=None,
                    help="instead of the contract line, print a per-workload table: 'all' or "
                         "a comma list of " + ",".join(CONFIG_TABLE))
    ap.add_argument("--kernel-case", default=None, choices=KERNEL_CASES,
                    help="instead of the contract line, run one kernel's workload on its own "
                         "(for profiling): " + ",".join(KERNEL_CASES))
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel_case:
        return run_kernel_case(args)
    if args.configs:
        return run_configs(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
