#!/usr/bin/env python
"""Throughput of the MoE expert block on GB300: forward + backward of one batch.

    python bench.py [--gpus N --steps K --warmup W] [--impl ours|reference]

One step is one pass of the whole block over one batch: route, dispatch,
gate_up GEMM + SwiGLU, down GEMM, combine, then the backward (G scatter, dH GEMM +
SwiGLU backward, dW_down, dXp GEMM, dW_gu, dX gather), through the C ABI. The
headline workload is the largest single-GPU configuration, the long-sequence
gpt-oss-20b-like block (T=65536 tokens, d=2880, E=32 experts, k=4, f=2880, seed 4;
synthetic inputs); the other four seeded configurations (tiny, Qwen3-MoE-like,
gpt-oss-20b-like, skewed load) are measured the same way and reported in the
line's `workloads` record. Rank 0 prints one JSON line.

  value     tokens/s over all ranks, device-timed with CUDA events (L2 flushed
            before every timed step, outside the timed events)
  e2e       the same through the Python API with pinned host inputs copied in and
            Y and dX copied out inside the timed region (uploads and downloads on
            two copy streams)
  roofline  the dominant kernel (largest share of step time): algorithmic work
            per launch / its mean launch time from library-recorded CUDA events,
            against the measured burst bf16 peak (or the HBM copy rate)
  cpu_baseline  the CPU oracle timed on the host cores on a bounded token sample
  --impl reference  times the CPU oracle alone (rank 0), as the reference arm.

Under torchrun (N > 1) every rank runs its own replica of the workload (weak
scaling, no data-path collective); the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "MoE layer tokens/s and grouped-GEMM TFLOPS (% of GB300 bf16 peak), 1 GPU"
UNIT = "tokens/s"
WORKLOAD = "long"     # the largest single-GPU configuration (T=65536, forward+backward)
WORKLOAD_ORDER = ("tiny", "qwen3_moe", "gpt_oss_20b", "skewed", "long")
NOMINAL_BF16_TFLOPS = 2250.0     # GB300 dense bf16, nominal (context beside the measured peak)
L2_FLUSH_BYTES = 256 << 20       # > 129 MB L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_SOURCES = ("moe_expert_layer_route_gb300/csrc/grouped_gemm.cu",
                "moe_expert_layer_route_gb300/csrc/common.cuh")
BW_SOURCES = ("moe_expert_layer_route_gb300/csrc/route_dispatch.cu",
              "moe_expert_layer_route_gb300/csrc/common.cuh")


# ------------------------------------------------------------------ distributed
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int) -> None:
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of the ranks' values (all ranks get it)."""
    if world == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------- helpers
def peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return json.load(fh), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(paths) -> str:
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# fp32 SIMT peak for the router GEMM (plain ALU arithmetic, no tensor cores): 152 SMs x
# 128 fp32 lanes x 2 FLOP per fma x 2.07 GHz maximum SM clock
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
OVERLAPPED = " (overlapped)"


def gemm_bytes(wl: workloads.Workload, training: bool) -> dict:
    """Algorithmic HBM bytes of each grouped GEMM launch: its weights, and its activation
    rows read and written once (A = T*k rows; segment padding not counted)."""
    A, d, f, E = wl.A, wl.d, wl.f, wl.E
    wgu, wdown = E * d * 2 * f * 2, E * f * d * 2
    return {
        "gemm_gate_up_swiglu": wgu + A * d * 2 + A * f * 2 + (A * 2 * f * 2 if training else 0),
        "gemm_down": wdown + A * f * 2 + A * d * 2,
        "gemm_dgrad_h_swiglu_bwd": wdown + A * d * 2 + 2 * A * 2 * f * 2,
        "gemm_wgrad_down": A * f * 2 + A * d * 2 + wdown,
        "gemm_dgrad_x": wgu + A * 2 * f * 2 + A * d * 2,
        "gemm_wgrad_gu": A * d * 2 + A * 2 * f * 2 + wgu,
    }


def router_splits(T: int, d: int, E: int) -> int:
    cells = -(-d // 256) * -(-E // 32)
    return max(1, min(-(-304 // cells), -(-T // 32)))


def kernel_work(wl: workloads.Workload) -> dict:
    """Algorithmic work of one launch of each kernel: ('flop'|'alu_flop'|'byte', amount)."""
    T, d, E, k, f, A = wl.T, wl.d, wl.E, wl.k, wl.f, wl.A
    C = (T + 31) // 32
    return {
        "router_route_count": ("alu_flop", 2 * T * E * d),
        "router_dx": ("alu_flop", 2 * T * E * d),
        "router_dw": ("alu_flop", 2 * T * E * d),
        # the library's token splits of dW_r: about 2 x 152 blocks of 256 columns x 32 experts
        "router_dw_reduce": ("byte", (router_splits(T, d, E) + 1) * E * d * 4),
        "gemm_gate_up_swiglu": ("flop", 4 * A * d * f),
        "gemm_down": ("flop", 2 * A * d * f),
        "gemm_dgrad_h_swiglu_bwd": ("flop", 2 * A * d * f),
        "gemm_wgrad_down": ("flop", 2 * A * d * f),
        "gemm_dgrad_x": ("flop", 4 * A * d * f),
        "gemm_wgrad_gu": ("flop", 4 * A * d * f),
        # bandwidth kernels: bytes the stage must move at least once
        "route_count": ("byte", T * E * 4 + A * 12 + E * C * 4),
        "scan": ("byte", 2 * E * C * 4),
        # the forward's route + count with the scan run by the last block
        "route_count_scan": ("byte", T * E * 4 + A * 12 + 3 * E * C * 4),
        "scatter": ("byte", T * d * 2 + A * d * 2 + A * 16),
        "combine": ("byte", A * d * 2 + A * 8 + T * d * 2),
        "g_scatter": ("byte", T * d * 2 + A * d * 2 + A * 8),
        "g_scatter_router_grad": ("byte", T * d * 2 + 2 * A * d * 2 + A * 12 + T * E * 4),
        "aux_grad": ("byte", 2 * T * E * 4 + T * E * 4),
        "dx_gather": ("byte", A * d * 2 + A * 4 + T * d * 2),
    }


class ClockSampler:
    """nvidia-smi sampled every 50 ms while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict | None:
        if self.proc is None or self.path is None:
            return None
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx = max(mx, float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------- CPU oracle
def oracle_step(oracle, inp_np: dict, n_tok: int, k: int) -> float:
    """Forward (+ backward when the workload has one) of the oracle on the first n_tok
    tokens; returns seconds."""
    t0 = time.perf_counter()
    if inp_np.get("w_router") is not None:  # the fp32 router GEMM in front
        logits = oracle.router_logits(inp_np["x"][:n_tok], inp_np["w_router"])
    else:
        logits = inp_np["logits"][:n_tok]
    ref = oracle.forward(inp_np["x"][:n_tok], logits, inp_np["w_gu"], inp_np["w_down"], k)
    if inp_np["dy"] is not None:
        oracle.backward(inp_np["dy"][:n_tok], ref, inp_np["w_gu"], inp_np["w_down"])
    return time.perf_counter() - t0


def oracle_inputs(inp: workloads.Inputs, backward: bool, w_router=None) -> dict:
    """The workload's inputs as the oracle computes in them (fp64, exact widenings of the
    bf16 values), converted once here rather than expert by expert inside every call."""
    return {"x": inp.x.double().numpy(), "logits": inp.logits.numpy(),
            "w_gu": inp.w_gu.double().numpy(), "w_down": inp.w_down.double().numpy(),
            "dy": inp.dy.double().numpy() if backward else None,
            "w_router": None if w_router is None else w_router.double().numpy()}


def cpu_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except ImportError:
        pass
    return os.cpu_count() or 1


def cpu_baseline(wl, inp, seconds: float, w_router=None) -> dict:
    """The oracle as it stands on a bounded token sample sized to about `seconds`."""
    import oracle
    inp_np = oracle_inputs(inp, wl.backward, w_router)
    n = 16
    oracle_step(oracle, inp_np, n, wl.k)  # the first call pages in its fp64 buffers
    t = oracle_step(oracle, inp_np, n, wl.k)
    while t < seconds / 4 and n < wl.T:
        n = min(wl.T, n * 4)
        t = oracle_step(oracle, inp_np, n, wl.k)
    return {"value": n / t, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": f"first {n} of {wl.T} tokens of the {wl.name} workload, "
                      f"{'forward+backward' if wl.backward else 'forward'}"
                      f"{' with the router GEMM' if w_router is not None else ''} in fp64 numpy, "
                      f"{t:.1f} s"}


# ---------------------------------------------------------------------- our arm
def workload_of(args) -> workloads.Workload:
    wl = workloads.WORKLOADS[args.workload]
    over = {}
    if args.tokens is not None:
        over["T"] = args.tokens
    if args.experts is not None:
        over["E"] = args.experts
    if over:
        desc = wl.description + " with " + ", ".join(f"{k}={v}" for k, v in over.items())
        wl = wl.scaled(description=desc, **over)
    return wl


def gpu_index_of(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0]
    return int(vis) if vis.isdigit() else local_rank


def measure(moe, wl: workloads.Workload, args, K: int, W: int, world: int, dev,
            flush: torch.Tensor, want_graph: bool, want_e2e: bool) -> dict:
    """Device-timed, profiled, graph-replayed and end-to-end steps of one workload.

    A step is one pass of the whole block (forward, and the backward when the workload
    has one) over one batch through the C ABI. Returns the measurements as a dict."""
    inp = workloads.make_inputs(wl, with_dy=True)
    x, logits = inp.x.to(dev), inp.logits.to(dev)
    w_router = workloads.make_router_weight(wl).to(dev) if args.router_gemm else None
    dw_router = torch.empty(w_router.shape, dtype=torch.float32, device=dev) \
        if w_router is not None else None
    w_gu, w_down, dy = inp.w_gu.to(dev), inp.w_down.to(dev), inp.dy.to(dev)
    s = moe.shape(wl.T, wl.d, wl.E, wl.k, wl.f)
    ws = moe.new_workspace(s, wl.backward, dev)
    scratch = moe.new_scratch(s, dev)
    y = torch.empty_like(x)
    grads = (torch.empty_like(x), torch.empty_like(w_gu), torch.empty_like(w_down))
    router_grad = args.router_grad or args.aux_loss
    dlogits = torch.empty_like(logits) if router_grad else None
    sel_bias = torch.from_numpy(workloads.zipf_bias(wl.E)).to(dev) if args.selection_bias else None
    aux = torch.empty(2 * wl.E + 1, dtype=torch.float32, device=dev) if args.aux_loss else None
    views = moe.workspace_views(s, wl.backward, ws)
    r_scratch = torch.empty(max(16, moe.lib().moe_router_backward_scratch_size(s)),
                            dtype=torch.uint8, device=dev) if w_router is not None else None

    def run_step(x, logits, dy, y, dx):
        """One step through the library on the given input and output tensors (the
        workspace, scratch and weight gradients are shared)."""
        if w_router is not None:  # logits computed from x by the router GEMM
            moe.forward_router(x, w_router, w_gu, w_down, wl.k, training=wl.backward, ws=ws,
                               y=y, logits=logits, bias=sel_bias, aux_stats=aux)
        else:
            moe.forward(x, logits, w_gu, w_down, wl.k, training=wl.backward, ws=ws, y=y,
                        bias=sel_bias, aux_stats=aux)
        if wl.backward:
            moe.backward(s, dy, w_gu, w_down, ws, scratch, out=(dx, grads[1], grads[2]),
                         dlogits=dlogits)
            if aux is not None:
                moe.aux_loss_backward(s, logits, views["counts"], 0.01, dlogits)
            if w_router is not None and dlogits is not None:  # through the router GEMM
                moe.router_backward(s, x, w_router, dlogits, dx, dw_router, r_scratch)

    def step():
        run_step(x, logits, dy, y, grads[0])

    for _ in range(W):
        step()
    torch.cuda.synchronize()
    moe.check_device_status(ws)
    moe.check_device_status(scratch)

    # ---- device-timed region (no instrumentation inside: the library's per-launch
    # events of the profiled pass below would add their own gaps to the step)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    launches0 = moe.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_index_of(dev.index or 0)) as clk:
        for i in range(K):
            flush.zero_()
            starts[i].record()
            step()
            ends[i].record()
        torch.cuda.synchronize()
    barrier(world)
    launches = moe.launch_count() - launches0
    moe.check_device_status(ws)
    moe.check_device_status(scratch)
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    tokens_all = sum_over_ranks(wl.T, world, dev)

    # ---- end to end with host buffers, right after the device-timed region so that
    # both see the GPU in the same state (clocks under the power cap drift as it warms)
    e2e = None
    if want_e2e:
        e2e = measure_e2e(wl, inp, run_step, x, logits, dy, w_router is not None, K, world,
                          dev, tokens_all)

    # ---- profiled pass: the same K steps with an event pair around every launch, for
    # the per-kernel times, shares and the dominant kernel's roofline
    moe.profile_start(capacity=K * 24)
    for i in range(K):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    records = moe.profile_stop(capacity=K * 24)
    moe.check_device_status(ws)
    moe.check_device_status(scratch)

    # ---- per-kernel times and the roofline of the dominant kernel
    per = {}
    for name, t in records:
        per.setdefault(name, []).append(t)
    work = kernel_work(wl)
    pk, peak_src = peaks()
    bf16_peak = pk["bf16_tflops"]
    stages = {}
    # a launch the library ran on its side stream beside others is named "<kernel>
    # (overlapped)": its events span the kernels it overlaps, so it takes no share and
    # cannot be the dominant kernel; its time is an upper bound
    serial = {n: ts for n, ts in per.items() if not n.endswith(OVERLAPPED)}
    serial_total = max(sum(sum(v) for v in serial.values()), 1e-9)
    for name, ts in per.items():
        base = name[:-len(OVERLAPPED)] if name.endswith(OVERLAPPED) else name
        kind, amount = work.get(base, ("byte", 0))
        mean = statistics.mean(ts)
        entry = {"launches_per_step": len(ts) / K, "ms": mean,
                 "share": 0.0 if name not in serial else sum(ts) / serial_total}
        if name not in serial:
            entry["overlapped"] = True
        if amount:
            if kind == "flop":
                entry.update(achieved=amount / (mean * 1e-3) / 1e12, unit="TFLOP/s",
                             frac=amount / (mean * 1e-3) / 1e12 / bf16_peak)
            elif kind == "alu_flop":
                entry.update(achieved=amount / (mean * 1e-3) / 1e12, unit="TFLOP/s fp32",
                             frac=amount / (mean * 1e-3) / 1e12 / FP32_ALU_TFLOPS)
            else:
                entry.update(achieved=amount / (mean * 1e-3) / 1e9, unit="GB/s",
                             frac=amount / (mean * 1e-3) / 1e9 / pk["hbm_gbs"])
        stages[name] = entry
    dom = max(serial, key=lambda n: sum(serial[n]))
    dkind, damount = work[dom]
    dmean = statistics.mean(per[dom])
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        # {workload description: {kernel: {bytes_per_launch, source_hash, ...}}}
        with open(tpath) as fh:
            tr = json.load(fh).get(wl.description, {}).get(dom)
        srcs = GEMM_SOURCES if dom.startswith("gemm") else BW_SOURCES
        if tr and tr.get("source_hash") == source_hash(srcs):
            traffic = tr.get("bytes_per_launch")
    if dkind == "flop":
        ach = damount / (dmean * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": bf16_peak,
                "unit": "TFLOP/s", "frac": ach / bf16_peak,
                "traffic": traffic, "kernel": dom,
                "peak_source": f"{peak_src} bf16_tflops (cuBLAS burst)",
                "frac_of_nominal_dense": ach / NOMINAL_BF16_TFLOPS}
    else:
        ach = damount / (dmean * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": ach / pk["hbm_gbs"], "traffic": traffic, "kernel": dom,
                "peak_source": f"{peak_src} hbm_gbs (copy)"}
    gemm_names = [n for n in per if n.startswith("gemm")]
    gemm_flop = sum(work[n][1] * len(per[n]) for n in gemm_names) / K
    gemm_ms = sum(sum(per[n]) for n in gemm_names) / K
    gemm_tflops = gemm_flop / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else 0.0
    # the whole step against its roofline: the slower of its FLOPs at the bf16 peak and
    # its algorithmic bytes (every stage's, GEMMs included) at the HBM copy rate
    gb = gemm_bytes(wl, wl.backward)
    step_bytes = 0.0
    for n, ts in serial.items():
        kind, amount = work.get(n, ("byte", 0))
        step_bytes += (gb[n] if n in gb else amount if kind == "byte" else 0) * len(ts)
    step_bytes /= K
    t_flop = gemm_flop / (bf16_peak * 1e12) * 1e3
    t_bytes = step_bytes / (pk["hbm_gbs"] * 1e9) * 1e3
    step_roofline = {"flop": gemm_flop, "bytes": step_bytes, "t_flop_ms": t_flop,
                     "t_bytes_ms": t_bytes, "bound": "tensor" if t_flop >= t_bytes else "hbm",
                     "frac": max(t_flop, t_bytes) / ms}
    counts = views["counts"].cpu().numpy()
    experts = {"max": int(counts.max()), "min": int(counts.min()),
               "empty": int((counts == 0).sum())}

    # ---- the same step captured once in a CUDA graph and replayed (the calls allocate
    # nothing and never synchronise, so they capture): device time without launch gaps
    graph = None
    if want_graph:
        gstream = torch.cuda.Stream(device=dev)
        gstream.wait_stream(torch.cuda.current_stream(dev))
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=gstream):
            step()
        cg.replay()
        torch.cuda.synchronize()
        gs = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ge = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        barrier(world)
        for i in range(K):
            flush.zero_()
            gs[i].record()
            cg.replay()
            ge[i].record()
        torch.cuda.synchronize()
        gms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(gs, ge)), world,
                             dev)
        graph = {"ms_per_step": gms, "value": tokens_all / (gms * 1e-3), "unit": UNIT}
        del cg

    return {"wl": wl, "ms": ms, "value": tokens_all / (ms * 1e-3),
            "ms_median": statistics.median(step_ms), "stages": stages, "roofline": roof,
            "gemm_tflops": gemm_tflops, "gemm_flop": gemm_flop, "step_roofline": step_roofline,
            "experts": experts, "graph": graph, "e2e": e2e, "launches": launches,
            "clocks": clk.summary(), "router_grad": router_grad,
            "w_router": None if w_router is None else w_router.cpu(), "inp": inp}


def measure_e2e(wl, inp, run_step, x, logits, dy, router_gemm: bool, K: int, world: int, dev,
                tokens_all: float) -> dict:
    """End to end through the Python API with host buffers: every step uploads its inputs
    from pinned host memory and downloads its results (Y, and dX when the workload has a
    backward). Uploads run on one copy stream and downloads on another, so the two
    directions overlap each other and the kernels; four device buffer sets let step i+1's
    upload and the downloads of steps i-1 and i-2 run beside step i (events order each
    set's reuse). Host-side copy rates vary with what else the host is doing (one 755 MB
    download took 4.4 ms and, in the same run, 32.7 ms), so the downloads get three steps
    of slack before their set is needed again."""
    nset = 4
    ke = max(4, min(K, 50))
    hx = inp.x.pin_memory()
    hl = inp.logits.pin_memory()
    hdy = inp.dy.pin_memory() if wl.backward else None
    hy = [torch.empty_like(hx).pin_memory() for _ in range(nset)]
    hdx = [torch.empty_like(hx).pin_memory() for _ in range(nset)] if wl.backward else None
    dsets = [(torch.empty_like(x), torch.empty_like(logits),
              torch.empty_like(dy) if wl.backward else None, torch.empty_like(x),
              torch.empty_like(x) if wl.backward else None) for _ in range(nset)]
    comp = torch.cuda.current_stream(dev)
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    loaded = [torch.cuda.Event() for _ in range(nset)]      # the set's inputs are on the device
    computed = [torch.cuda.Event() for _ in range(nset)]    # the set's step has run
    drained = [torch.cuda.Event() for _ in range(nset)]     # the set's results are on the host
    used = [False] * nset

    def upload(i):
        b = i % nset
        bx, bl, bdy, _, _ = dsets[b]
        with torch.cuda.stream(up):
            if used[b]:
                up.wait_event(computed[b])      # the set's previous step read its inputs
            bx.copy_(hx, non_blocking=True)
            if not router_gemm:
                bl.copy_(hl, non_blocking=True)
            if wl.backward:
                bdy.copy_(hdy, non_blocking=True)
            loaded[b].record(up)

    def compute(i):
        b = i % nset
        bx, bl, bdy, by, bdx = dsets[b]
        comp.wait_event(loaded[b])
        if used[b]:
            comp.wait_event(drained[b])         # the set's previous results have left
        run_step(bx, bl, bdy, by, bdx)
        computed[b].record(comp)
        used[b] = True

    def download(i):
        b = i % nset
        _, _, _, by, bdx = dsets[b]
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            hy[b].copy_(by, non_blocking=True)
            if wl.backward:
                hdx[b].copy_(bdx, non_blocking=True)
            drained[b].record(down)

    def run(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)
            download(i)

    run(3)
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(gpu_index_of(dev.index or 0)) as clk:
        t0 = time.perf_counter()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(comp)
        up.wait_event(ev0)
        down.wait_event(ev0)
        run(ke)
        comp.wait_stream(down)          # the last download is part of the timed region
        ev1.record(comp)
        torch.cuda.synchronize()
        wall = (time.perf_counter() - t0) * 1e3 / ke
    ev_ms = ev0.elapsed_time(ev1) / ke
    e2e_ms = max_over_ranks(max(ev_ms, wall), world, dev)
    h2d = hx.numel() * 2 + (hl.numel() * 4 if not router_gemm else 0) + \
        (hdy.numel() * 2 if wl.backward else 0)
    d2h = hx.numel() * 2 * (2 if wl.backward else 1)

    # copy rates alone (no kernels beside them), for reading the e2e figure
    def rate(fn, nbytes):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(3):
            fn()
        b.record()
        torch.cuda.synchronize()
        return 3 * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9

    bx0 = dsets[0][0]
    h2d_gbs = rate(lambda: bx0.copy_(hx, non_blocking=True), hx.numel() * 2)
    d2h_gbs = rate(lambda: hy[0].copy_(bx0, non_blocking=True), hx.numel() * 2)
    return {"value": tokens_all / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "ms_per_step_events": ev_ms, "ms_per_step_wall": wall,
            "copy_gbs_alone": {"h2d": h2d_gbs, "d2h": d2h_gbs}, "clocks": clk.summary(),
            "copies": "uploads and downloads on two copy streams, four device buffer sets: "
                      "both directions overlap each other and the neighbouring steps' kernels"}


def passes_of(wl, args, router_grad: bool) -> str:
    return (("forward+backward" if wl.backward else "forward")
            + (" + fp32 router GEMM (logits from x)" if args.router_gemm else "")
            + (" + router-logit gradient" if router_grad and wl.backward else "")
            + (" + router GEMM gradient (dW_r, dX)" if args.router_gemm and router_grad
               and wl.backward else "")
            + (" + selection bias (Zipf)" if args.selection_bias else "")
            + (" + load-balancing statistics and gradient" if args.aux_loss else ""))


def summary_of(m: dict) -> dict:
    """The figures of one workload for the line's `workloads` record."""
    wl = m["wl"]
    gemms = {n: {"ms": v["ms"], "tflops": v.get("achieved"), "frac": v.get("frac")}
             for n, v in m["stages"].items() if n.startswith("gemm")}
    bw = {n: {"ms": v["ms"], "gbs": v.get("achieved"), "frac": v.get("frac")}
          for n, v in m["stages"].items()
          if not n.startswith("gemm") and v.get("unit") == "GB/s"}
    pk, _ = peaks()
    return {"workload": wl.description, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k, "f": wl.f,
            "seed": wl.seed, "passes": "forward+backward" if wl.backward else "forward",
            "value": m["value"], "unit": UNIT, "ms_per_step": m["ms"],
            "e2e": None if m["e2e"] is None else m["e2e"]["value"],
            "gemm_tflops": m["gemm_tflops"],
            "gemm_frac_of_bf16_peak": m["gemm_tflops"] / pk["bf16_tflops"],
            "gemm_frac_of_bf16_sustained": m["gemm_tflops"] / pk["bf16_tflops_sustained"],
            "gemm_frac_of_nominal_dense": m["gemm_tflops"] / NOMINAL_BF16_TFLOPS,
            "step_roofline_frac": m["step_roofline"]["frac"],
            "step_bound": m["step_roofline"]["bound"],
            "gemms": gemms, "bandwidth_kernels": bw, "experts": m["experts"],
            "clocks": m["clocks"]}


def run_ours(args, rank, world, local_rank) -> dict | None:
    import moe_expert_layer_route_gb300 as moe
    from moe_expert_layer_route_gb300 import _build
    if rank == 0 or not _build.up_to_date():
        if world == 1 or local_rank == 0:
            _build.build()
    barrier(world)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    wl = workload_of(args)
    head = measure(moe, wl, args, args.steps, args.warmup, world, dev, flush,
                   want_graph=not args.no_graph, want_e2e=not args.no_e2e)
    torch.cuda.empty_cache()
    others = {}
    if not args.no_workloads and args.tokens is None and args.experts is None:
        k_sub = max(5, min(args.steps, 30))
        for name in WORKLOAD_ORDER:
            if name == wl.name:
                continue
            m = measure(moe, workloads.WORKLOADS[name], args, k_sub, args.warmup, world, dev,
                        flush, want_graph=False, want_e2e=not args.no_e2e)
            others[name] = summary_of(m)
            del m
            torch.cuda.empty_cache()
    if rank != 0:
        return None
    pk, _ = peaks()
    out = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": wl.description, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k,
                   "f": wl.f, "seed": wl.seed,
                   "passes": passes_of(wl, args, head["router_grad"]),
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "flushed (256 MB write) before each timed step, outside its events; "
                         f"weights alone are {6 * wl.E * wl.d * wl.f / 1e9:.2f} GB"},
        "gemm_tflops": head["gemm_tflops"],
        "gemm_frac_of_bf16_peak": head["gemm_tflops"] / pk["bf16_tflops"],
        "gemm_frac_of_bf16_sustained": head["gemm_tflops"] / pk["bf16_tflops_sustained"],
        "gemm_frac_of_nominal_dense": head["gemm_tflops"] / NOMINAL_BF16_TFLOPS,
        "gemm_flop_per_step": head["gemm_flop"],
        "ms_per_step_median": head["ms_median"],
        "step_roofline": head["step_roofline"],
        "experts": head["experts"],
        "graph": head["graph"],
        "roofline": head["roofline"],
        "stages": head["stages"],
        "gpu_launches": head["launches"],
        "clocks": head["clocks"],
        "e2e": head["e2e"],
        "workloads": others,
    }
    if not args.no_cpu_baseline and world == 1:
        out["cpu_baseline"] = cpu_baseline(wl, head["inp"], args.cpu_seconds, head["w_router"])
    return out


# ---------------------------------------------------------------- reference arm
def run_reference(args, rank, world) -> dict | None:
    """The CPU oracle as the reference arm: each step a bounded token sample."""
    if rank != 0:
        return None
    import oracle
    wl = workload_of(args)
    inp = workloads.make_inputs(wl, with_dy=wl.backward)
    inp_np = oracle_inputs(inp, wl.backward,
                           workloads.make_router_weight(wl) if args.router_gemm else None)
    # each step a token sample sized so that the whole run (sizing, warm-up and the timed
    # steps) takes about --reference-seconds; the oracle's cost per step has a floor that
    # does not shrink with the sample (every expert it touches writes its whole fp64 dW),
    # so at many steps the sample is small and the tokens/s lower than the cpu_baseline of
    # our arm's line, which times one larger sample
    budget = args.reference_seconds / (args.steps + args.warmup + 3)
    n = 16
    oracle_step(oracle, inp_np, n, wl.k)  # the first call pages in its fp64 buffers
    t = oracle_step(oracle, inp_np, n, wl.k)
    while t < budget / 2 and n * 2 <= wl.T:
        n *= 2
        t = oracle_step(oracle, inp_np, n, wl.k)
    for _ in range(max(0, args.warmup - 1)):
        oracle_step(oracle, inp_np, n, wl.k)
    times = [oracle_step(oracle, inp_np, n, wl.k) for _ in range(args.steps)]
    sec = statistics.mean(times)
    value = n / sec
    cores = cpu_threads()
    sample = (f"first {n} of {wl.T} tokens of the {wl.name} workload per step, "
              f"{'forward+backward' if wl.backward else 'forward'}"
              f"{' with the router GEMM' if args.router_gemm else ''} in fp64 numpy")
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": wl.description, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k,
                   "f": wl.f, "seed": wl.seed,
                   "passes": ("forward+backward" if wl.backward else "forward")
                   + (" + fp32 router GEMM (logits from x)" if args.router_gemm else "")},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="skip the CUDA-graph replay timing of the step")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure only the headline workload (no `workloads` record)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=180.0)
    ap.add_argument("--router-grad", action="store_true",
                    help="also compute the router-logit gradient in the backward")
    ap.add_argument("--router-gemm", action="store_true",
                    help="compute the fp32 router logits from x in the step (fused with top-k)")
    ap.add_argument("--selection-bias", action="store_true",
                    help="route on logits + a per-expert selection bias (Zipf ranks)")
    ap.add_argument("--aux-loss", action="store_true",
                    help="load-balancing statistics in the forward, their gradient in the "
                         "backward (implies --router-grad)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (profiling a smaller case; not a headline line)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (profiling a smaller case; not a headline line)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        dist_init(world, "nccl")
        out = run_ours(args, rank, world, local_rank)
        if world > 1:
            torch.distributed.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
