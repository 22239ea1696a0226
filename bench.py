#!/usr/bin/env python
"""Throughput of the MoE layer forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config dsv3] [--impl ours|reference]

One step = one pass of the whole layer (route -> permute -> grouped gate/up GEMM
+ SwiGLU -> grouped down GEMM x gate weight -> combine) over one batch of
synthetic tokens, through the library's C ABI (moe_forward).  Inputs and
weights are resident in HBM before the timed region; they are larger than L2
(x 235 MB and 22.6 GB of expert weights at the DeepSeek-V3 shape), so no L2
flush is needed between steps.  Prints ONE JSON line on rank 0.

--impl reference times the CPU oracle (the fp64 definition of the layer) on a
bounded sample of the same workload per step, on the host cores.

Under torchrun (--gpus N > 1) every rank runs an independent replica of the
whole workload on its own GPU (the layer has no exchange step here): weak
scaling, value = tokens of all ranks / slowest rank's time.
"""
from __future__ import annotations

import os

# The oracle baseline runs single-threaded; set before numpy loads its BLAS.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import re  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workload as wl  # noqa: E402

METRIC = "MoE-layer prefill tokens/s and TFLOP/s (% of GB300 tensor peak), 1 GPU"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ distributed
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def dist_init(backend: str):
    rank, world, _ = dist_info()
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)
    return rank, world


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(v: float, device=None) -> float:
    """Largest value of v over all ranks (v itself without a process group)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0: float, t1: float):
        rows = []
        try:
            for ln in open(self.path):
                p = [x.strip() for x in ln.split(",")]
                if len(p) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(p[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + p[0].split(".")[1]) if "." in p[0] else 0.0
                    rows.append((ts, float(p[2]), float(p[3]), p[6:10], float(p[4])))
                except Exception:
                    continue
        except Exception:
            return None
        if not rows:
            return None
        inside = [r for r in rows if t0 - 0.06 <= r[0] <= t1 + 0.06] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "power_w_median": statistics.median(r[4] for r in inside),
                "samples": len(inside)}


# ------------------------------------------------------------------ helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# Source files that decide each profiled kernel's code: its own translation
# unit plus the shared headers.
KERNEL_SOURCES = {
    "bf16": ("grouped_gemm.cu", "moe_internal.h", "ptx.cuh"),
    "fp8": ("grouped_gemm_fp8.cu", "moe_internal.h", "ptx.cuh"),
    "nvfp4": ("grouped_gemm_nvfp4.cu", "nvfp4.cuh", "moe_internal.h", "ptx.cuh"),
}

# Dense tensor rate of fp4 (E2M1, block-scaled) relative to bf16 on GB300
# (nominal 13.5 vs 2.25 PFLOP/s): the fp4 peak is the measured bf16 peak x 6.
FP4_OVER_BF16 = 6.0


def _code_only(text: str) -> str:
    """Source text without comments and blank lines: edits to comments leave
    the kernel's code, and so the recorded hash, unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_source_hash(kind: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_expert_layer_router_gb300", "csrc")
    for f in KERNEL_SOURCES[kind]:
        h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, kind: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None when
    the summary is missing or was taken on other sources of that kernel."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_ncu.md")
    if not os.path.exists(p):
        return None
    vals = {}
    for ln in open(p):
        if ln.startswith("- ") and ":" in ln:
            k, _, v = ln[2:].partition(":")
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha") != kernel_source_hash(kind):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except Exception:
        return None


def weight_gb(lc) -> float:
    """Bytes of the layer's expert weights (routed + shared) as stored."""
    n = 3.0 * lc.H * (lc.E * lc.I + lc.I_shared)
    per = {"bf16": 2.0, "fp8_e4m3": 1.0 + 4.0 / 128 / 128, "nvfp4": 0.5 + 1.0 / 16}[lc.wtype]
    return n * per / 1e9


def describe(lc) -> str:
    s = (f"{lc.name}: T={lc.T} H={lc.H} E={lc.E} top-{lc.k} I={lc.I} {lc.score}"
         f"{' x' + str(lc.route_scale) if lc.route_scale != 1.0 else ''}")
    if lc.I_shared:
        s += f" + shared I={lc.I_shared}"
    if lc.zipf_bias:
        s += " + Zipf(1.2) router bias"
    return s + f", {lc.wtype}"


class Layer:
    """Seeded layer on one device; every expert matrix in its own allocation.
    fp8 layers: the fp32 weights are block-quantised by the library once, before
    any timing (W holds the fp32 originals, which the oracle baseline uses)."""

    def __init__(self, lc, dev, keep_fp32=True):
        import moe_expert_layer_router_gb300 as m
        self.lc = lc
        self.x = wl.gen_x(lc, dev)
        self.wr = wl.gen_router(lc, dev)
        b = wl.gen_bias(lc)
        self.bias = b.to(dev) if b is not None else None
        self.W = [tuple(wl.gen_expert(lc, e, w, dev) for w in ("gate", "up", "down"))
                  for e in range(lc.E)]
        self.S = (tuple(wl.gen_shared(lc, w, dev) for w in ("gate", "up", "down"))
                  if lc.I_shared else None)
        self.cfg = m.config_from(lc)
        if lc.wtype == "nvfp4":
            # NVFP4: the library quantises the bf16 weights (W keeps the bf16
            # originals, from which the oracle quantises its own copy)
            gx, gh = wl.nvfp4_act_scales(lc)
            self.weights = m.quantize_experts_nvfp4(
                self.cfg, [w[0] for w in self.W], [w[1] for w in self.W], [w[2] for w in self.W],
                shared=self.S, input_scale=gx, hidden_scale=gh)
            torch.cuda.synchronize(dev)
            if not keep_fp32:
                self.W = self.S = None
                torch.cuda.empty_cache()
        elif lc.wtype == "fp8_e4m3":
            Q = [tuple(m.moe_quantize_weight_fp8(t) for t in w3) for w3 in self.W]
            SQ = tuple(m.moe_quantize_weight_fp8(t) for t in self.S) if self.S else None
            self.Q, self.SQ = Q, SQ
            self.weights = m.ExpertWeights(
                self.cfg, [q[0][0] for q in Q], [q[1][0] for q in Q], [q[2][0] for q in Q],
                shared=tuple(t[0] for t in SQ) if SQ else None,
                scales=([q[0][1] for q in Q], [q[1][1] for q in Q], [q[2][1] for q in Q]),
                shared_scales=tuple(t[1] for t in SQ) if SQ else None)
            if not keep_fp32:  # only the quantised weights are needed
                self.W = self.S = None
                torch.cuda.empty_cache()
        else:
            self.weights = m.ExpertWeights(self.cfg, [w[0] for w in self.W],
                                           [w[1] for w in self.W], [w[2] for w in self.W],
                                           shared=self.S)


def route_ids(layer, ws, dev):
    """The routing decision of the layer's batch (one extra moe_route call, untimed)."""
    import moe_expert_layer_router_gb300 as m
    ids, _, _ = m.moe_route(layer.cfg, layer.x, layer.wr, layer.bias)
    torch.cuda.synchronize(dev)
    return ids


# ------------------------------------------------------------------ oracle baseline
_QCACHE = {}


def _oracle_fp8_weights(key, t):
    """The oracle's own 128x128 block quantisation of an fp32 weight matrix
    (input preparation, outside any timing; cached: the fp8 weights are the
    layer's inputs)."""
    from oracle import fp8 as of8
    if key not in _QCACHE:
        _QCACHE[key] = of8.quantize_weight_blocks(t.cpu().numpy())
    return _QCACHE[key]


def _oracle_nvfp4_expert(key, mats):
    """The oracle's own NVFP4 quantisation of one expert's bf16 matrices (input
    preparation, outside any timing; cached)."""
    from oracle import nvfp4 as onv
    if key not in _QCACHE:
        _QCACHE[key] = onv.dequantize_expert(*onv.quantize_expert(
            *(t.float().cpu().numpy() for t in mats)))
    return _QCACHE[key]


def oracle_sample(lc, layer, tokens):
    """Time the CPU oracle on `tokens` of the workload; returns (seconds, n)."""
    from oracle import moe as om
    idx = torch.tensor(tokens, device=layer.x.device)
    x = layer.x[idx].cpu()
    wr = layer.wr.cpu()
    b = None if layer.bias is None else layer.bias.cpu()
    # the weights the sample needs, moved to host memory outside the timing
    lg = om.router_logits(x, wr, b)
    need = sorted(set(om.select_topk(lg, lc.k).reshape(-1).tolist()))
    fp8 = lc.wtype == "fp8_e4m3"
    fp4 = lc.wtype == "nvfp4"
    if fp4:
        host = {e: _oracle_nvfp4_expert(e, layer.W[e]) for e in need}
        sh = _oracle_nvfp4_expert("s", layer.S) if layer.S is not None else None
    elif fp8:
        host = {e: tuple(_oracle_fp8_weights((e, i), t) for i, t in enumerate(layer.W[e]))
                for e in need}
        sh = (tuple(_oracle_fp8_weights(("s", i), t) for i, t in enumerate(layer.S))
              if layer.S is not None else None)
    else:
        host = {e: tuple(t.cpu() for t in layer.W[e]) for e in need}
        sh = tuple(t.cpu() for t in layer.S) if layer.S is not None else None
    t0 = time.perf_counter()
    if fp4:
        from oracle import nvfp4 as onv
        gx, gh = wl.nvfp4_act_scales(lc)
        onv.moe_layer_nvfp4(x, wr, b, lambda e: host[e], sh, lc.k, lc.score, lc.renormalize,
                            lc.route_scale, gx, gh)
    elif fp8:
        from oracle import fp8 as of8
        of8.moe_layer_fp8(x, wr, b, lambda e: tuple(of8.dequant_weight(*q) for q in host[e]),
                          tuple(of8.dequant_weight(*q) for q in sh) if sh is not None else None,
                          lc.k, lc.score, lc.renormalize, lc.route_scale)
    else:
        om.moe_layer(x, wr, b, lambda e: host[e], sh, lc.k, lc.score, lc.renormalize,
                     lc.route_scale)
    return time.perf_counter() - t0, len(tokens)


def cpu_baseline(lc, layer, n_tokens=None):
    if n_tokens is None:
        n_tokens = 2 if lc.wtype in ("fp8_e4m3", "nvfp4") else 8
    g = np.random.default_rng(1)
    tokens = sorted(g.choice(lc.T, size=n_tokens, replace=False).tolist())
    secs, n = oracle_sample(lc, layer, tokens)
    return {"value": n / secs, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} tokens of the {lc.name} workload through the fp64 oracle "
                      f"(routing, permutation, grouped experts, combine), {secs:.1f} s, "
                      f"1 thread"}


# ------------------------------------------------------------------ our arm
def run_ours(args, lc, rank, world, dev):
    import moe_expert_layer_router_gb300 as m
    from moe_expert_layer_router_gb300 import _native as N

    layer = Layer(lc, dev)
    cfg = layer.cfg
    ws = m.Workspace(cfg, "forward", dev)
    out = torch.empty(lc.T, lc.H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        m.moe_forward(cfg, layer.weights, layer.x, layer.wr, layer.bias, out=out, ws=ws,
                      stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    m.moe_get_device_error(ws)

    # kernel trace: one event before every kernel and one after the last, per step
    per_step = 16
    cap = per_step * args.steps
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(cap)]
    for e in evs:
        e.record(stream)      # creates the CUDA event on this device
    torch.cuda.synchronize(dev)
    ev_arr = (N.C.c_void_p * cap)(*[e.cuda_event for e in evs])
    kid = (N.C.c_int32 * cap)()
    trace = N.MoeTrace(N.C.cast(ev_arr, N.C.POINTER(N.C.c_void_p)),
                       N.C.cast(kid, N.C.POINTER(N.C.c_int32)), cap, 0)

    # inside the timed steps only GEMM1 is bracketed: an event before it and one
    # before GEMM2 (the dominant kernel's duration for the roofline)
    g1_cap = 2 * args.steps
    g1_evs = [torch.cuda.Event(enable_timing=True) for _ in range(g1_cap)]
    for e in g1_evs:
        e.record(stream)
    torch.cuda.synchronize(dev)
    g1_arr = (N.C.c_void_p * g1_cap)(*[e.cuda_event for e in g1_evs])
    g1_kid = (N.C.c_int32 * g1_cap)()
    g1_trace = N.MoeTrace(N.C.cast(g1_arr, N.C.POINTER(N.C.c_void_p)),
                          N.C.cast(g1_kid, N.C.POINTER(N.C.c_int32)), g1_cap, 0,
                          (1 << N.KERNEL_NAMES.index("gemm1_gate_up_swiglu"))
                          | (1 << N.KERNEL_NAMES.index("gemm2_down")))

    clocks = ClockSampler(dev.index if dev.index is not None else 0) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    # the timed steps: the plain calls, with two events per step around GEMM1
    N.check(N.lib().moe_set_trace(N.C.byref(g1_trace)), "moe_set_trace")
    w0 = time.time()
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    w1 = time.time()
    N.lib().moe_set_trace(None)
    barrier()
    ms_local = start.elapsed_time(end) / args.steps
    m.moe_get_device_error(ws)
    g1_timed = [g1_evs[i].elapsed_time(g1_evs[i + 1]) for i in range(0, g1_trace.count - 1, 2)
                if g1_kid[i] == N.KERNEL_NAMES.index("gemm1_gate_up_swiglu")]
    g1_ms_timed = sum(g1_timed) / len(g1_timed) if g1_timed else None
    # the same steps again with the trace hook: per-kernel durations and the
    # number of kernels each step launches
    N.check(N.lib().moe_set_trace(N.C.byref(trace)), "moe_set_trace")
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    N.lib().moe_set_trace(None)
    m.moe_get_device_error(ws)

    # per-kernel durations from the trace
    per_kernel = {}
    launches = 0
    for i in range(trace.count - 1):
        k = kid[i]
        if k < 0:
            continue
        launches += 1
        per_kernel.setdefault(N.KERNEL_NAMES[k], []).append(evs[i].elapsed_time(evs[i + 1]))
    kernels_ms = {k: sum(v) / len(v) for k, v in per_kernel.items()}

    # end to end through the public call with host buffers (pinned), copies included:
    # every step copies its x in from pinned host memory and its output back out.
    # As a serving loop would, x and out are double-buffered and the copies run on
    # their own streams, so step i+1's input and step i-1's output move while step
    # i computes; the timed region spans every copy of every step.
    x_host = layer.x.cpu().pin_memory()
    out_host = [torch.empty(lc.T, lc.H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(layer.x) for _ in range(2)]
    out_dev = [torch.empty_like(out) for _ in range(2)]
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    compute = torch.cuda.current_stream(dev)

    def e2e_run(n_steps):
        """n_steps pipelined steps; returns (first event, last event)."""
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(compute)
        h2d_stream.wait_stream(compute)
        d2h_stream.wait_stream(compute)
        in_ready = [None, None]
        fwd_done = [None, None]
        out_free = [None, None]

        def h2d(i):
            b = i % 2
            with torch.cuda.stream(h2d_stream):
                if fwd_done[b] is not None:      # step i-2 has finished reading x_dev[b]
                    h2d_stream.wait_event(fwd_done[b])
                x_dev[b].copy_(x_host, non_blocking=True)
                in_ready[b] = torch.cuda.Event()
                in_ready[b].record(h2d_stream)

        h2d(0)
        for i in range(n_steps):
            b = i % 2
            if i + 1 < n_steps:
                h2d(i + 1)
            compute.wait_event(in_ready[b])
            if out_free[b] is not None:          # step i-2's output has been copied out
                compute.wait_event(out_free[b])
            m.moe_forward(cfg, layer.weights, x_dev[b], layer.wr, layer.bias, out=out_dev[b],
                          ws=ws, stream=stream)
            fwd_done[b] = torch.cuda.Event()
            fwd_done[b].record(compute)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(fwd_done[b])
                out_host[b].copy_(out_dev[b], non_blocking=True)
                out_free[b] = torch.cuda.Event()
                out_free[b].record(d2h_stream)
        compute.wait_stream(h2d_stream)
        compute.wait_stream(d2h_stream)
        stop.record(compute)
        return start, stop

    e2e_run(2)
    torch.cuda.synchronize(dev)
    barrier()
    s2, e2 = e2e_run(args.steps)
    torch.cuda.synchronize(dev)
    e2e_ms_local = s2.elapsed_time(e2) / args.steps
    assert torch.equal(out_host[(args.steps - 1) % 2], out.cpu()), "e2e output differs"
    barrier()
    if clocks:
        clocks.stop()

    ms = max_over_ranks(ms_local, dev)
    e2e_ms = max_over_ranks(e2e_ms_local, dev)
    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    tokens = lc.T * world
    flops = lc.flops()
    tflops = flops * world / (ms * 1e-3) / 1e12
    # GEMM1's duration from the timed steps themselves (the traced second run's
    # split is kept in kernels_ms)
    g1_ms = g1_ms_timed if g1_ms_timed else kernels_ms.get("gemm1_gate_up_swiglu")
    # the timed region is a fraction of a second of back-to-back steps, so the
    # tensor-core denominators are the burst figures (fp4: the bf16 burst times
    # the nominal dense fp4 / bf16 ratio)
    fp4_peak = FP4_OVER_BF16 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    if lc.wtype == "nvfp4":
        # NVFP4 GEMM1: fp4 tensor cores or, if slower at the peaks, HBM (E2M1 codes
        # + one e4m3 scale per 16 of the gate/up weights of every expert with
        # tokens, the padded token rows in, h out) -- whichever takes longer
        g1_flops = 4.0 * lc.R * lc.H * lc.I + 4.0 * lc.T * lc.H * lc.I_shared
        counts = torch.bincount(route_ids(layer, ws, dev).reshape(-1).long(), minlength=lc.E)
        active = int((counts > 0).sum().item())
        rows_pad = int(((counts + 127) // 128 * 128).sum().item())
        t_pad = (lc.T + 127) // 128 * 128
        nib = 0.5 + 1.0 / 16  # bytes per element: code + scale
        g1_bytes = nib * (2.0 * active * lc.I * lc.H + 2.0 * lc.I_shared * lc.H
                          + (rows_pad + t_pad) * lc.H + rows_pad * lc.I + t_pad * lc.I_shared)
        hpeak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        if g1_bytes / (hpeak * 1e9) > g1_flops / (fp4_peak * 1e12):
            g1_ach = g1_bytes / (g1_ms * 1e-3) / 1e9 if g1_ms else None
            roof = {"kernel": "gemm1_gate_up_swiglu (nvfp4)", "bound": "hbm", "achieved": g1_ach,
                    "peak": hpeak, "unit": "GB/s", "frac": (g1_ach / hpeak) if g1_ach else None,
                    "peak_kind": f"HBM copy, of {peak_src}",
                    "algorithmic_bytes_per_launch": g1_bytes, "experts_with_tokens": active,
                    "traffic": recorded_traffic("gemm1_gate_up_swiglu", lc.name, "nvfp4")}
        else:
            g1_tf = g1_flops / (g1_ms * 1e-3) / 1e12 if g1_ms else None
            roof = {"kernel": "gemm1_gate_up_swiglu (nvfp4)", "bound": "tensor",
                    "achieved": g1_tf, "peak": fp4_peak, "unit": "TFLOP/s",
                    "frac": (g1_tf / fp4_peak) if g1_tf else None,
                    "peak_kind": f"fp4 = {FP4_OVER_BF16:g} x bf16 burst, of {peak_src}",
                    "algorithmic_flop_per_launch": g1_flops,
                    "algorithmic_bytes_per_launch": g1_bytes,
                    "traffic": recorded_traffic("gemm1_gate_up_swiglu", lc.name, "nvfp4")}
    elif lc.wtype == "fp8_e4m3":
        # small-batch fp8: GEMM1 streams the gate/up weights of every expert that
        # received a token (HBM-bound); algorithmic bytes per launch
        counts = torch.bincount(route_ids(layer, ws, dev).reshape(-1).long(), minlength=lc.E)
        active = int((counts > 0).sum().item())
        g1_bytes = (2.0 * active * lc.I * lc.H * (1 + 4.0 / 128 / 128)
                    + 2.0 * lc.I_shared * lc.H * (1 + 4.0 / 128 / 128)
                    + (lc.R + lc.T) * lc.H * (1 + 4.0 / 128)
                    + (lc.R * lc.I + lc.T * lc.I_shared) * (1 + 4.0 / 128))
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        g1_ach = g1_bytes / (g1_ms * 1e-3) / 1e9 if g1_ms else None
        roof = {"kernel": "gemm1_gate_up_swiglu (fp8)", "bound": "hbm", "achieved": g1_ach,
                "peak": peak, "unit": "GB/s", "frac": (g1_ach / peak) if g1_ach else None,
                "peak_kind": f"HBM copy, of {peak_src}", "algorithmic_bytes_per_launch": g1_bytes,
                "experts_with_tokens": active,
                "traffic": recorded_traffic("gemm1_gate_up_swiglu", lc.name, "fp8")}
    else:
        # bf16 GEMM1: bound by the tensor cores or, for small batches, by streaming
        # the gate/up weights of every expert that received a token -- whichever
        # takes longer at the measured peaks decides the roofline
        g1_flops = 4.0 * lc.R * lc.H * lc.I + 4.0 * lc.T * lc.H * lc.I_shared
        counts = torch.bincount(route_ids(layer, ws, dev).reshape(-1).long(), minlength=lc.E)
        active = int((counts > 0).sum().item())
        g1_bytes = 2.0 * (2.0 * active * lc.I * lc.H + 2.0 * lc.I_shared * lc.H
                          + (lc.R + lc.T) * lc.H + lc.R * lc.I + lc.T * lc.I_shared)
        tpeak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        hpeak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        if g1_bytes / (hpeak * 1e9) > g1_flops / (tpeak * 1e12):
            g1_ach = g1_bytes / (g1_ms * 1e-3) / 1e9 if g1_ms else None
            roof = {"kernel": "gemm1_gate_up_swiglu", "bound": "hbm", "achieved": g1_ach,
                    "peak": hpeak, "unit": "GB/s", "frac": (g1_ach / hpeak) if g1_ach else None,
                    "peak_kind": f"HBM copy, of {peak_src}",
                    "algorithmic_bytes_per_launch": g1_bytes, "experts_with_tokens": active,
                    "traffic": None}
        else:
            g1_tf = g1_flops / (g1_ms * 1e-3) / 1e12 if g1_ms else None
            roof = {"kernel": "gemm1_gate_up_swiglu", "bound": "tensor",
                    "achieved": g1_tf, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": (g1_tf / tpeak) if g1_tf else None,
                    "peak_kind": f"bf16 burst, of {peak_src}",
                    "algorithmic_flop_per_launch": g1_flops,
                    "traffic": recorded_traffic("gemm1_gate_up_swiglu", lc.name, "bf16")}
    res = {
        "metric": METRIC,
        "value": tokens / (ms * 1e-3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"fp8_e4m3": "fp8_e4m3 (fp32 accumulate)",
                  "nvfp4": "nvfp4 (E2M1 x E2M1, e4m3 scale per 16, fp32 accumulate)"}.get(
                      lc.wtype, "bf16"),
        "data": "synthetic (seeded counter-based generator; x ~N(0,1), weights ~N(0,0.02))",
        "config": {"workload": describe(lc), "tokens_per_gpu": lc.T,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (x and the expert weights: "
                         f"{weight_gb(lc):.1f} GB); no flush"},
        "tflops": tflops,
        "pct_of_peak": {"bf16_burst": 100 * tflops / world / float(
                            peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
                        "bf16_sustained": 100 * tflops / world / float(
                            peaks.get("bf16_tflops_sustained",
                                      FALLBACK_PEAKS["bf16_tflops_sustained"])),
                        "source": peak_src,
                        **({"fp4_burst": 100 * tflops / world / fp4_peak}
                           if lc.wtype == "nvfp4" else {})},
        "kernels_ms": {k: round(v, 4) for k, v in sorted(kernels_ms.items(),
                                                           key=lambda kv: -kv[1])},
        "kernels_ms_source": "a second run of the same steps with an event before every "
                             "kernel; the roofline's GEMM1 time is from the timed steps",
        "gemm1_ms_timed_steps": round(g1_ms_timed, 4) if g1_ms_timed else None,
        "roofline": roof,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s",
                "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": layer.x.numel() * 2, "d2h_bytes_per_step": out.numel() * 2,
                "copies": "pinned host x in and out every step, on their own streams, "
                          "overlapping the neighbouring steps' forward (double-buffered)"},
        "gpu_launches": launches,
        "clocks": clocks.summary(w0, w1) if clocks else None,
    }
    if args.stack:
        res["stack"] = stack_dispatch(args, lc, layer, dev)
    if world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(lc, layer, args.cpu_tokens)
    return res


def stack_dispatch(args, lc, layer, dev):
    """Layer-stack dispatch: L layers of the workload (seeds 0..L-1; layer 0 is the
    benchmarked one) run in turn on the same input, (a) one moe_forward call per
    layer, (b) one CUDA graph recorded once that, per layer, writes the layer index
    on the device and runs moe_forward_stack.  The kernels are the same; (b) takes
    the host out of the loop between layers."""
    import moe_expert_layer_router_gb300 as m
    L = args.stack
    layers = [layer] + [Layer(lc.with_(seed=s), dev, keep_fp32=False) for s in range(1, L)]
    cfg, x = layer.cfg, layer.x
    stream = torch.cuda.current_stream(dev)
    ws = m.Workspace(cfg, "forward", dev)
    out = torch.empty(lc.T, lc.H, dtype=torch.bfloat16, device=dev)
    biases = [Ly.bias for Ly in layers]
    stack = m.LayerStack(cfg, [Ly.weights for Ly in layers], [Ly.wr for Ly in layers],
                         biases if any(b is not None for b in biases) else None)
    index = torch.arange(L, dtype=torch.int32, device=dev)
    lid = torch.zeros(1, dtype=torch.int32, device=dev)

    def direct():
        for Ly in layers:
            m.moe_forward(cfg, Ly.weights, x, Ly.wr, Ly.bias, out=out, ws=ws, stream=stream)

    m.moe_forward_stack(cfg, stack, lid, x, out=out, ws=ws, stream=stream)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for l in range(L):
            lid.copy_(index[l:l + 1])
            m.moe_forward_stack(cfg, stack, lid, x, out=out, ws=ws,
                                stream=torch.cuda.current_stream())

    def timed(fn, reps):
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b)

    for _ in range(args.warmup):
        direct()
        graph.replay()
    # Segments in the order direct, graph, graph, direct, ...: a power-capped
    # GPU runs the first of two back-to-back measurements a few percent faster,
    # so each way is measured first as often as second.
    reps = max(1, args.steps // L)
    segs = 4
    tot = {"direct": 0.0, "graph": 0.0}
    for i in range(segs):
        pair = (("direct", direct), ("graph", graph.replay))
        for name, fn in (pair if i % 2 == 0 else pair[::-1]):
            tot[name] += timed(fn, reps)
    m.moe_get_device_error(ws)
    per = segs * reps * L
    return {"layers": L, "direct_ms_per_layer": tot["direct"] / per,
            "graph_ms_per_layer": tot["graph"] / per,
            "how": f"{segs} segments of {reps} rounds each way, alternating which way runs "
                   f"first, over {L} seeded layers on one input: moe_forward per layer vs "
                   f"one CUDA graph of moe_forward_stack (layer index written on the device)"}


# ------------------------------------------------------------------ reference arm
def run_reference(args, lc, rank, world, dev):
    if rank != 0:
        return None
    layer_dev = dev if torch.cuda.is_available() else torch.device("cpu")

    class HostLayer:  # inputs only; the oracle needs no descriptor table
        pass

    class Experts:  # an expert's matrices are generated the first time a sample needs them
        def __init__(self):
            self.cache = {}

        def __getitem__(self, e):
            if e not in self.cache:
                self.cache[e] = tuple(wl.gen_expert(lc, e, w, layer_dev)
                                      for w in ("gate", "up", "down"))
            return self.cache[e]

    L = HostLayer()
    L.x = wl.gen_x(lc, layer_dev)
    L.wr = wl.gen_router(lc, layer_dev)
    b = wl.gen_bias(lc)
    L.bias = b.to(layer_dev) if b is not None else None
    L.W = Experts()
    L.S = (tuple(wl.gen_shared(lc, w, layer_dev) for w in ("gate", "up", "down"))
           if lc.I_shared else None)
    g = np.random.default_rng(2)
    per = args.ref_tokens
    # fp8: draw the per-step samples from a small fixed pool of tokens, so the
    # (untimed, cached) oracle quantisation of their experts' weights is done once
    pool = (sorted(g.choice(lc.T, size=4, replace=False).tolist())
            if lc.wtype in ("fp8_e4m3", "nvfp4") else None)
    times, n_tok = [], 0
    for i in range(args.warmup + args.steps):
        if pool is not None:
            toks = sorted(g.choice(pool, size=min(per, len(pool)), replace=False).tolist())
        else:
            toks = sorted(g.choice(lc.T, size=per, replace=False).tolist())
        s, n = oracle_sample(lc, L, toks)
        if i >= args.warmup:
            times.append(s)
            n_tok += n
    total = sum(times)
    v = n_tok / total
    return {"metric": METRIC, "impl": "reference", "value": v, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / len(times), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": describe(lc), "tokens_per_step": per},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"{per} random tokens of the workload per step through "
                                       f"the fp64 oracle, 1 thread"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="dsv3", choices=sorted(wl.CONFIGS))
    ap.add_argument("--cpu-tokens", type=int, default=None)
    ap.add_argument("--ref-tokens", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stack", type=int, default=0,
                    help="also time L layers dispatched directly vs one graph of a layer stack")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    lc = wl.CONFIGS[args.config]
    rank, world, local = dist_info()
    if world > 1:
        torch.cuda.set_device(local)
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    rank, world = dist_init("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        res = run_reference(args, lc, rank, world, dev)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
        import moe_expert_layer_router_gb300.build as b
        b.build()
        torch.cuda.set_device(dev)
        res = run_ours(args, lc, rank, world, dev)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
