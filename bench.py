#!/usr/bin/env python3
"""Benchmark of the MoE layer forward (route -> dispatch -> grouped GEMM -> combine).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl b300|reference]

Prints ONE JSON line (rank 0). A step is one full moe_layer_forward over one batch of
synthetic, seeded inputs already resident in HBM. The default workload is the
gpt-oss-120b-shaped layer (8192 tokens x hidden 2880, 128 experts, top-4, SwiGLU
intermediate 2880, 8 logical EP partitions). Its 6.4 GB of expert weights are ~50x the
L2, so no L2 flush is needed between steps.

The line also carries, for the same workload, the per-stage rooflines, the training
step, the routing variants, an end-to-end figure with host copies and a `sustained`
figure (100 back-to-back forwards, long enough for the board's power cap to act; the
headline's 20-step region ends before it does), and (one GPU only) a `workloads`
object: the other forward rule on the same inputs and the PR1, 8-expert, skewed +
capacity and decode workloads, each with its stage rooflines, clocks and training
step.

Under torchrun (N > 1) every rank runs the same layer on its own batch (different
seed): the expert-parallel partitions live inside one GPU, so ranks share no data and
the scaling is weak, with no collective on the data path.

--impl reference times the fp64 CPU oracle instead (rank 0 only, one thread): every
step is the whole layer on a token slice of the same batch, and the line reports the
measured time of that work.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The CPU legs time the oracle on one core: numpy's BLAS reads its thread count when it
# loads, so the limit is set before numpy is imported (SingleThread also sets and checks
# it at run time).
os.environ["OPENBLAS_NUM_THREADS"] = "1"
os.environ["MKL_NUM_THREADS"] = "1"

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "MoE-layer tokens/s (route→dispatch→grouped GEMM→combine); % of roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ------------------------------------------------------------------ algorithmic work
def stage_work(shape, counts):
    """Algorithmic bytes and flops of each stage, given the kept per-expert counts.
    Only what the method must move or compute: every operand read once, every result
    written once (weights of experts that received no token are not touched)."""
    s = 2 if shape.dtype == "bf16" else 4
    N, H, I, E, k = shape.N, shape.H, shape.I, shape.E, shape.top_k
    A = int(np.sum(counts))                     # kept pairs
    touched = int(np.count_nonzero(counts))
    nseg = math.ceil(N / 64)
    bias = 4 * E if (shape.bias or shape.zipf_s) else 0
    return {
        "route": dict(bytes=N * H * s + E * H * s + bias + N * k * 8 + nseg * E * 4,
                      flops=2 * N * H * E),
        # counts, offsets and slots in one kernel (the assign stage is empty)
        "scan": dict(bytes=nseg * E * 4 + N * k * 8 + A * 4 + 4 * E * 4, flops=0),
        "assign": dict(bytes=0, flops=0),
        "permute": dict(bytes=N * H * s + A * H * s + N * k * 4, flops=0),
        "gate_up": dict(bytes=touched * 2 * I * H * s + A * H * s + A * I * s,
                        flops=4 * A * H * I),
        "down": dict(bytes=touched * H * I * s + A * I * s + A * H * s + A * 8,
                     flops=2 * A * H * I),
        "combine": dict(bytes=A * H * s + N * H * s + N * k * 4, flops=0),
    }


def fp32_alu_tflops(peaks):
    """FFMA peak of the fp32 path: 148 SMs x 128 fp32 lanes x 2 flops per clock at the
    measured maximum SM clock."""
    return 148 * 128 * 2 * float(peaks.get("sm_max_mhz", 2032.0)) * 1e6 / 1e12


def roofline_entry(work, ms, peaks, source, dtype):
    t = ms / 1e3
    hbm = peaks["hbm_gbs"]
    tf = peaks["bf16_tflops"] if dtype == "bf16" else None
    t_mem = work["bytes"] / (hbm * 1e9)
    t_flop = work["flops"] / (tf * 1e12) if tf else 0.0
    if dtype != "bf16" and work["flops"]:
        alu = fp32_alu_tflops(peaks)
        if work["flops"] / (alu * 1e12) >= t_mem:
            ach = work["flops"] / t / 1e12
            return dict(bound="alu", achieved=round(ach, 2), peak=round(alu, 1),
                        unit="TFLOP/s", frac=round(ach / alu, 4),
                        peak_source="148 SMs x 128 fp32 lanes x 2 flop x max SM clock",
                        hbm_frac=round(work["bytes"] / t / 1e9 / hbm, 4))
    if tf and t_flop >= t_mem:
        ach = work["flops"] / t / 1e12
        return dict(bound="tensor", achieved=round(ach, 2), peak=tf, unit="TFLOP/s",
                    frac=round(ach / tf, 4), peak_source=f"{source} bf16 burst",
                    hbm_frac=round(work["bytes"] / t / 1e9 / hbm, 4))
    ach = work["bytes"] / t / 1e9
    out = dict(bound="hbm", achieved=round(ach, 1), peak=hbm, unit="GB/s",
               frac=round(ach / hbm, 4), peak_source=f"{source} copy bandwidth")
    if tf and work["flops"]:
        out["tensor_frac"] = round(work["flops"] / t / 1e12 / tf, 4)
    return out


# ------------------------------------------------------------------ ranks
def slowest_rank_ms(ms, dist, device):
    """The step time of the slowest rank (every rank gets the same value); `dist` is None
    for a single process."""
    if dist is None:
        return ms
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms):
    """Whole-job throughput: every rank processes its own batch (weak scaling), the job
    takes as long as the slowest rank."""
    return world * tokens_per_rank / (ms / 1e3)


# ------------------------------------------------------------------ measured DRAM traffic
TRAFFIC_SOURCES = ("grouped_gemm_pair.cu", "sm100.cuh", "common.cuh")


def gemm_sources_sha256():
    """Hash of the grouped-GEMM sources: a traffic record holds only for this code."""
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "expert_token_dispatch_gemm_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(workload, kernel):
    """DRAM bytes (read + write) per launch of `kernel` from the committed ncu record of
    this workload, or None when there is none or the kernel has changed since."""
    path = os.path.join(ROOT, "profiles", f"grouped_gemm_pair_traffic_{workload}.json")
    if kernel not in ("gate_up", "down") or not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("sources_sha256") != gemm_sources_sha256():
        return None
    b = rec["per_launch_bytes"][kernel]
    return int(b["dram_read"]) + int(b["dram_write"])


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        time.sleep(0.2)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        rows = []
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smmax=float(f[2]), power=float(f[3]),
                                 hw=f[5], hwt=f[6], swt=f[7], swpc=f[8]))
            except ValueError:
                continue
        if not rows:
            return None
        loaded = [r for r in rows if r["power"] > 0.5 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swpc", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(r["sm"] for r in loaded),
                    sm_max_mhz=max(r["smmax"] for r in rows), samples=len(loaded),
                    power_w_max=max(r["power"] for r in rows), reasons=sorted(reasons))


# ------------------------------------------------------------------ CPU oracle timing
def host_cpu():
    """The host's CPU model and logical core count."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return dict(model=model, logical_cores=os.cpu_count())


def _openblas_libs():
    """The OpenBLAS libraries loaded into this process (numpy's), by path."""
    import ctypes
    paths = []
    try:
        with open("/proc/self/maps") as f:
            for ln in f:
                path = ln.split()[-1] if len(ln.split()) >= 6 else ""
                if "openblas" in os.path.basename(path).lower() and ".so" in path and path not in paths:
                    paths.append(path)
    except OSError:
        return []
    libs = []
    for path in paths:
        try:
            libs.append(ctypes.CDLL(path))
        except OSError:
            continue
    return libs


def _blas_fn(lib, what):
    """OpenBLAS's openblas_{get,set}_num_threads under the names its builds export."""
    for name in (f"openblas_{what}_num_threads", f"scipy_openblas_{what}_num_threads64_",
                 f"openblas_{what}_num_threads64_", f"scipy_openblas_{what}_num_threads"):
        fn = getattr(lib, name, None)
        if fn is not None:
            return fn
    return None


class SingleThread:
    """Limits numpy's BLAS to one thread for the timed oracle work and reports the thread
    count in force, read back from the library: through threadpoolctl when it is
    installed, else through OpenBLAS's own get/set calls. Raises when neither can
    confirm one thread: the CPU figures claim one core."""

    def __enter__(self):
        self._undo = None
        try:
            from threadpoolctl import threadpool_info, threadpool_limits
        except ImportError:
            threadpool_info = None
        if threadpool_info is not None:
            ctx = threadpool_limits(limits=1)
            ctx.__enter__()
            self._undo = lambda *a: ctx.__exit__(*a)
            pools = threadpool_info()
            self.threads = max([int(i.get("num_threads", 1)) for i in pools] or [1])
            self.pools = sorted({f"{i.get('user_api')}:{i.get('internal_api')}" for i in pools})
        else:
            libs = [(lib, _blas_fn(lib, "get"), _blas_fn(lib, "set")) for lib in _openblas_libs()]
            libs = [x for x in libs if x[1] is not None and x[2] is not None]
            if not libs:
                raise RuntimeError("no OpenBLAS thread control found to pin the oracle to one thread")
            before = [int(get()) for _, get, _ in libs]
            for _, _, set_ in libs:
                set_(1)
            self._undo = lambda *a: [set_(n) for (_, _, set_), n in zip(libs, before)]
            self.threads = max(int(get()) for _, get, _ in libs)
            self.pools = [f"blas:openblas (set through its API; OPENBLAS_NUM_THREADS="
                          f"{os.environ.get('OPENBLAS_NUM_THREADS')})"]
        if self.threads != 1:
            raise RuntimeError(f"the oracle's BLAS still uses {self.threads} threads: {self.pools}")
        return self

    def __exit__(self, *a):
        if self._undo is not None:
            self._undo(*a)
        return False


# Token sample of the CPU runs: as many tokens as fit about 2e11 expert flops (1024 at the
# gpt-oss shape), so one pass of the fp64 oracle takes a few seconds on one core.
CPU_SAMPLE_FLOPS = 2.0e11


def cpu_sample_tokens(shape):
    per_token = 6.0 * shape.top_k * shape.H * shape.I
    return int(max(1, min(shape.N, CPU_SAMPLE_FLOPS // per_token)))


def time_oracle_slice(shape, x, w_router, b_router, expert_fn, t0, S, mode="dispatch"):
    """The fp64 oracle's whole layer (route, capacity, dispatch layout, permute, every
    expert that received rows, combine) on the S tokens t0 .. t0+S-1, as a layer call
    of its own. Only the oracle's work is timed: expert_fn(e) hands over an expert's
    fp64 weights outside the timed region (they are resident, as on the GPU side).
    Returns (timed seconds, detail)."""
    import oracle
    k, E, P = shape.top_k, shape.E, shape.ep_size
    xs = x[t0:t0 + S]
    c0 = time.perf_counter()
    logits, idx, w = oracle.route(xs, w_router, b_router, k)
    C = oracle.expert_capacity(shape.capacity_factor, S, k, E)
    lay = oracle.dispatch_layout(idx, E, P, C)
    send = oracle.permute(xs, lay["perm"], k)
    y = np.zeros((send.shape[0], shape.H))
    t_route = time.perf_counter() - c0
    t_ffn = 0.0
    busy = 0
    for e in range(E):
        a, b = int(lay["expert_offsets"][e]), int(lay["expert_offsets"][e + 1])
        if b == a:
            continue
        busy += 1
        wg, wu, wd = expert_fn(e)
        c1 = time.perf_counter()
        y[a:b] = oracle.swiglu_expert(send[a:b], wg, wu, wd)
        t_ffn += time.perf_counter() - c1
    c2 = time.perf_counter()
    if mode == "dispatch":
        oracle.combine_dispatch(y, lay["slot_pos"], w, S, k)
    else:
        oracle.combine_mask_sum(y, lay["slot_pos"], idx, w, E, P)
    t_combine = time.perf_counter() - c2
    total = t_route + t_ffn + t_combine
    return total, dict(route_dispatch_s=t_route, experts_s=t_ffn, combine_s=t_combine,
                       tokens=S, kept_pairs=int(lay["expert_offsets"][-1]), busy_experts=busy)


def host_inputs_for_oracle(shape, inp):
    f = lambda t: None if t is None else t.detach().to("cpu", torch.float64).numpy()
    return f(inp["x"]), f(inp["w_router"]), f(inp["b_router"])


def cpu_baseline_from_device(shape, inp, mode="dispatch"):
    """The oracle on one core on a bounded token sample of the bench workload: the whole
    layer (every step, every expert the sample reaches) on the first S tokens, each
    expert's weights copied from the device and widened to fp64 outside the timing."""
    x, wr, b = host_inputs_for_oracle(shape, inp)
    S = cpu_sample_tokens(shape)

    def expert_fn(e):
        return tuple(inp[k][e].detach().to("cpu", torch.float64).numpy()
                     for k in ("w_gate", "w_up", "w_down"))

    with SingleThread() as st:
        total, detail = time_oracle_slice(shape, x, wr, b, expert_fn, 0, S, mode)
    return dict(value=round(S / total, 2), unit="tokens/s", cores=st.threads, kind="oracle",
                sample=f"fp64 oracle, one thread: the whole layer on tokens 0..{S - 1} of the "
                       f"{shape.N}-token batch as one call ({detail['kept_pairs']} kept pairs, "
                       f"{detail['busy_experts']} experts)",
                seconds=round(total, 3), host=host_cpu(), thread_pools=st.pools,
                detail={k: (round(v, 4) if isinstance(v, float) else v) for k, v in detail.items()})


def resident_expert_weights(shape, seed=0):
    """Every expert's fp64 weights drawn on the CPU (the GPU arm's seeded weights), held
    in host memory when they fit in half of it; else None and they are drawn per use."""
    need = 3 * shape.E * shape.I * shape.H * 8
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        avail = 0
    if need > avail // 2:
        return None
    return {key: [workloads.expert_weight(shape, key, e, seed, "cpu").double().numpy()
                  for e in range(shape.E)] for key in ("w_gate", "w_up", "w_down")}


def run_reference(args, shape):
    """--impl reference: the fp64 CPU oracle as it stands, on one core. Every step (warm-up
    and timed) is the whole layer on a slice of S tokens of the bench batch, a different
    slice per step; ms_per_step is the measured time of that work and value the tokens it
    processed per second."""
    inp = workloads.layer_inputs(shape, seed=0, variant="perf", device="cpu",
                                 with_experts=False)
    x, wr, b = host_inputs_for_oracle(shape, inp)
    S = cpu_sample_tokens(shape)
    res = resident_expert_weights(shape)

    def expert_fn(e):
        if res is not None:
            return res["w_gate"][e], res["w_up"][e], res["w_down"][e]
        return tuple(workloads.expert_weight(shape, k, e, 0, "cpu").double().numpy()
                     for k in ("w_gate", "w_up", "w_down"))

    slices = max(1, shape.N // S)
    totals, details = [], []
    with SingleThread() as st:
        for i in range(args.warmup):
            time_oracle_slice(shape, x, wr, b, expert_fn, (i % slices) * S, S, args.mode)
        for i in range(args.steps):
            t, det = time_oracle_slice(shape, x, wr, b, expert_fn,
                                       ((args.warmup + i) % slices) * S, S, args.mode)
            totals.append(t)
            details.append(det)
    sec = float(np.mean(totals))
    value = S / sec
    sample = (f"per step: fp64 oracle, one thread, the whole layer on a {S}-token slice of "
              f"the {shape.N}-token batch as one call (slice i*{S} of step i)")
    world = args.gpus
    line = dict(metric=METRIC, value=round(value, 3), unit="tokens/s", n_gpus=world,
                steps=args.steps, warmup=args.warmup, ms_per_step=round(sec * 1e3, 3),
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data=DATA, config=run_config(shape, args.mode, world), impl="reference",
                cpu_baseline=dict(value=round(value, 3), unit="tokens/s", cores=st.threads,
                                  kind="oracle", sample=sample, host=host_cpu(),
                                  thread_pools=st.pools,
                                  weights="resident fp64" if res is not None
                                  else "drawn per use, outside the timing"),
                e2e=dict(value=round(value, 3), unit="tokens/s", h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0),
                detail=dict(tokens_per_step=S,
                            kept_pairs_per_step=int(np.mean([d["kept_pairs"] for d in details])),
                            experts_s=round(float(np.mean([d["experts_s"] for d in details])), 4),
                            route_dispatch_s=round(float(np.mean([d["route_dispatch_s"]
                                                                  for d in details])), 4),
                            combine_s=round(float(np.mean([d["combine_s"] for d in details])), 4)))
    print(json.dumps(line), flush=True)


def load_summary(shape, routed, kept):
    """The routing example's load quantities on the bench batch: per expert and per
    partition (expert // (E / ep_size)) pairs before capacity, and the dropped pairs."""
    parts = routed.reshape(shape.ep_size, -1).sum(axis=1)
    return dict(expert_max=int(routed.max()), expert_min=int(routed.min()),
                expert_mean=round(float(routed.mean()), 2),
                partition_max=int(parts.max()), partition_min=int(parts.min()),
                partition_mean=round(float(parts.mean()), 2),
                routed_pairs=int(routed.sum()), dropped_pairs=int(routed.sum() - kept.sum()))


def backward_launches(dtype):
    """Kernels of one moe_layer_backward call: permute, (bf16: the transposed copy of x,)
    the 4 expert GEMMs, logit gradients, dx combine, histogram, scan, 2 router-gradient."""
    return 12 if dtype == "bf16" else 11


def time_backward(moe, args, shape, inp, packed, dist, dev, stream, mode=None):
    """A training step on the same workload: moe_layer_forward with training = 1, then
    moe_layer_backward (CUDA events around each, `steps` timed after `warmup`). The four
    expert GEMMs of the backward are 2 x the forward's 6 A' H I flops."""
    cfg = moe.config(shape.N, shape.H, shape.I, shape.E, shape.top_k, shape.ep_size,
                     shape.capacity_factor, mode or args.mode, shape.dtype,
                     has_bias=inp["b_router"] is not None, training=True)
    ws = moe.alloc_workspace(cfg, dev)
    x, wr, b, wd = inp["x"], inp["w_router"], inp["b_router"], inp["w_down"]
    out = torch.empty(shape.N, shape.H, dtype=shape.torch_dtype, device=dev)
    gen = torch.Generator(device=dev).manual_seed(7)
    dout = torch.randn(shape.N, shape.H, device=dev, generator=gen).to(shape.torch_dtype)
    g = dict(dx=torch.empty_like(x), dw_router=torch.empty(shape.E, shape.H, device=dev),
             db_router=torch.empty(shape.E, device=dev), dw_gate=torch.empty_like(inp["w_gate"]),
             dw_up=torch.empty_like(inp["w_up"]), dw_down=torch.empty_like(wd))
    counts_t = torch.empty(shape.E, dtype=torch.int32, device=dev)

    def step(i, evs=None):
        if evs is not None:
            evs[0].record(stream)
        moe.moe_layer_forward(cfg, x, wr, b, packed, wd, out, ws,
                              dict(counts=counts_t) if i == 0 else None)
        if evs is not None:
            evs[1].record(stream)
        moe.moe_layer_backward(cfg, x, wr, packed, wd, dout, g["dx"], g["dw_router"],
                               g["db_router"], g["dw_gate"], g["dw_up"], g["dw_down"], ws)
        if evs is not None:
            evs[2].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    kept = int(counts_t.sum().item())
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        torch.cuda._sleep(2_000_000)
        for i in range(args.steps):
            step(1, evs[i])
        torch.cuda.synchronize()
    if moe.moe_read_device_status(cfg, ws):
        raise RuntimeError("device status flags set after the backward steps")
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    bwd_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    step_ms = slowest_rank_ms(fwd_ms + bwd_ms, dist, dev)
    bwd_ms = slowest_rank_ms(bwd_ms, dist, dev)
    world = dist.get_world_size() if dist is not None else 1
    flops = 12.0 * kept * shape.H * shape.I
    peaks, source = load_peaks()
    if shape.dtype == "bf16":
        bound, peak, psrc = "tensor", peaks.get("bf16_tflops_sustained"), f"bf16_tflops_sustained ({source})"
    else:
        bound, peak, psrc = "alu", fp32_alu_tflops(peaks), "FFMA: 148 SMs x 128 lanes x 2 x max SM clock"
    ach = flops / (bwd_ms * 1e-3) / 1e12
    return dict(train_tokens_per_s=round(job_tokens_per_s(shape.N, world, step_ms), 1),
                forward_training_ms=round(fwd_ms, 4), backward_ms=round(bwd_ms, 4),
                expert_gemm_tflop=round(flops / 1e12, 4),
                roofline=dict(bound=bound, achieved=round(ach, 1), unit="TFLOP/s",
                              peak=peak, frac=round(ach / peak, 4) if peak else None,
                              source=psrc,
                              note="whole backward time against the expert GEMMs' flops"),
                gpu_launches=(FORWARD_LAUNCHES + backward_launches(shape.dtype)) * args.steps,
                clocks=clk.summary())


def _event_ms(stream, fn, steps):
    """Mean CUDA-event time of fn over `steps` runs (after one warm-up run)."""
    fn()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a longer device-side delay before `start`: the host enqueues all steps of these
    # few-microsecond kernels ahead of the GPU
    torch.cuda._sleep(20_000_000)
    s0.record(stream)
    for _ in range(steps):
        fn()
    s1.record(stream)
    torch.cuda.synchronize()
    return s0.elapsed_time(s1) / steps


def time_variants(moe, args, shape, inp, packed, dev, stream):
    """The widened rows on the same workload: the forward with slot-major capacity
    priority (beside the token-priority forward timed the same way), the router load
    statistics (moe_balance_stats over the logits the forward writes) and the TP split's
    padded ordered sum (tp = 2). Timed before the backward."""
    peaks, source = load_peaks()
    bw = peaks["hbm_gbs"]
    s = 2 if shape.dtype == "bf16" else 4
    x, wr, b, wd = inp["x"], inp["w_router"], inp["b_router"], inp["w_down"]
    out = torch.empty(shape.N, shape.H, dtype=shape.torch_dtype, device=dev)
    res = {}
    # token and slot priority alternate step by step, each step between its own events,
    # so both see the same clock and power state
    cfgs, wss = {}, {}
    for prio in ("token", "slot"):
        cfgs[prio] = moe.config(shape.N, shape.H, shape.I, shape.E, shape.top_k, shape.ep_size,
                                shape.capacity_factor, args.mode, shape.dtype,
                                has_bias=b is not None, capacity_priority=prio)
        wss[prio] = moe.alloc_workspace(cfgs[prio], dev)
        moe.moe_layer_forward(cfgs[prio], x, wr, b, packed, wd, out, wss[prio])
    evs = {p: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] for p in cfgs}
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        torch.cuda._sleep(1_000_000)
        for i in range(args.steps):
            for prio in ("token", "slot"):
                evs[prio][i][0].record(stream)
                moe.moe_layer_forward(cfgs[prio], x, wr, b, packed, wd, out, wss[prio])
                evs[prio][i][1].record(stream)
        torch.cuda.synchronize()
    res["clocks"] = clk.summary()
    for prio in ("token", "slot"):
        ms = float(np.mean([a.elapsed_time(z) for a, z in evs[prio]]))
        res[f"{prio}_priority_forward"] = dict(ms=round(ms, 4),
                                               tokens_per_s=round(shape.N / (ms * 1e-3), 1),
                                               gpu_launches_per_step=FORWARD_LAUNCHES + (prio == "slot"))
    cfg, ws = cfgs["slot"], wss["slot"]
    logits = torch.empty(shape.N, shape.E, device=dev)
    routed = torch.empty(shape.E, dtype=torch.int32, device=dev)
    moe.moe_layer_forward(cfg, x, wr, b, packed, wd, out, ws,
                          dict(router_logits=logits, routed_counts=routed))
    load = torch.empty(shape.E, device=dev)
    prob = torch.empty(shape.E, device=dev)
    ms = _event_ms(stream, lambda: moe.moe_balance_stats(cfg, logits, routed, load, prob, ws),
                   args.steps)
    nbytes = shape.N * shape.E * 4 + shape.E * 12
    res["balance_stats"] = dict(ms=round(ms, 4), bound="hbm", achieved=round(nbytes / ms / 1e6, 1),
                                peak=bw, unit="GB/s", frac=round(nbytes / ms / 1e6 / bw, 4),
                                gpu_launches_per_step=STATS_LAUNCHES)
    padded = torch.zeros(2, shape.N, shape.H, dtype=shape.torch_dtype, device=dev)
    ms = _event_ms(stream, lambda: moe.moe_tp_reduce(cfg, 2, padded, out), args.steps)
    nbytes = 3 * shape.N * shape.H * s
    res["tp_reduce_tp2"] = dict(ms=round(ms, 4), bound="hbm", achieved=round(nbytes / ms / 1e6, 1),
                                peak=bw, unit="GB/s", frac=round(nbytes / ms / 1e6 / bw, 4),
                                gpu_launches_per_step=TP_REDUCE_LAUNCHES,
                                note="inputs below L2 size at small workloads: fractions above "
                                     "1 are L2 hits")
    res["peak_source"] = source
    return res


DATA = "synthetic (seeded; x~N(0,1), router~U(+-1/sqrt(H)), experts~N(0,0.02))"


def workload_config(shape):
    return dict(workload=shape.name, tokens=shape.N, hidden=shape.H, intermediate=shape.I,
                experts=shape.E, top_k=shape.top_k, ep_size=shape.ep_size,
                capacity_factor=shape.capacity_factor, router_zipf_s=shape.zipf_s,
                values="perf (continuous)",
                l2=("inputs larger than L2 (expert weights >> 126 MB); no flush"
                    if 3 * shape.E * shape.H * shape.I * (2 if shape.dtype == "bf16" else 4) > 126e6
                    else "inputs within L2 size: steps may hit L2; no flush"))


def run_config(shape, mode, world):
    """The `config` object of both arms' lines (the same dict for the same run)."""
    return dict(workload_config(shape), mode=mode,
                parallelism=f"replicas x{world} (one layer per GPU)")


# ------------------------------------------------------------------ GPU arm
class Layer:
    """One workload's inputs, packed weights, workspace and output on the device."""

    def __init__(self, moe, shape, mode, dev, seed, inp=None, packed=None):
        self.shape, self.mode = shape, mode
        self.inp = inp if inp is not None else workloads.layer_inputs(shape, seed=seed,
                                                                      variant="perf", device=dev)
        self.cfg = moe.config(shape.N, shape.H, shape.I, shape.E, shape.top_k, shape.ep_size,
                              shape.capacity_factor, mode, shape.dtype,
                              has_bias=self.inp["b_router"] is not None)
        self.packed = packed if packed is not None else moe.moe_pack_weights(
            self.cfg, self.inp["w_gate"], self.inp["w_up"])
        self.ws = moe.alloc_workspace(self.cfg, dev)
        self.out = torch.empty(shape.N, shape.H, dtype=shape.torch_dtype, device=dev)

    def forward(self, moe, diag=None, events=None, x=None, out=None):
        i = self.inp
        moe.moe_layer_forward(self.cfg, i["x"] if x is None else x, i["w_router"], i["b_router"],
                              self.packed, i["w_down"], self.out if out is None else out,
                              self.ws, diag, events)


FORWARD_LAUNCHES = 6   # route, scan/assign, permute, gate_up, down, combine
STATS_LAUNCHES = 2     # moe_balance_stats: per-block partial sums, their ordered total
TP_REDUCE_LAUNCHES = 1


def time_forward(moe, L, steps, warmup, dist, dev, stream, clocks=True):
    """`warmup` untimed steps, then two timed passes of `steps` forward steps, each between
    a barrier and a synchronize on both sides (CUDA events on the launching stream):
      1. the layer calls alone -- the step time (an event between two kernels would
         stop the next one from launching while the previous drains, so none is
         recorded inside this pass);
      2. the same calls with the library recording an event at every stage boundary --
         each kernel's duration.
    Returns the slowest rank's step time, the mean stage times, the kept and routed
    counts and the clock record of pass 1."""
    shape = L.shape
    counts_t = torch.empty(shape.E, dtype=torch.int32, device=dev)
    routed_t = torch.empty(shape.E, dtype=torch.int32, device=dev)
    L.forward(moe, dict(counts=counts_t, routed_counts=routed_t))
    torch.cuda.synchronize()
    counts, routed = counts_t.cpu().numpy(), routed_t.cpu().numpy()
    nst = moe.binding.MOE_NUM_STAGES
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(steps)]
    for row in evs:
        for e in row:
            e.record(stream)     # creates the handles before the library re-records them
    for _ in range(warmup):
        L.forward(moe)
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    sampler = ClockSampler(dev.index or 0) if clocks else contextlib.nullcontext()
    with sampler as clk:
        # a short device-side delay lets the host enqueue ahead of the timed steps, so
        # the first step does not wait for its launches (the delay is before `start`)
        torch.cuda._sleep(2_000_000)
        start.record(stream)
        for i in range(steps):
            L.forward(moe)
        end.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_step = slowest_rank_ms(start.elapsed_time(end) / steps, dist, dev)
    # pass 2: stage boundaries
    barrier()
    torch.cuda._sleep(2_000_000)
    for i in range(steps):
        L.forward(moe, None, evs[i])
    torch.cuda.synchronize()
    barrier()
    stage_ms = {name: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)]))
                for j, name in enumerate(moe.binding.STAGE_NAMES)}
    staged_ms = float(np.mean([evs[i][0].elapsed_time(evs[i][nst]) for i in range(steps)]))
    flags = moe.moe_read_device_status(L.cfg, L.ws)
    if flags:
        raise RuntimeError(f"device status flags {flags} after the timed steps of {shape.name}")
    return dict(ms_step=ms_step, stage_ms=stage_ms, staged_ms=staged_ms, counts=counts,
                routed=routed, clocks=clk.summary() if clocks else None)


def stage_rooflines(shape, stage_ms, counts, names):
    peaks, source = load_peaks()
    work = stage_work(shape, counts)
    return {n: dict(ms=round(stage_ms[n], 4),
                    **{k: v for k, v in roofline_entry(work[n], max(stage_ms[n], 1e-6), peaks,
                                                       source, shape.dtype).items()
                       if k in ("bound", "achieved", "unit", "frac", "hbm_frac", "tensor_frac")})
            for n in names}


def dominant_roofline(shape, stage_ms, counts, with_traffic=True):
    peaks, source = load_peaks()
    work = stage_work(shape, counts)
    dom = max(("gate_up", "down", "route", "permute", "combine"), key=lambda n: stage_ms[n])
    roof = roofline_entry(work[dom], stage_ms[dom], peaks, source, shape.dtype)
    return dict(kernel=dom, **roof,
                traffic=measured_traffic(shape.name, dom) if with_traffic else None)


SUSTAINED_STEPS = 100


def time_sustained(moe, L, dev, stream, steps=SUSTAINED_STEPS):
    """Back-to-back forwards for ~0.2 s (device time), with their own clock record: the
    rate once the board's power management has reacted. The headline's timed region
    (20 steps by default) ends before it does; this is reported beside it, not in it."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        torch.cuda._sleep(2_000_000)
        a.record(stream)
        for _ in range(steps):
            L.forward(moe)
        b.record(stream)
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    return dict(steps=steps, ms_per_step=round(ms, 4),
                tokens_per_s=round(L.shape.N / (ms * 1e-3), 1), clocks=clk.summary())


def time_e2e(moe, L, steps, dist, dev, stream):
    """End to end through the C ABI: every step copies its input from pinned host memory
    to the device and reads its output back. Copies run on their own streams, double
    buffered, so step i+1's upload and step i-1's download overlap step i's compute."""
    x, out = L.inp["x"], L.out
    x_host = [x.cpu().pin_memory() for _ in range(2)]
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty_like(out) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run_pipeline(n):
        uploaded = [torch.cuda.Event() for _ in range(n)]
        computed = [torch.cuda.Event() for _ in range(n)]
        downloaded = [torch.cuda.Event() for _ in range(n)]
        for i in range(n):
            bb = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(computed[i - 2])     # x_dev[bb] no longer read
                x_dev[bb].copy_(x_host[bb], non_blocking=True)
                uploaded[i].record(up)
            stream.wait_event(uploaded[i])
            if i >= 2:
                stream.wait_event(downloaded[i - 2])   # out_dev[bb] already read back
            L.forward(moe, x=x_dev[bb], out=out_dev[bb])
            computed[i].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[i])
                out_host[bb].copy_(out_dev[bb], non_blocking=True)
                downloaded[i].record(down)
        stream.wait_event(downloaded[n - 1])

    run_pipeline(3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    run_pipeline(steps)
    s1.record(stream)
    torch.cuda.synchronize()
    world = dist.get_world_size() if dist is not None else 1
    e2e_ms = slowest_rank_ms(s0.elapsed_time(s1) / steps, dist, dev)
    return dict(value=round(job_tokens_per_s(L.shape.N, world, e2e_ms), 1), unit="tokens/s",
                ms_per_step=round(e2e_ms, 4), h2d_bytes_per_step=x.numel() * x.element_size(),
                d2h_bytes_per_step=out.numel() * out.element_size(),
                overlap="uploads and downloads on their own streams, double buffered")


# The other workloads of the layer, timed after the headline one in the default run
# (forward, its stage rooflines and clocks, and the training step): the PR1 fp32 layer,
# the 8-expert and skewed + capacity layers (where the grouped GEMM is tensor bound) and
# the decode batch (weight-read bound; its step time is the layer's latency).
EXTRA_WORKLOADS = (workloads.PR1_FP32, workloads.E8_TOP2, workloads.SKEWED_CAP, workloads.DECODE)


def workload_entry(moe, args, L, dist, dev, stream, backward=True):
    shape = L.shape
    world = dist.get_world_size() if dist is not None else 1
    r = time_forward(moe, L, args.steps, args.warmup, dist, dev, stream)
    stages = ("route", "scan", "permute", "gate_up", "down", "combine")
    entry = dict(mode=L.mode, tokens_per_s=round(job_tokens_per_s(shape.N, world, r["ms_step"]), 1),
                 ms_per_step=round(r["ms_step"], 4), dtype=shape.dtype,
                 config=workload_config(shape),
                 roofline=dominant_roofline(shape, r["stage_ms"], r["counts"], with_traffic=False),
                 stages=stage_rooflines(shape, r["stage_ms"], r["counts"], stages),
                 stage_pass_ms_per_step=round(r["staged_ms"], 4),
                 kept_pairs=int(r["counts"].sum()), load=load_summary(shape, r["routed"], r["counts"]),
                 clocks=r["clocks"], gpu_launches=FORWARD_LAUNCHES * args.steps)
    if shape.N <= 256:
        entry["latency_ms"] = round(r["ms_step"], 4)
    if backward:
        entry["backward"] = time_backward(moe, args, shape, L.inp, L.packed, dist, dev, stream,
                                          mode=L.mode)
    return entry


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=workloads.GPTOSS.name, choices=sorted(workloads.BY_NAME))
    ap.add_argument("--impl", default="b300", choices=["b300", "reference"])
    ap.add_argument("--mode", default="dispatch", choices=["dispatch", "mask_sum"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-sustained", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads and the mask-and-sum line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    shape = workloads.BY_NAME[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, shape)
        return

    import expert_token_dispatch_gemm_b300 as moe
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    L = Layer(moe, shape, args.mode, dev, seed=rank)
    r = time_forward(moe, L, args.steps, args.warmup, dist, dev, stream)
    ms_step = r["ms_step"]
    value = job_tokens_per_s(shape.N, world, ms_step)
    counts = r["counts"]

    variants = None
    if not args.no_variants:   # before the backward's long high-power stretch
        variants = time_variants(moe, args, shape, L.inp, L.packed, dev, stream)
    backward = None
    if not args.no_backward:
        backward = time_backward(moe, args, shape, L.inp, L.packed, dist, dev, stream)
    e2e = None if args.no_e2e else time_e2e(moe, L, args.steps, dist, dev, stream)
    # last on this workload: its stretch at the power cap would slow what follows
    sustained = None if args.no_sustained else time_sustained(moe, L, dev, stream)

    roof = dominant_roofline(shape, r["stage_ms"], counts)
    per_stage = stage_rooflines(shape, r["stage_ms"], counts, moe.binding.STAGE_NAMES)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_from_device(shape, L.inp, args.mode)

    # the other forward rule on the same inputs, then the other workloads (one replica
    # per GPU; skipped under torchrun, where only the headline line is compared)
    others = None
    if world == 1 and not args.no_workloads:
        others = {}
        other_mode = "mask_sum" if args.mode == "dispatch" else "dispatch"
        M = Layer(moe, shape, other_mode, dev, seed=rank, inp=L.inp, packed=L.packed)
        others[f"{shape.name}:{other_mode}"] = workload_entry(moe, args, M, dist, dev, stream,
                                                             backward=False)
        del M, L
        torch.cuda.empty_cache()
        for extra in EXTRA_WORKLOADS:
            if extra.name == shape.name:
                continue
            X = Layer(moe, extra, "dispatch", dev, seed=rank)
            others[extra.name] = workload_entry(moe, args, X, dist, dev, stream,
                                                backward=not args.no_backward)
            del X
            torch.cuda.empty_cache()

    if rank == 0:
        line = dict(metric=METRIC, value=round(value, 1), unit="tokens/s", n_gpus=world,
                    steps=args.steps, warmup=args.warmup, ms_per_step=round(ms_step, 4),
                    higher_is_better=True, scaling="weak", vs_baseline=None, dtype=shape.dtype,
                    data=DATA, config=run_config(shape, args.mode, world),
                    roofline=roof, stages=per_stage,
                    stage_pass_ms_per_step=round(r["staged_ms"], 4),
                    cpu_baseline=cpu, e2e=e2e,
                    gpu_launches=FORWARD_LAUNCHES * args.steps, clocks=r["clocks"],
                    kept_pairs=int(counts.sum()), load=load_summary(shape, r["routed"], counts),
                    sustained=sustained, backward=backward, variants=variants,
                    workloads=others, impl="b300")
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
