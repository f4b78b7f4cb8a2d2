"""The benchmark's claims checked on the GPU: how many of the library's kernels one
forward and one backward call launch (what `bench.py` reports as `gpu_launches`),
counted by the CUDA profiler, and one `bench.py` line on a small workload carrying every
field of its contract."""
import json
import os
import subprocess
import sys

import pytest
import torch

import bench
import expert_token_dispatch_gemm_b300 as moe
import workloads
from moe_gpu_harness import Layer

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def library_kernels(fn):
    """Names of the library's kernels (namespace moe) that fn launches."""
    from torch.profiler import ProfilerActivity, profile
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    return [e.name for e in prof.events()
            if e.device_type == torch.autograd.DeviceType.CUDA and "moe::" in e.name]


def small_layer(dtype, mode="dispatch", capacity_priority="token"):
    shape = workloads.LayerShape("launches_" + dtype, N=700, H=128, I=96, E=8, top_k=2,
                                 ep_size=4, capacity_factor=1.0, dtype=dtype, bias=True)
    return shape, Layer(shape, workloads.layer_inputs(shape, seed=5, variant="perf"), mode=mode,
                        capacity_priority=capacity_priority)


@pytest.mark.parametrize("dtype,mode,prio", [("bf16", "dispatch", "token"),
                                             ("bf16", "mask_sum", "token"),
                                             ("fp32", "dispatch", "token"),
                                             ("bf16", "dispatch", "slot")])
def test_forward_launches_what_the_bench_counts(dtype, mode, prio):
    """6 kernels per forward; slot-major capacity priority adds its histogram kernel."""
    shape, layer = small_layer(dtype, mode, prio)
    out = torch.empty(shape.N, shape.H, dtype=shape.torch_dtype, device="cuda")

    def fwd():
        moe.moe_layer_forward(layer.cfg, layer.x, layer.w_router, layer.b_router, layer.packed,
                              layer.w_down, out, layer.ws)
    fwd()                                   # kernel set-up outside the profile
    torch.cuda.synchronize()
    kernels = library_kernels(fwd)
    assert len(kernels) == bench.FORWARD_LAUNCHES + (prio == "slot"), kernels


def test_stats_and_tp_reduce_launch_what_the_bench_counts():
    """moe_balance_stats: partial sums and their ordered total (2 kernels); moe_tp_reduce
    for two slices: one kernel."""
    shape, layer = small_layer("bf16")
    dev = layer.x.device
    out = torch.empty(shape.N, shape.H, dtype=shape.torch_dtype, device=dev)
    logits = torch.empty(shape.N, shape.E, device=dev)
    routed = torch.empty(shape.E, dtype=torch.int32, device=dev)
    moe.moe_layer_forward(layer.cfg, layer.x, layer.w_router, layer.b_router, layer.packed,
                          layer.w_down, out, layer.ws,
                          dict(router_logits=logits, routed_counts=routed))
    load = torch.empty(shape.E, device=dev)
    prob = torch.empty(shape.E, device=dev)
    padded = torch.zeros(2, shape.N, shape.H, dtype=shape.torch_dtype, device=dev)

    def stats():
        moe.moe_balance_stats(layer.cfg, logits, routed, load, prob, layer.ws)

    def reduce():
        moe.moe_tp_reduce(layer.cfg, 2, padded, out)
    stats()
    reduce()
    torch.cuda.synchronize()
    assert len(library_kernels(stats)) == bench.STATS_LAUNCHES
    assert len(library_kernels(reduce)) == bench.TP_REDUCE_LAUNCHES


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_backward_launches_what_the_bench_counts(dtype):
    shape, layer = small_layer(dtype)
    layer.cfg.training = 1
    layer.ws = moe.alloc_workspace(layer.cfg)
    dev = layer.x.device
    out = torch.empty(shape.N, shape.H, dtype=shape.torch_dtype, device=dev)
    dout = torch.randn(shape.N, shape.H, device=dev).to(shape.torch_dtype)
    g = dict(dx=torch.empty_like(layer.x), dw_router=torch.empty(shape.E, shape.H, device=dev),
             db_router=torch.empty(shape.E, device=dev), dw_gate=torch.empty_like(layer.w_gate),
             dw_up=torch.empty_like(layer.w_up), dw_down=torch.empty_like(layer.w_down))

    def bwd():
        moe.moe_layer_backward(layer.cfg, layer.x, layer.w_router, layer.packed, layer.w_down,
                               dout, g["dx"], g["dw_router"], g["db_router"], g["dw_gate"],
                               g["dw_up"], g["dw_down"], layer.ws)
    moe.moe_layer_forward(layer.cfg, layer.x, layer.w_router, layer.b_router, layer.packed,
                          layer.w_down, out, layer.ws)
    bwd()
    torch.cuda.synchronize()
    kernels = library_kernels(bwd)
    assert len(kernels) == bench.backward_launches(dtype), kernels


def test_bench_line_carries_its_contract():
    """One `bench.py` run on the 16-expert gpt-oss-shaped workload: a single JSON line
    with the headline fields, the dominant kernel's roofline against a measured peak,
    the oracle's one-thread CPU baseline, the end-to-end figure with its copied bytes,
    the launch count and the clocks sampled during the timed region."""
    shape = workloads.BY_NAME["gptoss_profile_n1024_h2880_e16_k4"]
    steps = 3
    r = subprocess.run([sys.executable, "bench.py", "--workload", shape.name, "--steps",
                        str(steps), "--warmup", "3", "--no-variants", "--no-workloads"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] == 3
    assert d["dtype"] == "bf16" and d["data"].startswith("synthetic")
    assert d["config"] == bench.run_config(shape, "dispatch", 1)
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert abs(d["value"] - shape.N / (d["ms_per_step"] * 1e-3)) <= 1e-3 * d["value"]
    roof = d["roofline"]
    assert roof["bound"] in ("hbm", "tensor") and roof["unit"] in ("GB/s", "TFLOP/s")
    assert roof["peak"] > 0 and roof["achieved"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] > 0 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["unit"] == "tokens/s" and 0 < e2e["value"]
    assert e2e["h2d_bytes_per_step"] == shape.N * shape.H * 2
    assert e2e["d2h_bytes_per_step"] == shape.N * shape.H * 2
    assert d["gpu_launches"] == bench.FORWARD_LAUNCHES * steps
    clk = d["clocks"]
    assert clk["sm_mhz"] > 0 and clk["sm_max_mhz"] > 0 and isinstance(clk["reasons"], list)
    sus = d["sustained"]
    assert sus["steps"] == bench.SUSTAINED_STEPS and sus["ms_per_step"] > 0
    assert abs(sus["tokens_per_s"] - shape.N / (sus["ms_per_step"] * 1e-3)) <= 1e-3 * sus["tokens_per_s"]
    bwd = d["backward"]
    assert bwd["backward_ms"] > 0 and bwd["roofline"]["frac"] > 0
    assert bwd["gpu_launches"] == (bench.FORWARD_LAUNCHES + bench.backward_launches("bf16")) * steps
