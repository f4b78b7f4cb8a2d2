"""The benchmark's host arithmetic, on CPU: algorithmic work per stage (closed forms of
each stage's byte and flop counts on a hand-checked shape), the roofline's choice of
bound and fraction, the traffic record's guard on the GEMM sources, whole-job
throughput, the load summary, the CPU legs (one-thread pinning, token sample, the same
config in both arms), and the reference arm's line (run on a small workload)."""
import json
import math

import numpy as np
import pytest

import bench
import workloads


def test_stage_work_closed_forms():
    shape = workloads.LayerShape("w", N=128, H=64, I=32, E=4, top_k=2, ep_size=2)
    counts = np.array([100, 0, 80, 76])                 # 256 kept pairs, 3 experts touched
    w = bench.stage_work(shape, counts)
    s, N, H, I, E, k, A = 2, 128, 64, 32, 4, 2, 256
    assert w["permute"]["bytes"] == N * H * s + A * H * s + N * k * 4
    assert w["gate_up"]["bytes"] == 3 * 2 * I * H * s + A * H * s + A * I * s
    assert w["gate_up"]["flops"] == 4 * A * H * I
    assert w["down"]["flops"] == 2 * A * H * I
    assert w["down"]["bytes"] == 3 * H * I * s + A * I * s + A * H * s + 8 * A
    assert w["combine"]["bytes"] == A * H * s + N * H * s + N * k * 4
    assert w["route"]["flops"] == 2 * N * H * E
    assert w["route"]["bytes"] == N * H * s + E * H * s + N * k * 8 + math.ceil(N / 64) * E * 4


PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0, "sm_max_mhz": 2000.0}


def test_roofline_picks_the_binding_resource():
    # memory-bound: 6 GB in 1 ms at 6 TB/s is exactly the peak
    r = bench.roofline_entry(dict(bytes=6e9, flops=1e12), 1.0, PEAKS, "m", "bf16")
    assert r["bound"] == "hbm" and r["frac"] == pytest.approx(1.0)
    assert r["tensor_frac"] == pytest.approx(1e12 / 1e-3 / 1e12 / 1800, abs=1e-4)   # rounded
    # compute-bound: 1.8 PFLOP/s worth of flops
    r = bench.roofline_entry(dict(bytes=1e6, flops=0.9e12), 1.0, PEAKS, "m", "bf16")
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(0.5)
    # fp32: FFMA peak 148 x 128 x 2 x 2 GHz
    alu = 148 * 128 * 2 * 2000e6 / 1e12
    assert bench.fp32_alu_tflops(PEAKS) == pytest.approx(alu)
    r = bench.roofline_entry(dict(bytes=1e6, flops=alu * 1e9 / 2), 1.0, PEAKS, "m", "fp32")
    assert r["bound"] == "alu" and r["frac"] == pytest.approx(0.5)


def test_job_throughput_is_weak_scaling():
    assert bench.job_tokens_per_s(8192, 4, 2.0) == pytest.approx(4 * 8192 / 2e-3)
    assert bench.slowest_rank_ms(3.5, None, None) == 3.5


def test_traffic_record_holds_only_for_its_sources(tmp_path, monkeypatch):
    rec = dict(sources_sha256=bench.gemm_sources_sha256(),
               per_launch_bytes=dict(gate_up=dict(dram_read=10, dram_write=5),
                                     down=dict(dram_read=7, dram_write=1)))
    (tmp_path / "profiles").mkdir()
    path = tmp_path / "profiles" / "grouped_gemm_pair_traffic_wl.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "gemm_sources_sha256", lambda: rec["sources_sha256"])
    assert bench.measured_traffic("wl", "gate_up") == 15
    assert bench.measured_traffic("wl", "down") == 8
    assert bench.measured_traffic("wl", "route") is None
    assert bench.measured_traffic("other", "gate_up") is None
    monkeypatch.setattr(bench, "gemm_sources_sha256", lambda: "changed")
    assert bench.measured_traffic("wl", "gate_up") is None


def test_committed_traffic_record_matches_the_current_sources():
    assert bench.measured_traffic(workloads.GPTOSS.name, "gate_up") is not None


def test_load_summary():
    shape = workloads.LayerShape("l", N=10, H=8, I=8, E=4, top_k=2, ep_size=2)
    routed = np.array([7, 3, 6, 4])
    kept = np.array([5, 3, 5, 4])
    s = bench.load_summary(shape, routed, kept)
    assert (s["expert_max"], s["expert_min"], s["expert_mean"]) == (7, 3, 5.0)
    assert (s["partition_max"], s["partition_min"]) == (10, 10)
    assert s["routed_pairs"] == 20 and s["dropped_pairs"] == 3


def test_cpu_legs_run_on_one_thread():
    from threadpoolctl import threadpool_info
    with bench.SingleThread() as st:
        assert st.threads == 1
        assert all(int(i.get("num_threads", 1)) == 1 for i in threadpool_info())
    info = bench.host_cpu()
    assert info["logical_cores"] == __import__("os").cpu_count()


def test_cpu_legs_pin_openblas_without_threadpoolctl(monkeypatch):
    # hosts without threadpoolctl: the limit is set and read back through OpenBLAS's API
    import sys
    monkeypatch.setitem(sys.modules, "threadpoolctl", None)
    libs = bench._openblas_libs()
    if not any(bench._blas_fn(lib, "get") for lib in libs):
        pytest.skip("numpy here is not linked against OpenBLAS")
    with bench.SingleThread() as st:
        assert st.threads == 1 and "openblas" in st.pools[0]


def test_cpu_sample_tokens_is_a_flop_budget():
    # about 2e11 expert flops: 6 k H I per token
    g = workloads.GPTOSS
    assert bench.cpu_sample_tokens(g) == int(2e11 // (6 * 4 * 2880 * 2880)) == 1004
    assert bench.cpu_sample_tokens(workloads.DECODE) == 128          # the whole batch
    assert 1 <= bench.cpu_sample_tokens(workloads.E8_TOP2) < workloads.E8_TOP2.N


def test_oracle_slice_is_a_layer_call_of_its_own():
    import oracle
    shape = workloads.LayerShape("slice", N=96, H=16, I=8, E=4, top_k=2, ep_size=2,
                                 capacity_factor=1.0)
    inp = workloads.layer_inputs(shape, seed=3, variant="perf")
    f = lambda t: None if t is None else t.double().numpy()
    x, wr = f(inp["x"]), f(inp["w_router"])
    W = {k: f(inp[k]) for k in ("w_gate", "w_up", "w_down")}
    t, det = bench.time_oracle_slice(shape, x, wr, None,
                                     lambda e: (W["w_gate"][e], W["w_up"][e], W["w_down"][e]),
                                     32, 40)
    assert t > 0 and det["tokens"] == 40
    # the slice's capacity is its own: ceil(1.0 * 40 * 2 / 4) = 20 per expert
    ref = oracle.layer_forward(x[32:72], wr, None, W["w_gate"], W["w_up"], W["w_down"],
                               2, 2, capacity_factor=1.0)
    assert det["kept_pairs"] == int(ref["expert_offsets"][-1])
    assert det["busy_experts"] == int((ref["counts"] > 0).sum())


def test_both_arms_share_one_config():
    c1 = bench.run_config(workloads.GPTOSS, "dispatch", 1)
    c2 = bench.run_config(workloads.GPTOSS, "dispatch", 1)
    assert c1 == c2 and c1["workload"] == workloads.GPTOSS.name
    assert c1["mode"] == "dispatch" and "parallelism" in c1


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` on a small workload: one JSON line whose metric,
    config and timing fields match the GPU arm's, with the oracle's one-thread CPU
    baseline and an end-to-end figure that moves no bytes between host and device."""
    import os
    import subprocess
    import sys
    shape = workloads.PR1_FP32
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        shape.name, "--steps", "1", "--warmup", "3"], cwd=root,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["config"] == bench.run_config(shape, "dispatch", 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert isinstance(cb["sample"], str) and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm runs on rank 0 alone; another rank exits 0
    without output, and rank 0's line counts the launch's GPUs."""
    import os
    import subprocess
    import sys
    shape = workloads.PR1_FP32
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", shape.name,
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    for rank in (1, 0):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2")
        r = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
        if rank:
            assert lines == []
        else:
            assert len(lines) == 1
            d = json.loads(lines[0])
            assert d["n_gpus"] == 2 and d["config"] == bench.run_config(shape, "dispatch", 2)
