"""Parity of the CUDA path (called through the C ABI) with the fp64 oracle.

Small shapes span several M/N/K tiles with ragged tails and are checked in full; the
five workloads run at full size in the launch configuration the benchmark times and are
checked bit-exactly on routing and dispatch and on sampled token outputs.
Bars: routing ids, counts, offsets, perm and slot_pos bit-exact (exact variant: dyadic
router inputs make fp32 logits exact); outputs max|err| <= 2e-2 max|ref| (bf16) or
1e-4 max|ref| (fp32).
"""
import numpy as np
import pytest
import torch

import workloads
from moe_gpu_harness import (Layer, assert_close, assert_routing_and_layout_exact, f64,
                             full_size_reference_routing, oracle_layer, routing_margin,
                             sampled_token_check, tol_for)

pytestmark = pytest.mark.gpu

S = workloads.LayerShape
SMALL = [
    # several m tiles per expert, ragged rows, ragged I (Ipad 256), ragged H n-tiles
    S("bf16_ragged", N=1000, H=320, I=200, E=4, top_k=2, ep_size=2),
    S("bf16_e16_k4_cap_zipf", N=777, H=128, I=136, E=16, top_k=4, ep_size=4,
      capacity_factor=1.0, zipf_s=1.1),
    S("bf16_bias_e8", N=333, H=256, I=264, E=8, top_k=2, ep_size=4, bias=True),
    S("bf16_k8_e64", N=515, H=192, I=128, E=64, top_k=8, ep_size=8),
    S("fp32_ragged", N=333, H=96, I=72, E=6, top_k=3, ep_size=3, dtype="fp32", bias=True),
    S("fp32_cap", N=640, H=64, I=40, E=8, top_k=2, ep_size=2, dtype="fp32",
      capacity_factor=0.75, zipf_s=1.1),
    # ~550 tokens per expert: three 256-token tiles, the last one nearly empty
    S("bf16_long_segments", N=1100, H=136, I=72, E=2, top_k=1, ep_size=2),
]


def _inputs(shape, seed=0, variant="exact"):
    return workloads.layer_inputs(shape, seed=seed, variant=variant)


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
@pytest.mark.parametrize("mode", ["dispatch", "mask_sum"])
def test_small_layer_matches_oracle(shape, mode):
    inp = _inputs(shape, seed=3)
    ref = oracle_layer(shape, inp, mode)
    layer = Layer(shape, inp, mode)
    out, diag = layer.forward()
    assert_routing_and_layout_exact(diag, ref, shape)
    assert_close(out, ref["out"], tol_for(shape))
    assert layer.device_status() == 0


@pytest.mark.parametrize("shape", SMALL[:3] + SMALL[4:5], ids=lambda s: s.name)
def test_step_entry_points_match_fused_forward(shape):
    inp = _inputs(shape, seed=4)
    layer = Layer(shape, inp)
    out_fused, diag_fused = layer.forward()
    out_steps, diag_steps, send, slots = layer.steps()
    for k in diag_fused:
        assert torch.equal(diag_fused[k], diag_steps[k]), k
    assert torch.equal(out_fused, out_steps)
    # send rows are exact copies of the routed tokens' hidden states
    kept = int(diag_steps["expert_offsets"][-1])
    perm = diag_steps["perm"][:kept].long()
    assert torch.equal(send[:kept], layer.x[perm // shape.top_k])
    # per-partition expert launches give the same slots as one launch
    _, _, _, slots_p = layer.steps(per_partition=True)
    assert torch.equal(slots, slots_p)


@pytest.mark.parametrize("shape", [SMALL[0], SMALL[4]], ids=lambda s: s.name)
def test_perf_variant_small(shape):
    inp = _inputs(shape, seed=0, variant="perf")
    ref = oracle_layer(shape, inp)
    # precondition from the oracle alone: every routing gap exceeds twice the standard
    # bound on fp32 summation error, (H+1) * 2^-24 * sum_h |x w|, so the fp32 router
    # cannot reorder experts
    x, wr = f64(inp["x"]), f64(inp["w_router"])
    bound = (shape.H + 1) * 2.0 ** -24 * float((np.abs(x) @ np.abs(wr).T).max())
    assert routing_margin(ref["logits"], shape.top_k) > 2 * bound
    layer = Layer(shape, inp)
    out, diag = layer.forward()
    assert np.array_equal(diag["topk_idx"].cpu().numpy(), ref["topk_idx"])
    assert_close(out, ref["out"], tol_for(shape))


def test_dispatch_and_mask_modes_agree_on_gpu():
    shape = SMALL[1]
    inp = _inputs(shape, seed=6)
    a, _ = Layer(shape, inp, "dispatch").forward()
    m, _ = Layer(shape, inp, "mask_sum").forward()
    ref = oracle_layer(shape, inp)
    assert_close(m, f64(a), tol_for(shape), "mask vs dispatch")
    assert_close(m, ref["out"], tol_for(shape))


def test_repeated_runs_are_bitwise_identical():
    shape = SMALL[1]
    layer = Layer(shape, _inputs(shape, seed=7))
    o1, d1 = layer.forward()
    o2, d2 = layer.forward()
    assert torch.equal(o1, o2)
    for k in d1:
        assert torch.equal(d1[k], d2[k])


# ------------------------------------------------------------------ edge cases
EDGE = [
    S("one_token", N=1, H=64, I=32, E=4, top_k=2, ep_size=2),
    S("single_expert_k1", N=200, H=64, I=48, E=1, top_k=1, ep_size=1),
    S("k_equals_e", N=150, H=64, I=32, E=4, top_k=4, ep_size=4),
    S("max_experts_max_k", N=130, H=64, I=32, E=256, top_k=32, ep_size=8),
    S("capacity_one", N=300, H=64, I=32, E=8, top_k=2, ep_size=4, capacity_factor=1e-4),
    S("ragged_segments", N=65, H=136, I=24, E=3, top_k=2, ep_size=1),
    S("fp32_one_token", N=1, H=32, I=16, E=2, top_k=1, ep_size=2, dtype="fp32"),
    # the smallest sizes the boundary accepts (multiples of 8): every copy box is wider
    # than the tensor it reads
    S("min_sizes_bf16", N=300, H=8, I=8, E=4, top_k=2, ep_size=2, bias=True),
    S("min_sizes_fp32", N=300, H=8, I=8, E=4, top_k=2, ep_size=2, dtype="fp32", bias=True),
    # the FFMA router and experts at the most experts and slots
    S("fp32_max_experts_max_k", N=130, H=64, I=32, E=256, top_k=32, ep_size=8, dtype="fp32"),
]


@pytest.mark.parametrize("mode", ["dispatch", "mask_sum"])
@pytest.mark.parametrize("shape", EDGE, ids=lambda s: s.name)
def test_edge_cases(shape, mode):
    inp = _inputs(shape, seed=8)
    ref = oracle_layer(shape, inp, mode)
    layer = Layer(shape, inp, mode)
    out, diag = layer.forward()
    assert_routing_and_layout_exact(diag, ref, shape)
    assert_close(out, ref["out"], tol_for(shape))


# A row of H values is nvec = H / (8 bf16 or 4 fp32) 16-byte vectors, one per lane, 32 at
# a time: with H = 264 (bf16) or 136 (fp32) the last pass over a row has 1 or 2 active
# lanes, fewer than the k = 12 slots whose owners the warp must still see together.
RAGGED_ROWS = [
    S("k12_ragged_rows_bf16", N=300, H=264, I=64, E=32, top_k=12, ep_size=4, bias=True),
    S("k12_ragged_rows_fp32", N=300, H=136, I=32, E=32, top_k=12, ep_size=4, dtype="fp32"),
]


@pytest.mark.parametrize("mode", ["dispatch", "mask_sum"])
@pytest.mark.parametrize("shape", RAGGED_ROWS, ids=lambda s: s.name)
def test_many_slots_with_a_ragged_last_row_pass(shape, mode):
    inp = _inputs(shape, seed=12)
    ref = oracle_layer(shape, inp, mode=mode)
    out, diag = Layer(shape, inp, mode=mode).forward()
    assert_routing_and_layout_exact(diag, ref, shape)
    assert_close(out, ref["out"], tol_for(shape))


def _skewed_router(shape, hot_experts, seed=9):
    """All tokens prefer `hot_experts` (large bias), leaving other experts and whole
    partitions empty."""
    inp = _inputs(shape, seed=seed)
    b = torch.zeros(shape.E, dtype=torch.float32)
    b[list(hot_experts)] = 8.0
    inp["b_router"] = b
    return inp


def test_empty_experts_and_partitions():
    shape = S("empty_parts", N=500, H=64, I=32, E=16, top_k=2, ep_size=4, bias=True)
    inp = _skewed_router(shape, [0, 1, 2])
    ref = oracle_layer(shape, inp)
    assert np.all(ref["counts"][3:] == 0)
    for mode in ("dispatch", "mask_sum"):
        ref = oracle_layer(shape, inp, mode)
        out, diag = Layer(shape, inp, mode).forward()
        assert_routing_and_layout_exact(diag, ref, shape)
        assert_close(out, ref["out"], tol_for(shape))


def test_all_tokens_to_one_expert_with_capacity():
    shape = S("one_hot", N=700, H=64, I=32, E=8, top_k=1, ep_size=2, bias=True,
              capacity_factor=2.0)
    inp = _skewed_router(shape, [5])
    ref = oracle_layer(shape, inp)
    assert ref["routed_counts"][5] == 700 and ref["counts"][5] == ref["capacity"] == 175
    out, diag = Layer(shape, inp).forward()
    assert_routing_and_layout_exact(diag, ref, shape)
    assert_close(out, ref["out"], tol_for(shape))
    dropped = (diag["slot_pos"].view(700) < 0).cpu().numpy()
    assert np.all(f64(out)[dropped] == 0.0)


def test_bad_expert_id_is_dropped_and_flagged():
    shape = S("bad_id", N=100, H=64, I=32, E=4, top_k=2, ep_size=2)
    layer = Layer(shape, _inputs(shape, seed=10))
    _, diag = layer.forward()
    assert layer.device_status() == 0
    idx = diag["topk_idx"].clone()
    idx[7, 1] = 99
    idx[20, 0] = -3
    d = layer.diag_buffers()
    send = torch.zeros((200, 64), dtype=torch.bfloat16, device="cuda")
    import expert_token_dispatch_gemm_b300 as moe
    moe.moe_dispatch(layer.cfg, idx, layer.x, d["routed_counts"], d["counts"],
                     d["expert_offsets"], d["part_offsets"], d["perm"], d["slot_pos"], send,
                     layer.ws)
    torch.cuda.synchronize()
    assert layer.device_status() & moe.MOE_DEV_BAD_EXPERT_ID
    sp = d["slot_pos"].view(100, 2).cpu().numpy()
    assert sp[7, 1] == -1 and sp[20, 0] == -1
    assert int(d["routed_counts"].sum()) == 198


def test_empty_batch():
    shape = S("empty", N=0, H=64, I=32, E=4, top_k=2, ep_size=2)
    import expert_token_dispatch_gemm_b300 as moe
    from moe_gpu_harness import make_cfg
    cfg = make_cfg(shape)
    ws = moe.alloc_workspace(cfg)
    counts = torch.full((4,), 5, dtype=torch.int32, device="cuda")
    out = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_forward(cfg, w, w, None, w, w, out, ws, dict(counts=counts))
    torch.cuda.synchronize()
    assert counts.tolist() == [0, 0, 0, 0]


# ------------------------------------------------------------------ full-size workloads
def test_pr1_fp32_full_layer_both_modes():
    shape = workloads.PR1_FP32
    inp = _inputs(shape, seed=0)
    for mode in ("dispatch", "mask_sum"):
        ref = oracle_layer(shape, inp, mode)
        out, diag = Layer(shape, inp, mode).forward()
        assert_routing_and_layout_exact(diag, ref, shape)
        assert_close(out, ref["out"], tol_for(shape))


def test_routing_example_on_gpu():
    """The worked routing example: the GPU router reproduces the printed loads."""
    x, w, b = workloads.snippet_inputs()
    shape = S("ul_example", N=4096, H=512, I=8, E=8, top_k=2, ep_size=4, dtype="fp32",
              bias=True)
    import expert_token_dispatch_gemm_b300 as moe
    from moe_gpu_harness import make_cfg
    cfg = make_cfg(shape)
    idx = torch.empty((4096, 2), dtype=torch.int32, device="cuda")
    tw = torch.empty((4096, 2), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, x.cuda(), w.cuda(), b.cuda(), idx, tw)
    torch.cuda.synchronize()
    counts = np.bincount(idx.cpu().numpy().ravel(), minlength=8)
    parts = np.bincount(idx.cpu().numpy().ravel() // 2, minlength=4)
    assert (counts.min(), counts.max(), counts.sum()) == (948, 1087, 8192)
    assert (parts.min(), parts.max()) == (1968, 2139)


FULL = [workloads.GPTOSS, workloads.E8_TOP2, workloads.SKEWED_CAP, workloads.DECODE]


@pytest.mark.parametrize("shape", FULL, ids=lambda s: s.name)
def test_full_size_workload(shape):
    torch.manual_seed(0)
    inp = workloads.layer_inputs(shape, seed=0, variant="exact", device="cuda")
    layer = Layer(shape, inp)
    del inp
    out, diag = layer.forward()
    ref = full_size_reference_routing(layer)
    assert_routing_and_layout_exact(diag, ref, shape)
    rng = np.random.default_rng(0)
    n_sample = min(shape.N, 48)
    sample = np.sort(rng.choice(shape.N, n_sample, replace=False))
    if ref["capacity"] is not None:   # add tokens with dropped pairs
        sp = ref["slot_pos"].reshape(shape.N, shape.top_k)
        dropped_tokens = np.nonzero((sp < 0).any(axis=1))[0]
        assert dropped_tokens.size > 0
        sample = np.unique(np.concatenate([sample, dropped_tokens[:8], dropped_tokens[-8:]]))
    sampled_token_check(layer, diag, out, ref, sample, tol_for(shape))
    assert layer.device_status() == 0
