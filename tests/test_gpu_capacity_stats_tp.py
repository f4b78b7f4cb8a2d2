"""Slot-major capacity priority, router load statistics and the TP row split on the
GPU, through the C ABI, against the fp64 oracle.

* Slot-major priority (GShard-style; Ultralytics glossary "Expert Parallelism", "Load
  balancing and capacity"): routing, counts, offsets, perm and slot_pos bit-exact on
  the exact input variant, outputs within the dtype's tolerance; both modes, both
  dtypes, through moe_layer_forward and through moe_dispatch.
* Load statistics: the router logits (exact variant: bit-exact), load shares and mean
  router probabilities (fp32 rounding of a fp64 mean: 1e-5 relative).
* TP row split (Hugging Face docs "Expert parallelism", "With tensor parallelism"): one
  layer call per token slice into zero-padded outputs, then moe_tp_reduce; uneven and
  empty slices and a single decode token.
"""
import numpy as np
import pytest
import torch

import expert_token_dispatch_gemm_b300 as moe
import oracle
import workloads
from moe_gpu_harness import (Layer, assert_close, assert_routing_and_layout_exact, f64,
                             make_cfg, oracle_layer, tol_for)

pytestmark = pytest.mark.gpu

S = workloads.LayerShape
PRIORITY_SHAPES = [
    S("p_bf16_cap", N=1000, H=128, I=64, E=16, top_k=4, ep_size=4, capacity_factor=0.8),
    S("p_bf16_tight", N=4500, H=64, I=32, E=8, top_k=2, ep_size=2, capacity_factor=0.3,
      bias=True),
    S("p_bf16_k8_skew", N=2048, H=128, I=64, E=64, top_k=8, ep_size=8, capacity_factor=1.25,
      zipf_s=1.1),
    S("p_bf16_nocap", N=777, H=64, I=32, E=8, top_k=3, ep_size=4),
    S("p_fp32_cap", N=613, H=96, I=72, E=8, top_k=2, ep_size=4, capacity_factor=0.6,
      dtype="fp32", bias=True),
    S("p_one_token", N=1, H=64, I=32, E=4, top_k=2, ep_size=2, capacity_factor=0.5),
    # more slots per token than the register-list combine kernels take (k > 8), and the
    # most (k = 32): spans of 64k tokens, k segments each
    S("p_bf16_k12_cap", N=1500, H=136, I=32, E=32, top_k=12, ep_size=4, capacity_factor=0.9),
    S("p_bf16_k32_cap", N=300, H=64, I=32, E=64, top_k=32, ep_size=8, capacity_factor=1.1),
]


@pytest.mark.parametrize("mode", ["dispatch", "mask_sum"])
@pytest.mark.parametrize("shape", PRIORITY_SHAPES, ids=lambda s: s.name)
def test_slot_priority_layer_matches_oracle(shape, mode):
    inp = workloads.layer_inputs(shape, seed=41, variant="exact")
    ref = oracle_layer(shape, inp, mode=mode, capacity_priority="slot")
    layer = Layer(shape, inp, mode=mode, capacity_priority="slot")
    out, diag = layer.forward()
    assert layer.device_status() == 0
    assert_routing_and_layout_exact(diag, ref, shape)
    assert_close(out, ref["out"], tol_for(shape))


def test_slot_priority_keeps_other_pairs_than_token_priority():
    shape = PRIORITY_SHAPES[1]
    inp = workloads.layer_inputs(shape, seed=42, variant="exact")
    a = Layer(shape, inp, capacity_priority="token").forward()[1]["slot_pos"].cpu().numpy()
    b = Layer(shape, inp, capacity_priority="slot").forward()[1]["slot_pos"].cpu().numpy()
    assert (a >= 0).sum() == (b >= 0).sum()          # the same kept counts per expert
    assert not np.array_equal(a >= 0, b >= 0)        # but other pairs


@pytest.mark.parametrize("shape", PRIORITY_SHAPES[:3], ids=lambda s: s.name)
def test_slot_priority_dispatch_entry_point(shape):
    inp = workloads.layer_inputs(shape, seed=43, variant="exact")
    ref = oracle_layer(shape, inp, capacity_priority="slot")
    layer = Layer(shape, inp, capacity_priority="slot")
    _, d, send, _ = layer.steps()
    assert_routing_and_layout_exact(d, ref, shape)
    kept = int(ref["expert_offsets"][-1])
    np.testing.assert_array_equal(f64(send[:kept]), ref["send"])


def test_slot_priority_noalloc_dispatch():
    shape = PRIORITY_SHAPES[2]
    inp = workloads.layer_inputs(shape, seed=44, variant="exact")
    ref = oracle_layer(shape, inp, capacity_priority="slot")
    layer = Layer(shape, inp, capacity_priority="slot")
    d = layer.diag_buffers()
    moe.moe_route(layer.cfg, layer.x, layer.w_router, layer.b_router, d["topk_idx"], d["topk_w"])
    send = torch.zeros((shape.N * shape.top_k, shape.H), dtype=shape.torch_dtype, device="cuda")
    moe.moe_dispatch_noalloc(layer.cfg, d["topk_idx"], layer.x, d["routed_counts"], d["counts"],
                             d["expert_offsets"], d["part_offsets"], d["perm"], d["slot_pos"],
                             send)
    torch.cuda.synchronize()
    assert_routing_and_layout_exact(d, ref, shape)


# ------------------------------------------------------------------ load statistics
STAT_SHAPES = [
    S("s_bf16_e128", N=3000, H=256, I=32, E=128, top_k=4, ep_size=8),       # 2 slices
    S("s_bf16_e16", N=700, H=128, I=32, E=16, top_k=2, ep_size=4, bias=True),
    S("s_bf16_e20", N=300, H=64, I=32, E=20, top_k=2, ep_size=4),            # E % 4 != 0
    S("s_fp32_e8", N=513, H=96, I=32, E=8, top_k=2, ep_size=2, dtype="fp32", bias=True),
    S("s_bf16_group", N=640, H=64, I=32, E=64, top_k=4, ep_size=8),
]


@pytest.mark.parametrize("shape", STAT_SHAPES, ids=lambda s: s.name)
def test_router_logits_and_balance_stats_match_oracle(shape):
    inp = workloads.layer_inputs(shape, seed=45, variant="exact")
    gl = 2 if shape.name == "s_bf16_group" else 0
    ref = oracle_layer(shape, inp, group_limit=gl)
    layer = Layer(shape, inp, group_limit=gl)
    d = layer.diag_buffers()
    d["router_logits"] = torch.full((shape.N, shape.E), float("nan"), device="cuda")
    out = torch.empty((shape.N, shape.H), dtype=shape.torch_dtype, device="cuda")
    moe.moe_layer_forward(layer.cfg, layer.x, layer.w_router, layer.b_router, layer.packed,
                          layer.w_down, out, layer.ws, d)
    load = torch.full((shape.E,), float("nan"), device="cuda")
    prob = torch.full((shape.E,), float("nan"), device="cuda")
    moe.moe_balance_stats(layer.cfg, d["router_logits"], d["routed_counts"], load, prob, layer.ws)
    torch.cuda.synchronize()
    # exact variant: every logit is exact in fp32
    np.testing.assert_array_equal(d["router_logits"].cpu().numpy().astype(np.float64),
                                  ref["logits"])
    st = oracle.balance_stats(ref["logits"], ref["routed_counts"], shape.N, shape.top_k)
    np.testing.assert_allclose(f64(load), st["load_frac"], rtol=1e-7, atol=0)
    np.testing.assert_allclose(f64(prob), st["prob_mean"], rtol=1e-5, atol=1e-9)
    assert abs(float(prob.sum()) - 1.0) < 1e-5


def test_balance_stats_of_an_empty_batch_are_zero():
    shape = STAT_SHAPES[1]
    cfg = make_cfg(shape, N=0)
    ws = moe.alloc_workspace(cfg)
    load = torch.full((shape.E,), 5.0, device="cuda")
    prob = torch.full((shape.E,), 5.0, device="cuda")
    counts = torch.zeros(shape.E, dtype=torch.int32, device="cuda")
    moe.moe_balance_stats(cfg, None, counts, load, prob, ws)
    torch.cuda.synchronize()
    assert not load.any() and not prob.any()


# ------------------------------------------------------------------ TP row split
TP_SHAPES = [
    S("t_bf16", N=1001, H=128, I=64, E=16, top_k=4, ep_size=4),
    S("t_bf16_cap", N=900, H=64, I=32, E=8, top_k=2, ep_size=2, capacity_factor=0.7, bias=True),
    S("t_fp32", N=301, H=96, I=72, E=8, top_k=2, ep_size=4, dtype="fp32"),
    S("t_decode", N=1, H=128, I=64, E=16, top_k=4, ep_size=4),
]


def _tp_forward(shape, inp, tp, mode):
    dev = "cuda"
    padded = torch.zeros((tp, shape.N, shape.H), dtype=shape.torch_dtype, device=dev)
    full = Layer(shape, inp, mode=mode)      # device copies of the weights, packed once
    for s in range(tp):
        b, e = moe.moe_tp_slice(shape.N, tp, s)
        if e == b:
            continue                          # an empty slice dispatches nothing
        sub = shape.replace(N=e - b)
        cfg = make_cfg(sub, mode)
        ws = moe.alloc_workspace(cfg)
        moe.moe_layer_forward(cfg, full.x[b:e], full.w_router, full.b_router, full.packed,
                              full.w_down, padded[s, b:e], ws)
    out = torch.full((shape.N, shape.H), float("nan"), dtype=shape.torch_dtype, device=dev)
    moe.moe_tp_reduce(full.cfg, tp, padded, out)
    torch.cuda.synchronize()
    return padded, out


@pytest.mark.parametrize("tp", [2, 3, 4])
@pytest.mark.parametrize("mode", ["dispatch", "mask_sum"])
@pytest.mark.parametrize("shape", TP_SHAPES, ids=lambda s: s.name)
def test_tp_row_split_matches_oracle(shape, mode, tp):
    inp = workloads.layer_inputs(shape, seed=46, variant="exact")
    padded, out = _tp_forward(shape, inp, tp, mode)
    b = inp["b_router"]
    ref_pad, ref = oracle.tp_row_split_forward(
        f64(inp["x"]), f64(inp["w_router"]), None if b is None else f64(b), f64(inp["w_gate"]),
        f64(inp["w_up"]), f64(inp["w_down"]), shape.top_k, shape.ep_size, tp,
        shape.capacity_factor, mode)
    assert_close(out, ref, tol_for(shape))
    # the padded sum adds exact zeros: out is bitwise each slice's own rows
    for s in range(tp):
        lo, hi = moe.moe_tp_slice(shape.N, tp, s)
        assert torch.equal(out[lo:hi], padded[s, lo:hi])


@pytest.mark.parametrize("shape", [workloads.SKEWED_CAP, workloads.GPTOSS], ids=lambda s: s.name)
def test_slot_priority_at_full_size(shape):
    """Slot-major priority on the full skewed + capacity workload (where the keep set
    depends on it) and the gpt-oss workload, in the bench's launch configuration:
    routing and the whole dispatch layout bit-exact against the oracle's full-batch
    layout, outputs on sampled tokens (tokens with dropped pairs included)."""
    from moe_gpu_harness import full_size_reference_routing, sampled_token_check
    torch.manual_seed(0)
    inp = workloads.layer_inputs(shape, seed=0, variant="exact", device="cuda")
    layer = Layer(shape, inp, capacity_priority="slot")
    del inp
    out, diag = layer.forward()
    ref = full_size_reference_routing(layer)
    lay = oracle.dispatch_layout(ref["topk_idx"], shape.E, shape.ep_size, ref["capacity"],
                                 priority="slot")
    ref = dict(ref, **lay)
    assert_routing_and_layout_exact(diag, ref, shape)
    rng = np.random.default_rng(2)
    sample = np.sort(rng.choice(shape.N, 32, replace=False))
    if ref["capacity"] is not None:
        sp = ref["slot_pos"].reshape(shape.N, shape.top_k)
        dropped = np.nonzero((sp < 0).any(axis=1))[0]
        assert dropped.size > 0
        sample = np.unique(np.concatenate([sample, dropped[:8], dropped[-8:]]))
        tok = oracle.dispatch_layout(ref["topk_idx"], shape.E, shape.ep_size, ref["capacity"])
        assert not np.array_equal(tok["slot_pos"] >= 0, lay["slot_pos"] >= 0)
    sampled_token_check(layer, diag, out, ref, sample, tol_for(shape))
    assert layer.device_status() == 0
