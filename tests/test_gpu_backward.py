"""Backward of the layer on the GPU (moe_layer_backward), through the C ABI, against the
fp64 oracle's chain rule (oracle.layer_backward) on the same seeded inputs.

Bar: every gradient within 2e-2 * max|ref| for bf16 layers (the forward's bf16 rule: the
operands and the intermediate gradients are bf16, every product accumulates in fp32)
and 1e-4 * max|ref| for fp32 layers (the forward's fp32 rule).
Routing is exact on the dyadic input variant, so both sides differentiate the same
selection. The shapes span several M / N / K tiles with ragged tails (H and I not
multiples of 64 or 128), capacity drops, slot-major priority, mask-and-sum mode, a
single token, experts that receive no rows, segments of more than 256 and of more
than 512 rows, and more tiles than the GPU runs at once (persistent tile loops).
"""
import numpy as np
import pytest
import torch

import expert_token_dispatch_gemm_b300 as moe
import oracle
import workloads
from moe_gpu_harness import BF16_TOL, assert_close, f64, make_cfg, tol_for

pytestmark = pytest.mark.gpu

S = workloads.LayerShape
SHAPES = [
    S("b_e8_k2", N=600, H=256, I=192, E=8, top_k=2, ep_size=4, bias=True),
    S("b_ragged", N=777, H=200, I=136, E=16, top_k=4, ep_size=4),
    S("b_cap", N=900, H=128, I=256, E=8, top_k=2, ep_size=2, capacity_factor=0.6),
    S("b_skew_cap", N=1024, H=256, I=128, E=32, top_k=8, ep_size=8, capacity_factor=1.25,
      zipf_s=1.1),
    S("b_sparse", N=20, H=128, I=64, E=32, top_k=2, ep_size=8),     # most experts get no rows
    S("b_one", N=1, H=64, I=64, E=4, top_k=2, ep_size=2),
    S("b_long_seg", N=1200, H=192, I=320, E=4, top_k=1, ep_size=2),  # segments > 256 rows
    # segments of ~1150 rows: several 256-token tiles per expert
    S("b_multi_tile", N=2300, H=128, I=96, E=2, top_k=1, ep_size=2),
    # more tiles than clusters of two SMs in all four GEMMs: each cluster runs several
    # tiles, the ring and both accumulators cycle through several phases
    S("b_persistent", N=2048, H=512, I=256, E=64, top_k=8, ep_size=8),
    # the most experts the tile tables hold (256), ~16 rows each: most segments end
    # inside their only 64-row block of the transposed operands
    S("b_max_experts", N=512, H=128, I=64, E=256, top_k=8, ep_size=8),
    # the smallest hidden and intermediate sizes (8): one K block and one weight tile,
    # mostly outside the tensors
    S("b_min_sizes", N=300, H=8, I=8, E=4, top_k=2, ep_size=2, bias=True),
    # 33 vectors per row: the last pass of dx combine has one active lane for 4 slots
    S("b_ragged_rows", N=300, H=264, I=64, E=16, top_k=4, ep_size=4),
    # more slots per token than 8 (with drops), and the most (32)
    S("b_k12_cap", N=500, H=136, I=64, E=32, top_k=12, ep_size=4, capacity_factor=0.9),
    S("b_k32", N=200, H=64, I=32, E=64, top_k=32, ep_size=8),
    S("f_k12_cap", N=400, H=72, I=40, E=32, top_k=12, ep_size=4, capacity_factor=0.9,
      dtype="fp32", bias=True),
    # fp32 layers (FFMA kernels): ragged tiles, drops, the PR1 configuration
    S("f_ragged", N=333, H=96, I=72, E=8, top_k=2, ep_size=4, dtype="fp32", bias=True),
    S("f_cap", N=500, H=64, I=136, E=4, top_k=2, ep_size=2, capacity_factor=0.6, dtype="fp32"),
    workloads.PR1_FP32,
]


def _run(shape, inp, dout, mode="dispatch", capacity_priority="token", group_limit=0,
         selection_bias=None):
    dev = "cuda"
    cfg = make_cfg(shape, mode, capacity_priority=capacity_priority, group_limit=group_limit,
                   selection_bias=selection_bias)
    cfg.training = 1
    x = inp["x"].to(dev).contiguous()
    wr = inp["w_router"].to(dev).contiguous()
    b = inp["b_router"]
    br = None if b is None else b.to(dev, torch.float32).contiguous()
    wg, wu, wd = (inp[n].to(dev).contiguous() for n in ("w_gate", "w_up", "w_down"))
    packed = moe.moe_pack_weights(cfg, wg, wu)
    ws = moe.alloc_workspace(cfg)
    out = torch.empty((shape.N, shape.H), dtype=shape.torch_dtype, device=dev)
    moe.moe_layer_forward(cfg, x, wr, br, packed, wd, out, ws)
    g = dict(dx=torch.full_like(x, float("nan")),
             dw_router=torch.full((shape.E, shape.H), float("nan"), device=dev),
             db_router=torch.full((shape.E,), float("nan"), device=dev),
             dw_gate=torch.full_like(wg, float("nan")), dw_up=torch.full_like(wu, float("nan")),
             dw_down=torch.full_like(wd, float("nan")))
    moe.moe_layer_backward(cfg, x, wr, packed, wd, dout.to(dev).contiguous(), g["dx"],
                           g["dw_router"], g["db_router"], g["dw_gate"], g["dw_up"], g["dw_down"],
                           ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(cfg, ws) == 0
    return out, g


def _dout(shape, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn((shape.N, shape.H), generator=gen).to(shape.torch_dtype)


def _oracle(shape, inp, dout, capacity_priority="token", group_limit=None, selection_bias=None):
    b = inp["b_router"]
    return oracle.layer_backward(f64(inp["x"]), f64(inp["w_router"]), None if b is None else f64(b),
                                 f64(inp["w_gate"]), f64(inp["w_up"]), f64(inp["w_down"]),
                                 shape.top_k, shape.ep_size, f64(dout), shape.capacity_factor,
                                 selection_bias=selection_bias, group_limit=group_limit,
                                 capacity_priority=capacity_priority)


def _compare(g, ref, tol=BF16_TOL):
    for key in ("dx", "dw_router", "db_router", "dw_gate", "dw_up", "dw_down"):
        assert_close(g[key], ref[key], tol, key)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_layer_backward_matches_oracle(shape):
    inp = workloads.layer_inputs(shape, seed=51, variant="exact")
    dout = _dout(shape, 52)
    _, g = _run(shape, inp, dout)
    _compare(g, _oracle(shape, inp, dout), tol_for(shape))


def test_backward_with_slot_priority_and_mask_mode():
    shape = SHAPES[3]
    inp = workloads.layer_inputs(shape, seed=53, variant="exact")
    dout = _dout(shape, 54)
    _, g = _run(shape, inp, dout, mode="mask_sum", capacity_priority="slot")
    _compare(g, _oracle(shape, inp, dout, capacity_priority="slot"))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_backward_with_selection_bias_and_group_limit(dtype):
    """DeepSeek-V3-style routing (a selection-only bias, at most 2 partitions per token):
    the routing weights stay the softmax of the chosen experts' raw logits, so the same
    chain rule applies; the selection bias gets no gradient."""
    shape = S("b_variant", N=640, H=128, I=96, E=32, top_k=4, ep_size=8, capacity_factor=1.0,
              dtype=dtype)
    inp = workloads.layer_inputs(shape, seed=60, variant="exact")
    rng = np.random.default_rng(60)
    beta = np.round(rng.uniform(-0.05, 0.05, shape.E) * 1024) / 1024
    sel = torch.as_tensor(beta, dtype=torch.float32, device="cuda")
    dout = _dout(shape, 61)
    _, g = _run(shape, inp, dout, group_limit=2, selection_bias=sel)
    _compare(g, _oracle(shape, inp, dout, group_limit=2, selection_bias=beta), tol_for(shape))


def test_backward_is_deterministic():
    shape = SHAPES[1]
    inp = workloads.layer_inputs(shape, seed=55, variant="exact")
    dout = _dout(shape, 56)
    _, a = _run(shape, inp, dout)
    _, b = _run(shape, inp, dout)
    for key in a:
        assert torch.equal(a[key], b[key]), key


def test_experts_without_rows_get_zero_weight_gradients():
    shape = SHAPES[4]
    inp = workloads.layer_inputs(shape, seed=57, variant="exact")
    _, g = _run(shape, inp, _dout(shape, 58))
    ref = _oracle(shape, inp, _dout(shape, 58))
    empty = [e for e in range(shape.E) if not np.any(ref["dw_down"][e])]
    assert empty, "the shape should leave experts without rows"
    for e in empty:
        assert not g["dw_gate"][e].any() and not g["dw_up"][e].any() and not g["dw_down"][e].any()


def test_training_forward_output_and_diagnostics_are_unchanged():
    shape = SHAPES[0]
    inp = workloads.layer_inputs(shape, seed=59, variant="exact")
    dev = "cuda"
    outs = []
    for training in (0, 1):
        cfg = make_cfg(shape)
        cfg.training = training
        x = inp["x"].to(dev)
        wg, wu, wd = (inp[n].to(dev).contiguous() for n in ("w_gate", "w_up", "w_down"))
        packed = moe.moe_pack_weights(cfg, wg, wu)
        ws = moe.alloc_workspace(cfg)
        out = torch.empty((shape.N, shape.H), dtype=torch.bfloat16, device=dev)
        diag = dict(topk_idx=torch.empty((shape.N, shape.top_k), dtype=torch.int32, device=dev),
                    slot_pos=torch.empty(shape.N * shape.top_k, dtype=torch.int32, device=dev))
        moe.moe_layer_forward(cfg, x, inp["w_router"].to(dev), inp["b_router"].to(dev), packed, wd,
                              out, ws, diag)
        torch.cuda.synchronize()
        outs.append((out, diag))
    assert torch.equal(outs[0][0], outs[1][0])
    for key in ("topk_idx", "slot_pos"):
        assert torch.equal(outs[0][1][key], outs[1][1][key])


# ------------------------------------------------------------------ full size, sampled
FULL = [workloads.GPTOSS, workloads.E8_TOP2, workloads.SKEWED_CAP, workloads.DECODE]


def _sampled_experts(shape, counts):
    """The most loaded expert plus, where cheap enough in fp64 on the host, a median one
    (the 8-expert workload's experts hold ~4096 rows of 4096 x 14336: none is sampled)."""
    if shape.I * shape.H * int(counts.max()) > 3e10:
        return []
    order = np.argsort(counts, kind="stable")
    picks = [int(order[-1]), int(order[len(order) // 2])]
    return sorted(set(e for e in picks if counts[e] > 0))


@pytest.mark.parametrize("shape", FULL, ids=lambda s: s.name)
def test_full_size_backward_sampled(shape):
    """The bench's workloads at full size, in the bench's launch configuration (fused
    training forward, then moe_layer_backward): dx on sampled tokens (tokens with
    dropped pairs included) and the weight gradients of sampled experts against the
    oracle's per-token / per-expert chain rule, with the oracle's own routing and drops.
    The router weight gradient needs every pair's expert output, i.e. the whole fp64
    layer, so it is checked at the small sizes above only."""
    from moe_gpu_harness import Layer, full_size_reference_routing
    torch.manual_seed(0)
    inp = workloads.layer_inputs(shape, seed=0, variant="exact", device="cuda")
    layer = Layer(shape, inp)
    del inp
    layer.cfg.training = 1
    layer.ws = moe.alloc_workspace(layer.cfg)
    dout = _dout(shape, 61).cuda()
    out = torch.empty((shape.N, shape.H), dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_forward(layer.cfg, layer.x, layer.w_router, layer.b_router, layer.packed,
                          layer.w_down, out, layer.ws)
    g = dict(dx=torch.empty_like(layer.x),
             dw_router=torch.empty((shape.E, shape.H), device="cuda"),
             dw_gate=torch.empty_like(layer.w_gate), dw_up=torch.empty_like(layer.w_up),
             dw_down=torch.empty_like(layer.w_down))
    moe.moe_layer_backward(layer.cfg, layer.x, layer.w_router, layer.packed, layer.w_down,
                           dout, g["dx"], g["dw_router"], None, g["dw_gate"], g["dw_up"],
                           g["dw_down"], layer.ws)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    ref = full_size_reference_routing(layer)
    sp = ref["slot_pos"].reshape(shape.N, shape.top_k)
    rng = np.random.default_rng(1)
    sample = np.sort(rng.choice(shape.N, min(shape.N, 24), replace=False))
    if ref["capacity"] is not None:
        dropped = np.nonzero((sp < 0).any(axis=1))[0]
        assert dropped.size > 0
        sample = np.unique(np.concatenate([sample, dropped[:4], dropped[-4:]]))
    s_dev = torch.as_tensor(sample, device="cuda")

    def weights(e):
        return f64(layer.w_gate[e]), f64(layer.w_up[e]), f64(layer.w_down[e])

    want = oracle.token_input_grads(f64(layer.x[s_dev]), f64(dout[s_dev]), ref["topk_idx"][sample],
                                    ref["topk_w"][sample], sp[sample] >= 0, f64(layer.w_router),
                                    weights)
    assert_close(g["dx"][s_dev], want, BF16_TOL, "sampled dx")
    counts = np.asarray(ref["counts"])
    w_flat = np.asarray(ref["topk_w"]).reshape(-1)
    for e in _sampled_experts(shape, counts):
        a, z = int(ref["expert_offsets"][e]), int(ref["expert_offsets"][e + 1])
        pairs = np.asarray(ref["perm"][a:z])
        t_dev = torch.as_tensor(pairs // shape.top_k, device="cuda")
        dg, du, dd = oracle.expert_weight_grads(f64(layer.x[t_dev]), f64(dout[t_dev]),
                                                w_flat[pairs], *weights(e))
        assert_close(g["dw_gate"][e], dg, BF16_TOL, f"dW_gate[{e}]")
        assert_close(g["dw_up"][e], du, BF16_TOL, f"dW_up[{e}]")
        assert_close(g["dw_down"][e], dd, BF16_TOL, f"dW_down[{e}]")
