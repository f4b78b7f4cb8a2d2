"""The tensor-core router's launch shapes, through moe_route (C ABI), against the fp64
oracle's routing (Ultralytics glossary "Expert Parallelism", "How tokens move between
GPUs", step 1) on the exact input variant: ids bit-exact, weights to fp32 rounding, and
the selection-bias variant's ids bit-exact.

The router picks its shape from the sizes: one CTA per 128-token tile, or, when there
are fewer tiles than SMs and at least two K blocks, a cluster of two CTAs per tile that
split the hidden dimension and exchange partial logits; four column slices when the
CTAs fit one per SM, two otherwise; a ring as deep as the shared memory allows (the
split falls back to one CTA per tile where two stages would not fit); plain top-k of up
to 4 by rank keys, longer lists by insertion. These shapes reach each of those paths
with ragged tails (token counts not multiples of 128, E not a multiple of 16 or 32).
"""
import numpy as np
import pytest
import torch

import expert_token_dispatch_gemm_b300 as moe
import oracle
import workloads
from moe_gpu_harness import f64, make_cfg

pytestmark = pytest.mark.gpu

S = workloads.LayerShape
SHAPES = [
    # split pairs, four slices: 256 expert columns (3 ring stages), keyed top-4
    S("r_split_e256_k4", N=515, H=320, I=32, E=256, top_k=4, ep_size=8),
    # split pairs, four slices, k = 8 by insertion, E = 40 (bn 48: a ragged slice)
    S("r_split_e40_k8", N=300, H=200, I=32, E=40, top_k=8, ep_size=8),
    # split pairs with exactly two K blocks (H = 128), one token
    S("r_split_two_kb_one_token", N=1, H=128, I=32, E=8, top_k=2, ep_size=2),
    # 74 .. 147 tiles: split pairs with two column slices (two CTAs per SM)
    S("r_split_two_slices", N=100 * 128 - 77, H=192, I=32, E=20, top_k=3, ep_size=4),
    # 74 .. 147 tiles at 256 experts: two stages do not fit a split pair, one CTA per tile
    S("r_fallback_e256", N=90 * 128 + 9, H=128, I=32, E=256, top_k=2, ep_size=8),
    # one K block (H = 64): never split
    S("r_one_kb", N=700, H=64, I=32, E=16, top_k=4, ep_size=4),
    # more tiles than SMs: one CTA per tile, two slices, keyed top-1
    S("r_many_tiles_k1", N=160 * 128 + 5, H=128, I=32, E=24, top_k=1, ep_size=4),
]


def _route(shape, inp, sel_bias=None):
    dev = "cuda"
    sb = None if sel_bias is None else torch.as_tensor(sel_bias, dtype=torch.float32).to(dev)
    cfg = make_cfg(shape, selection_bias=sb)
    idx = torch.full((shape.N, shape.top_k), -7, dtype=torch.int32, device=dev)
    w = torch.full((shape.N, shape.top_k), -1.0, dtype=torch.float32, device=dev)
    b = inp["b_router"]
    moe.moe_route(cfg, inp["x"].to(dev), inp["w_router"].to(dev),
                  None if b is None else b.to(dev, torch.float32), idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_router_paths_match_oracle(shape):
    inp = workloads.layer_inputs(shape, seed=71, variant="exact", with_experts=False)
    b = inp["b_router"]
    logits, idx, w = oracle.route(f64(inp["x"]), f64(inp["w_router"]),
                                  None if b is None else f64(b), shape.top_k)
    gi, gw = _route(shape, inp)
    np.testing.assert_array_equal(gi, idx)
    np.testing.assert_allclose(gw, w, rtol=0, atol=2e-6)


@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[3]], ids=lambda s: s.name)
def test_router_paths_with_selection_bias(shape):
    inp = workloads.layer_inputs(shape, seed=72, variant="exact", with_experts=False)
    rng = np.random.default_rng(73)
    sel = np.round(rng.uniform(-0.05, 0.05, shape.E) * 1024) / 1024   # 2^-10 grid
    b = inp["b_router"]
    logits, idx, w = oracle.route_variant(f64(inp["x"]), f64(inp["w_router"]),
                                          None if b is None else f64(b), shape.top_k,
                                          selection_bias=sel, ep_size=shape.ep_size)
    gi, gw = _route(shape, inp, sel)
    np.testing.assert_array_equal(gi, idx)
    np.testing.assert_allclose(gw, w, rtol=0, atol=2e-6)


def test_router_logits_exchange_is_symmetric():
    """Both CTAs of a split pair add the same two partials (own + received), so the
    logits the router writes equal the oracle's exactly on the exact variant, for tokens
    owned by either CTA of the pair."""
    shape = SHAPES[0]
    inp = workloads.layer_inputs(shape, seed=74, variant="exact", with_experts=False)
    cfg = make_cfg(shape)
    dev = "cuda"
    pairs = shape.N * shape.top_k
    i32 = dict(dtype=torch.int32, device=dev)
    d = dict(topk_idx=torch.empty((shape.N, shape.top_k), **i32),
             topk_w=torch.empty((shape.N, shape.top_k), dtype=torch.float32, device=dev),
             routed_counts=torch.empty(shape.E, **i32), counts=torch.empty(shape.E, **i32),
             expert_offsets=torch.empty(shape.E + 1, **i32),
             part_offsets=torch.empty(shape.ep_size + 1, **i32),
             perm=torch.empty(pairs, **i32), slot_pos=torch.empty(pairs, **i32),
             router_logits=torch.full((shape.N, shape.E), float("nan"), device=dev))
    full = workloads.layer_inputs(shape, seed=74, variant="exact")
    packed = moe.moe_pack_weights(cfg, full["w_gate"].to(dev), full["w_up"].to(dev))
    ws = moe.alloc_workspace(cfg)
    out = torch.empty((shape.N, shape.H), dtype=torch.bfloat16, device=dev)
    moe.moe_layer_forward(cfg, full["x"].to(dev), full["w_router"].to(dev), None, packed,
                          full["w_down"].to(dev), out, ws, d)
    torch.cuda.synchronize()
    ref = oracle.router_logits(f64(inp["x"]), f64(inp["w_router"]), None)
    np.testing.assert_array_equal(d["router_logits"].cpu().numpy().astype(np.float64), ref)
