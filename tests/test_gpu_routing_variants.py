"""Routing variants on the GPU, through the C ABI, against the fp64 oracle
(Ultralytics glossary "Expert Parallelism", "Load balancing and capacity": DeepSeek-V3's
selection-only bias, updated after each step, and its limit on the nodes a token uses).

Bars as for the plain layer: routing ids, counts, offsets, perm and slot_pos bit-exact
on the exact variant (dyadic inputs and a selection bias on the 2^-10 grid, so logits
and selection scores are exact in fp32), outputs within the dtype's tolerance. The
shapes cover the tensor-core router with four and two column slices, a top-k longer
than 8, the fp32 router, and up to 64 partitions.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_gpu_harness import Layer, assert_close, assert_routing_and_layout_exact, oracle_layer, tol_for

pytestmark = pytest.mark.gpu

S = workloads.LayerShape
SHAPES = [
    # tiles fit one CTA per SM: four column slices
    S("v_bf16_e16_k4", N=600, H=128, I=64, E=16, top_k=4, ep_size=8),
    # more tiles than SMs: two column slices
    S("v_bf16_many_tiles", N=19200, H=64, I=32, E=32, top_k=2, ep_size=4, bias=True),
    # top-k longer than 8: a single slice
    S("v_bf16_k12", N=300, H=64, I=32, E=64, top_k=12, ep_size=8),
    # fp32 layers: the FFMA router
    S("v_fp32", N=333, H=96, I=72, E=8, top_k=2, ep_size=4, dtype="fp32", bias=True),
    S("v_fp32_p64", N=200, H=64, I=32, E=64, top_k=2, ep_size=64, dtype="fp32"),
]
VARIANTS = [("selection_bias", None), ("group_limit", 2), ("both", 2), ("both_one_group", 1)]


def _bias(shape, seed, scale=0.05):
    rng = np.random.default_rng(seed)
    return np.round(rng.uniform(-scale, scale, shape.E) * 1024) / 1024   # 2^-10 grid


def _group(shape, m):
    per = shape.E // shape.ep_size
    return max(m, -(-shape.top_k // per))   # enough experts for top_k


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: v[0])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_routing_variant_matches_oracle(shape, variant):
    name, m = variant
    inp = workloads.layer_inputs(shape, seed=31, variant="exact")
    beta = None if name == "group_limit" else _bias(shape, 5)
    gl = 0 if m is None else _group(shape, m)
    ref = oracle_layer(shape, inp, group_limit=gl, selection_bias=beta)
    layer = Layer(shape, inp, group_limit=gl, selection_bias=beta)
    out, diag = layer.forward()
    assert layer.device_status() == 0
    assert_routing_and_layout_exact(diag, ref, shape)
    np.testing.assert_allclose(diag["topk_w"].cpu().numpy(), ref["topk_w"], rtol=2e-6, atol=1e-7)
    assert_close(out, ref["out"], tol_for(shape))


def test_selection_bias_forces_an_expert_but_not_its_weight():
    shape = SHAPES[0]
    inp = workloads.layer_inputs(shape, seed=32, variant="exact")
    beta = np.zeros(shape.E)
    beta[5] = 64.0        # every token selects expert 5 first
    layer = Layer(shape, inp, selection_bias=beta)
    out, diag = layer.forward()
    idx = diag["topk_idx"].cpu().numpy()
    assert np.all(idx[:, 0] == 5)
    ref = oracle_layer(shape, inp, selection_bias=beta)
    assert_routing_and_layout_exact(diag, ref, shape)
    np.testing.assert_allclose(diag["topk_w"].cpu().numpy(), ref["topk_w"], rtol=2e-6, atol=1e-7)
    assert_close(out, ref["out"], tol_for(shape))


def test_group_limited_mask_and_sum_mode():
    shape = SHAPES[0]
    inp = workloads.layer_inputs(shape, seed=33, variant="exact")
    ref = oracle_layer(shape, inp, mode="mask_sum", group_limit=3)
    layer = Layer(shape, inp, mode="mask_sum", group_limit=3)
    out, diag = layer.forward()
    assert_routing_and_layout_exact(diag, ref, shape)
    assert_close(out, ref["out"], tol_for(shape))


@pytest.mark.parametrize("E,N,k", [(64, 4096, 8), (7, 5, 3), (256, 1000, 32)])
def test_selection_bias_update_is_bit_exact(E, N, k):
    import expert_token_dispatch_gemm_b300 as moe
    rng = np.random.default_rng(E)
    share = N * k // E
    counts = rng.integers(max(0, share - 3), share + 4, E).astype(np.int32)
    counts[0] = N * k / E if (N * k) % E == 0 else counts[0]
    beta = rng.standard_normal(E).astype(np.float32)
    gamma = 1e-3
    ref = oracle.update_selection_bias(beta, counts, N, k, gamma)
    cfg = moe.config(N, 64, 64, E, k, 1)
    d_counts = torch.from_numpy(counts).cuda()
    d_beta = torch.from_numpy(beta.copy()).cuda()
    moe.moe_update_selection_bias(cfg, d_counts, d_beta, gamma)
    torch.cuda.synchronize()
    got = d_beta.cpu().numpy()
    assert got.tobytes() == ref.tobytes()
