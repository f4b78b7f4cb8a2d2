"""Parity at full size on the inputs the benchmark times: the perf variant (continuous
values, seed 0) of every workload, in the benchmark's launch configuration, through the
C ABI.

With continuous inputs the fp32 router logits differ from the fp64 oracle's by rounding,
so the routing is unique only where the oracle's logit gaps exceed that rounding. Per
token t the error of any order of fp32 summation of the H products and the bias is at
most (H + 1) u sum_h |x_th w_eh| + |b_e| u with u = 2^-24 (the standard bound for a
recursive sum); it is doubled here, to 2^-23, to cover accumulators that do not round
to nearest:  bound_t = (H + 1) 2^-23 max_e (sum_h |x_th w_eh| + |b_e|).
Checks, per workload:
  1. every logit the GPU router produced is within bound_t of the oracle's;
  2. tokens whose oracle gaps among the k + 1 best logits all exceed 2 bound_t ("clear"
     tokens): topk_idx equal to the oracle's, topk_w within 2 bound_t + 2e-6;
  3. every other token: the GPU's choice is valid (distinct ids, each chosen logit within
     2 bound_t of the oracle's k-th best, in descending order up to 2 bound_t);
  4. the dispatch layout (counts, offsets, perm, slot_pos) bit-exact against the
     oracle's dispatch of the GPU's own routing ids (dispatch is integer work on them);
  5. outputs of >= 48 sampled clear tokens (plus clear tokens with dropped pairs on the
     skewed + capacity workload) within 2e-2 max|ref| (bf16) or 1e-4 max|ref| (fp32) of
     the oracle evaluated token by token, with the keep decisions of 4.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from moe_gpu_harness import Layer, assert_close, f64, tol_for

pytestmark = pytest.mark.gpu

CASES = [(workloads.PR1_FP32, "dispatch"), (workloads.GPTOSS, "dispatch"),
         (workloads.GPTOSS, "mask_sum"), (workloads.E8_TOP2, "dispatch"),
         (workloads.SKEWED_CAP, "dispatch"), (workloads.DECODE, "dispatch")]


def _bound(x, wr, b, H):
    s = np.abs(x) @ np.abs(wr).T
    if b is not None:
        s = s + np.abs(b)[None, :]
    return (H + 1) * 2.0 ** -23 * s.max(axis=1)


@pytest.mark.parametrize("shape,mode", CASES, ids=lambda v: getattr(v, "name", v))
def test_perf_inputs_full_size(shape, mode):
    torch.manual_seed(0)
    inp = workloads.layer_inputs(shape, seed=0, variant="perf", device="cuda")
    layer = Layer(shape, inp, mode)
    del inp
    N, E, k, P = shape.N, shape.E, shape.top_k, shape.ep_size
    d = layer.diag_buffers()
    d["router_logits"] = torch.full((N, E), float("nan"), device="cuda")
    out = torch.full((N, shape.H), float("nan"), dtype=shape.torch_dtype, device="cuda")
    import expert_token_dispatch_gemm_b300 as moe
    moe.moe_layer_forward(layer.cfg, layer.x, layer.w_router, layer.b_router, layer.packed,
                          layer.w_down, out, layer.ws, d)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    g = {key: v.cpu().numpy() for key, v in d.items()}

    x, wr = f64(layer.x), f64(layer.w_router)
    b = None if layer.b_router is None else f64(layer.b_router)
    logits = oracle.router_logits(x, wr, b)
    bound = _bound(x, wr, b, shape.H)
    # 1. the router's logits
    dev = np.abs(g["router_logits"].astype(np.float64) - logits)
    assert np.all(dev <= bound[:, None]), f"logit error {dev.max():.3e} beyond the bound"

    # 2. clear tokens: routing unique
    srt = -np.sort(-logits, axis=1)
    top = srt[:, :min(k + 1, E)]
    gaps = top[:, :-1] - top[:, 1:]
    clear = np.all(gaps > 2 * bound[:, None], axis=1) if gaps.size else np.ones(N, bool)
    assert clear.mean() > 0.5, f"only {clear.mean():.2f} of the tokens have clear routing"
    ref_idx = oracle.top_k_experts(logits, k)
    ref_w = oracle.routing_weights(logits, ref_idx)
    np.testing.assert_array_equal(g["topk_idx"][clear], ref_idx[clear])
    werr = np.abs(g["topk_w"][clear] - ref_w[clear])
    assert np.all(werr <= 2 * bound[clear, None] + 2e-6), f"topk_w error {werr.max():.3e}"

    # 3. near ties: any valid choice
    gi = g["topk_idx"].astype(np.int64)
    assert np.all((gi >= 0) & (gi < E))
    if k > 1:
        ids = np.sort(gi, axis=1)
        assert np.all(ids[:, 1:] != ids[:, :-1]), "an expert chosen twice"
    chosen = np.take_along_axis(logits, gi, axis=1)
    assert np.all(chosen >= srt[:, k - 1:k] - 2 * bound[:, None])
    if k > 1:
        assert np.all(chosen[:, 1:] <= chosen[:, :-1] + 2 * bound[:, None])

    # 4. dispatch of the GPU's routing
    C = oracle.expert_capacity(shape.capacity_factor, N, k, E)
    lay = oracle.dispatch_layout(gi, E, P, C)
    for key in ("routed_counts", "counts", "expert_offsets", "part_offsets", "slot_pos"):
        np.testing.assert_array_equal(g[key], lay[key], err_msg=key)
    kept = int(lay["expert_offsets"][-1])
    np.testing.assert_array_equal(g["perm"][:kept], lay["perm"])

    # 5. sampled outputs of clear tokens
    rng = np.random.default_rng(0)
    pool = np.nonzero(clear)[0]
    sample = np.sort(rng.choice(pool, min(pool.size, 48), replace=False))
    keep = lay["slot_pos"].reshape(N, k) >= 0
    if C is not None:
        dropped = np.nonzero(clear & ~keep.all(axis=1))[0]
        assert dropped.size > 0
        sample = np.unique(np.concatenate([sample, dropped[:8], dropped[-8:]]))

    def weights(e):
        return f64(layer.w_gate[e]), f64(layer.w_up[e]), f64(layer.w_down[e])

    ref = oracle.token_outputs(x[sample], ref_idx[sample], ref_w[sample], keep[sample], weights)
    assert_close(out[torch.as_tensor(sample, device="cuda")], ref, tol_for(shape),
                 f"{shape.name} {mode} sampled out")
