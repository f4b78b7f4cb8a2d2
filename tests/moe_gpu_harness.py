"""Runs the CUDA library (through its C ABI) and the fp64 oracle on the same seeded
inputs, and compares them. Used by the -m gpu tests and by the smoke check."""
from __future__ import annotations

import numpy as np
import torch

import expert_token_dispatch_gemm_b300 as moe
import oracle
import workloads

BF16_TOL = 2e-2    # max|err| <= BF16_TOL * max|ref| for bf16 layers
FP32_TOL = 1e-4    # max|err| <= FP32_TOL * max|ref| for fp32 layers


def tol_for(shape) -> float:
    return BF16_TOL if shape.dtype == "bf16" else FP32_TOL


def make_cfg(shape, mode="dispatch", N=None, group_limit=0, selection_bias=None,
             capacity_priority="token"):
    return moe.config(shape.N if N is None else N, shape.H, shape.I, shape.E, shape.top_k,
                      shape.ep_size, shape.capacity_factor, mode, shape.dtype,
                      has_bias=shape.bias or shape.zipf_s is not None,
                      group_limit=group_limit, selection_bias=selection_bias,
                      capacity_priority=capacity_priority)


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


class Layer:
    """Device copies of one layer's inputs plus packed weights and a workspace."""

    def __init__(self, shape, inputs, mode="dispatch", group_limit=0, selection_bias=None,
                 capacity_priority="token"):
        self.shape, self.mode = shape, mode
        dev = "cuda"
        # the config holds the selection bias' device address: keep the tensor alive
        self.sel_bias = (None if selection_bias is None
                         else torch.as_tensor(selection_bias, dtype=torch.float32).to(dev))
        self.cfg = make_cfg(shape, mode, group_limit=group_limit, selection_bias=self.sel_bias,
                            capacity_priority=capacity_priority)
        self.x = inputs["x"].to(dev).contiguous()
        self.w_router = inputs["w_router"].to(dev).contiguous()
        b = inputs["b_router"]
        self.b_router = None if b is None else b.to(dev, torch.float32).contiguous()
        self.w_gate = inputs["w_gate"].to(dev).contiguous()
        self.w_up = inputs["w_up"].to(dev).contiguous()
        self.w_down = inputs["w_down"].to(dev).contiguous()
        self.packed = moe.moe_pack_weights(self.cfg, self.w_gate, self.w_up)
        self.ws = moe.alloc_workspace(self.cfg)

    def diag_buffers(self):
        s = self.shape
        i32 = dict(dtype=torch.int32, device="cuda")
        pairs = s.N * s.top_k
        return dict(topk_idx=torch.full((s.N, s.top_k), -7, **i32),
                    topk_w=torch.full((s.N, s.top_k), -1.0, dtype=torch.float32, device="cuda"),
                    routed_counts=torch.full((s.E,), -7, **i32),
                    counts=torch.full((s.E,), -7, **i32),
                    expert_offsets=torch.full((s.E + 1,), -7, **i32),
                    part_offsets=torch.full((s.ep_size + 1,), -7, **i32),
                    perm=torch.full((pairs,), -7, **i32),
                    slot_pos=torch.full((pairs,), -7, **i32))

    def forward(self, with_diag=True):
        s = self.shape
        out = torch.full((s.N, s.H), float("nan"), dtype=s.torch_dtype, device="cuda")
        diag = self.diag_buffers() if with_diag else None
        moe.moe_layer_forward(self.cfg, self.x, self.w_router, self.b_router, self.packed,
                              self.w_down, out, self.ws, diag)
        torch.cuda.synchronize()
        return out, diag

    def steps(self, per_partition=False):
        """The same layer through the four step entry points."""
        s = self.shape
        d = self.diag_buffers()
        pairs = s.N * s.top_k
        moe.moe_route(self.cfg, self.x, self.w_router, self.b_router, d["topk_idx"], d["topk_w"])
        send = torch.zeros((pairs, s.H), dtype=s.torch_dtype, device="cuda")
        moe.moe_dispatch(self.cfg, d["topk_idx"], self.x, d["routed_counts"], d["counts"],
                         d["expert_offsets"], d["part_offsets"], d["perm"], d["slot_pos"], send,
                         self.ws)
        slots = torch.zeros((pairs, s.H), dtype=s.torch_dtype, device="cuda")
        ranges = ([(p * s.E // s.ep_size, (p + 1) * s.E // s.ep_size) for p in range(s.ep_size)]
                  if per_partition else [(0, s.E)])
        for b, e in ranges:
            moe.moe_expert_ffn(self.cfg, send, d["expert_offsets"], b, e, self.packed,
                               self.w_down, d["perm"], d["topk_w"], slots, self.ws)
        out = torch.full((s.N, s.H), float("nan"), dtype=s.torch_dtype, device="cuda")
        moe.moe_combine(self.cfg, slots, d["topk_idx"], d["slot_pos"], out, self.ws)
        torch.cuda.synchronize()
        return out, d, send, slots

    def device_status(self):
        return moe.moe_read_device_status(self.cfg, self.ws, reset=True)


def oracle_layer(shape, inputs, mode="dispatch", group_limit=None, selection_bias=None,
                 capacity_priority="token"):
    b = inputs["b_router"]
    return oracle.layer_forward(f64(inputs["x"]), f64(inputs["w_router"]),
                                None if b is None else f64(b), f64(inputs["w_gate"]),
                                f64(inputs["w_up"]), f64(inputs["w_down"]), shape.top_k,
                                shape.ep_size, shape.capacity_factor, mode,
                                selection_bias=(None if selection_bias is None
                                                else np.asarray(selection_bias, np.float64)),
                                group_limit=group_limit or None,
                                capacity_priority=capacity_priority)


def assert_routing_and_layout_exact(diag, ref, shape):
    """Integer outputs bit-exact; routing weights to fp32 rounding."""
    g = {k: v.cpu().numpy() for k, v in diag.items()}
    np.testing.assert_array_equal(g["topk_idx"], ref["topk_idx"])
    np.testing.assert_allclose(g["topk_w"], ref["topk_w"], rtol=0, atol=2e-6)
    np.testing.assert_array_equal(g["routed_counts"], ref["routed_counts"])
    np.testing.assert_array_equal(g["counts"], ref["counts"])
    np.testing.assert_array_equal(g["expert_offsets"], ref["expert_offsets"])
    np.testing.assert_array_equal(g["part_offsets"], ref["part_offsets"])
    kept = int(ref["expert_offsets"][-1])
    np.testing.assert_array_equal(g["perm"][:kept], ref["perm"])
    np.testing.assert_array_equal(g["slot_pos"], ref["slot_pos"])


def assert_close(got, ref, tol, what="out"):
    got = f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert err <= tol * max(scale, 1e-30), f"{what}: max|err| {err:.3e} > {tol} * {scale:.3e}"
    return err, scale


def routing_margin(logits, k):
    """Smallest gap between the k-th and (k+1)-th logit and between consecutive chosen
    logits: routing is insensitive to fp32 rounding where this is large."""
    s = -np.sort(-logits, axis=1)
    gaps = s[:, :-1] - s[:, 1:]
    return float(gaps[:, :min(k, gaps.shape[1])].min()) if gaps.size else np.inf


def sampled_token_check(layer, diag, out, ref_route, sample, tol, expert_chunk=None):
    """Output of `sample` tokens against the oracle evaluated token by token, with the
    oracle's own routing and keep decisions (from its full-batch dispatch layout)."""
    s = layer.shape
    idx = ref_route["topk_idx"][sample]
    w = ref_route["topk_w"][sample]
    keep = (ref_route["slot_pos"].reshape(s.N, s.top_k) >= 0)[sample]
    x_rows = f64(layer.x[torch.as_tensor(sample, device="cuda")])

    def weights(e):
        return f64(layer.w_gate[e]), f64(layer.w_up[e]), f64(layer.w_down[e])

    ref = oracle.token_outputs(x_rows, idx, w, keep, weights)
    got = out[torch.as_tensor(sample, device="cuda")]
    return assert_close(got, ref, tol, "sampled out")


def full_size_reference_routing(layer):
    """Oracle routing + dispatch layout for the whole batch (fp64 on the host)."""
    s = layer.shape
    x = f64(layer.x)
    b = None if layer.b_router is None else f64(layer.b_router)
    logits, idx, w = oracle.route(x, f64(layer.w_router), b, s.top_k)
    C = oracle.expert_capacity(s.capacity_factor, s.N, s.top_k, s.E)
    lay = oracle.dispatch_layout(idx, s.E, s.ep_size, C)
    return dict(logits=logits, topk_idx=idx, topk_w=w, capacity=C, **lay)
