"""Seeded synthetic inputs for the MoE layer forward.

This module is shared by the tests, the benchmark and the smoke check. It only draws
random numbers and rounds them to the storage dtype: it holds none of the layer's
arithmetic (no routing, no counting, no expert math), so the oracle and the CUDA path
can both consume its tensors without sharing any computation.

Workload shapes follow the MoE layers the pages describe (expert-parallel MoE forward:
route -> dispatch -> local experts -> weighted combine). No dataset or trained weights
exist for them, so every tensor is drawn from the distribution stated per shape below.

Two value variants exist for every shape:
  * ``perf``  -- continuous values, used for timing and tolerance parity;
  * ``exact`` -- hidden states and router parameters on dyadic grids (multiples of a
    power of two), so that every fp32 partial sum of a router logit is exactly
    representable and routing must agree bit for bit with the fp64 oracle.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

# tensor ids mixed into the seed so every tensor draws from its own stream
_T_X, _T_WR, _T_B, _T_WG, _T_WU, _T_WD, _T_ZIPF = 1, 2, 3, 4, 5, 6, 7


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Sizes of one MoE layer forward call.

    N tokens of hidden size H; E experts, each a SwiGLU FFN with intermediate size I;
    top_k experts per token; ep_size logical expert-parallel partitions (experts split
    contiguously, E/ep_size each). capacity_factor None means no capacity limit.
    zipf_s adds a per-expert router-logit bias -s*ln(rank) (rank a seeded permutation
    of 1..E) so that a few experts are popular.
    """
    name: str
    N: int
    H: int
    I: int
    E: int
    top_k: int
    ep_size: int
    dtype: str = "bf16"            # "bf16" or "fp32": storage and I/O type
    bias: bool = False             # router bias drawn like nn.Linear's
    capacity_factor: Optional[float] = None
    zipf_s: Optional[float] = None
    x_std: float = 1.0             # hidden states ~ N(0, x_std^2)
    w_std: float = 0.02            # expert weights ~ N(0, w_std^2)

    def replace(self, **kw) -> "LayerShape":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


# The five workloads. The first is the routing example of the Ultralytics glossary page
# (4096 tokens x 512, router Linear 512->8 with bias, top-2, 4 partitions of 2 experts)
# extended with an FFN; the others are shaped like the MoE layers the pages name.
PR1_FP32 = LayerShape("pr1_fp32_n4096_h512_e8_k2", N=4096, H=512, I=256, E=8, top_k=2,
                      ep_size=4, dtype="fp32", bias=True)
GPTOSS = LayerShape("gptoss_n8192_h2880_e128_k4", N=8192, H=2880, I=2880, E=128, top_k=4,
                    ep_size=8)
E8_TOP2 = LayerShape("e8k2_n16384_h4096_i14336", N=16384, H=4096, I=14336, E=8, top_k=2,
                     ep_size=4)
SKEWED_CAP = LayerShape("skewed_cap_n32768_h2048_e64_k8", N=32768, H=2048, I=1408, E=64,
                        top_k=8, ep_size=8, capacity_factor=1.25, zipf_s=1.1)
DECODE = LayerShape("decode_n128_h2880_e128_k4", N=128, H=2880, I=2880, E=128, top_k=4,
                    ep_size=8)

ALL_SHAPES = (PR1_FP32, GPTOSS, E8_TOP2, SKEWED_CAP, DECODE)

# The gpt-oss-shaped layer scaled down to 16 experts and 1024 tokens: the same per-expert
# GEMM shapes (about 256 rows per expert) with ~1.5 GB on the device, small enough for
# full profiler captures.
GPTOSS_PROFILE = LayerShape("gptoss_profile_n1024_h2880_e16_k4", N=1024, H=2880, I=2880,
                            E=16, top_k=4, ep_size=8)

# The gpt-oss router (8192 tokens x 2880, 128 experts, top-4) in front of small experts
# (intermediate 128): under 1 GB on the device, for profiler captures of the routing and
# dispatch kernels at their full gpt-oss size.
ROUTE_PROFILE = LayerShape("route_profile_n8192_h2880_e128_k4", N=8192, H=2880, I=128,
                           E=128, top_k=4, ep_size=8)

# The decode router (128 tokens) in front of the same small experts.
ROUTE_PROFILE_DECODE = LayerShape("route_profile_n128_h2880_e128_k4", N=128, H=2880, I=128,
                                  E=128, top_k=4, ep_size=8)

# The 8-expert layer's per-expert GEMMs (4096 rows per expert, hidden 4096, intermediate
# 14336) on 2 experts: every token routes to both, ~1.5 GB on the device.
E8K2_PROFILE = LayerShape("e8k2_profile_n4096_h4096_e2_k2", N=4096, H=4096, I=14336, E=2,
                          top_k=2, ep_size=2)

# The skewed + capacity layer's per-expert GEMMs at its capacity (5120 rows per expert,
# hidden 2048, intermediate 1408) on 8 experts: every token routes to all 8, under 1 GB.
SKEWED_PROFILE = LayerShape("skewed_profile_n5120_h2048_e8_k8", N=5120, H=2048, I=1408, E=8,
                            top_k=8, ep_size=8)

PROFILE_SHAPES = (GPTOSS_PROFILE, ROUTE_PROFILE, ROUTE_PROFILE_DECODE, E8K2_PROFILE,
                  SKEWED_PROFILE)
BY_NAME = {s.name: s for s in ALL_SHAPES + PROFILE_SHAPES}


def _gen(seed: int, tensor_id: int, device, sub: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(1_000_003 * int(seed) + 7919 * tensor_id + 104_729 * sub + 17)
    return g


def _round_to_grid(t: torch.Tensor, step: float) -> torch.Tensor:
    return torch.round(t / step) * step


def router_grid_step(shape: LayerShape) -> float:
    """Grid of the router weights/bias in the exact variant: 2^-8 for fp32 layers, 2^-10
    for bf16 layers (hidden states always sit on 2^-8)."""
    return 2.0 ** -8 if shape.dtype == "fp32" else 2.0 ** -10


def layer_inputs(shape: LayerShape, seed: int = 0, variant: str = "perf",
                 device="cpu", with_experts: bool = True) -> dict:
    """Draw every input of one layer call.

    Returns a dict of torch tensors on ``device``:
      x         [N, H]      dtype   hidden states ~ N(0, x_std^2)
      w_router  [E, H]      dtype   router weight, nn.Linear layout, ~ U(+-1/sqrt(H))
      b_router  [E] fp32 or None    router bias (nn.Linear-like U(+-1/sqrt(H)) and/or the
                                    Zipf popularity bias)
      w_gate, w_up [E, I, H] dtype  SwiGLU gate/up projections, ~ N(0, w_std^2)
      w_down    [E, H, I]    dtype  down projection, ~ N(0, w_std^2)
    """
    if variant not in ("perf", "exact"):
        raise ValueError(variant)
    dt = shape.torch_dtype
    N, H, I, E = shape.N, shape.H, shape.I, shape.E
    out = {}

    z = torch.randn(N, H, generator=_gen(seed, _T_X, device), device=device,
                    dtype=torch.float32) * shape.x_std
    if variant == "exact":
        z = _round_to_grid(z, 2.0 ** -8)
    out["x"] = z.to(dt)
    del z

    bound = 1.0 / math.sqrt(H)
    wr = (torch.rand(E, H, generator=_gen(seed, _T_WR, device), device=device,
                     dtype=torch.float64) * 2 - 1) * bound
    step = router_grid_step(shape)
    if variant == "exact":
        wr = _round_to_grid(wr, step)
    out["w_router"] = wr.to(torch.float32).to(dt)

    b = None
    if shape.bias:
        b = (torch.rand(E, generator=_gen(seed, _T_B, device), device=device,
                        dtype=torch.float64) * 2 - 1) * bound
    if shape.zipf_s is not None:
        rank = torch.randperm(E, generator=_gen(seed, _T_ZIPF, "cpu")).to(torch.float64) + 1
        zb = (-shape.zipf_s * torch.log(rank)).to(device)
        b = zb if b is None else b + zb
    if b is not None:
        if variant == "exact":
            b = _round_to_grid(b, step)
        b = b.to(torch.float32)
    out["b_router"] = b

    if with_experts:
        for key in ("w_gate", "w_up", "w_down"):
            rows, cols = (H, I) if key == "w_down" else (I, H)
            w = torch.empty(E, rows, cols, device=device, dtype=dt)
            for e in range(E):   # per expert, to bound the fp32 temporary
                w[e] = expert_weight(shape, key, e, seed, device)
            out[key] = w
    return out


def expert_weight(shape: LayerShape, key: str, e: int, seed: int = 0, device="cpu"):
    """One expert's weight ("w_gate"/"w_up" [I, H] or "w_down" [H, I]) in the storage
    dtype, ~ N(0, w_std^2), from its own generator stream (so it can be drawn alone)."""
    tid = {"w_gate": _T_WG, "w_up": _T_WU, "w_down": _T_WD}[key]
    rows, cols = (shape.H, shape.I) if key == "w_down" else (shape.I, shape.H)
    g = _gen(seed, tid, device, sub=e + 1)
    return (torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32)
            * shape.w_std).to(shape.torch_dtype)


def snippet_inputs():
    """The worked routing example of the Ultralytics glossary page "Expert Parallelism"
    (section "How tokens move between GPUs"): torch's CPU generator seeded with 0 draws
    4096x512 standard-normal hidden states, then a 512->8 nn.Linear router is
    initialised (weight by nn.Linear's default Kaiming-uniform rule, which is
    U(+-1/sqrt(512)), then bias U(+-1/sqrt(512))). Returns fp32 CPU tensors
    (x [4096,512], w [8,512], b [8]). Draws are made on a private generator in the same
    order as that example, so they are the same numbers."""
    g = torch.Generator().manual_seed(0)
    x = torch.randn(4096, 512, generator=g)
    gain = math.sqrt(2.0 / (1 + 5))
    wb = math.sqrt(3.0) * (gain / math.sqrt(512))
    w = torch.empty(8, 512).uniform_(-wb, wb, generator=g)
    bb = 1.0 / math.sqrt(512)
    b = torch.empty(8).uniform_(-bb, bb, generator=g)
    return x, w, b
