"""moe_dispatch_noalloc: the dispatch step for callers that cannot allocate device
memory (no workspace argument; its scratch is a fixed array inside the library).

Checked through the C ABI against moe_dispatch on the same inputs, on two calls in a row
with different sizes, so that whatever the first call leaves in the shared scratch
cannot leak into the second. Dispatch results are integers and copies, so the bar is
bit-exact equality, as for moe_dispatch against the oracle.
"""
import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _dispatch_both(moe, shape, seed):
    from moe_gpu_harness import make_cfg
    inp = workloads.layer_inputs(shape, seed=seed, variant="exact", device="cuda",
                                 with_experts=False)
    cfg = make_cfg(shape)
    N, k, E, P, H = shape.N, shape.top_k, shape.E, shape.ep_size, shape.H
    i32 = dict(dtype=torch.int32, device="cuda")
    idx = torch.empty(N, k, **i32)
    tw = torch.empty(N, k, dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, inp["x"], inp["w_router"], inp["b_router"], idx, tw)

    def outputs():
        return dict(routed=torch.full((E,), -5, **i32), counts=torch.full((E,), -5, **i32),
                    eoff=torch.full((E + 1,), -5, **i32), poff=torch.full((P + 1,), -5, **i32),
                    perm=torch.full((N * k,), -5, **i32), slot=torch.full((N * k,), -5, **i32),
                    send=torch.zeros(N * k, H, dtype=shape.torch_dtype, device="cuda"))

    ref = outputs()
    ws = moe.alloc_workspace(cfg)
    moe.moe_dispatch(cfg, idx, inp["x"], ref["routed"], ref["counts"], ref["eoff"], ref["poff"],
                     ref["perm"], ref["slot"], ref["send"], ws)
    got = outputs()
    moe.moe_dispatch_noalloc(cfg, idx, inp["x"], got["routed"], got["counts"], got["eoff"],
                             got["poff"], got["perm"], got["slot"], got["send"])
    torch.cuda.synchronize()
    return ref, got


def test_noalloc_dispatch_matches_workspace_dispatch_twice():
    import expert_token_dispatch_gemm_b300 as moe
    S = workloads.LayerShape
    first = S("noalloc_a", N=3000, H=256, I=64, E=64, top_k=8, ep_size=8,
              capacity_factor=1.25, zipf_s=1.1)
    second = S("noalloc_b", N=777, H=128, I=64, E=16, top_k=2, ep_size=4)
    for shape, seed in ((first, 1), (second, 2)):
        ref, got = _dispatch_both(moe, shape, seed)
        for key in ref:
            assert torch.equal(ref[key], got[key]), (shape.name, key)
        assert int(got["eoff"][-1]) > 0


def test_noalloc_dispatch_rejects_sizes_beyond_its_scratch():
    import expert_token_dispatch_gemm_b300 as moe
    # ceil(70000 / 64) * 256 = 280064 > 262144: rejected on the host, nothing launched
    cfg = moe.config(70000, 64, 64, 256, 2, 8)
    fake = ctypes.c_void_p(1 << 20)
    st = moe.lib.moe_dispatch_noalloc(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake,
                                      fake, fake, fake, None)
    assert st == moe.binding.MOE_ERR_UNSUPPORTED
    assert "exceeds" in moe.lib.moe_last_error().decode()
    # slot-major priority counts its segments per slot: 7 * ceil(65436 / 448) = 1029
    # segments x 256 experts = 263424 > 262144, rejected, although the token-order count
    # of the same call, ceil(65436 / 64) * 256 = 261888, would fit
    cfg = moe.config(65436, 64, 64, 256, 7, 8, capacity_priority="slot")
    st = moe.lib.moe_dispatch_noalloc(ctypes.byref(cfg), fake, fake, fake, fake, fake, fake,
                                      fake, fake, fake, None)
    assert st == moe.binding.MOE_ERR_UNSUPPORTED
    assert "1029 histogram segments" in moe.lib.moe_last_error().decode()
