"""The whole forward enqueues no host synchronisation and allocates nothing, so it can be
captured in a CUDA graph and replayed; the replay must match eager calls bit for bit."""
import pytest
import torch

import workloads
from moe_gpu_harness import Layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_forward_replays_from_a_cuda_graph(dtype):
    shape = workloads.LayerShape("graph", N=700, H=128, I=96, E=8, top_k=2, ep_size=4,
                                 capacity_factor=1.0, dtype=dtype, bias=True)
    inp = workloads.layer_inputs(shape, seed=41, variant="perf")
    layer = Layer(shape, inp)
    eager, _ = layer.forward(with_diag=False)          # also sets the kernels up
    out = torch.empty_like(eager)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    import expert_token_dispatch_gemm_b300 as moe
    with torch.cuda.graph(g, stream=stream):
        moe.moe_layer_forward(layer.cfg, layer.x, layer.w_router, layer.b_router, layer.packed,
                              layer.w_down, out, layer.ws)
    for seed in (41, 42):
        fresh = workloads.layer_inputs(shape, seed=seed, variant="perf")
        layer.x.copy_(fresh["x"].to(layer.x.device))
        g.replay()
        torch.cuda.synchronize()
        ref, _ = layer.forward(with_diag=False)
        assert torch.equal(out, ref)
    assert layer.device_status() == 0
