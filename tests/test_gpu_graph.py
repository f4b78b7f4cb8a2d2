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


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_training_step_replays_from_a_cuda_graph(dtype):
    """Training forward + backward captured once, replayed on new inputs and upstream
    gradients: the same bits as eager calls."""
    import expert_token_dispatch_gemm_b300 as moe
    shape = workloads.LayerShape("graph_train", N=600, H=128, I=96, E=8, top_k=2, ep_size=4,
                                 capacity_factor=1.0, dtype=dtype, bias=True)
    inp = workloads.layer_inputs(shape, seed=43, variant="perf")
    layer = Layer(shape, inp)
    layer.cfg.training = 1
    layer.ws = moe.alloc_workspace(layer.cfg)
    dev = layer.x.device
    dout = torch.randn(shape.N, shape.H, device=dev).to(shape.torch_dtype)
    out = torch.empty(shape.N, shape.H, dtype=shape.torch_dtype, device=dev)

    def grads():
        return dict(dx=torch.empty_like(layer.x),
                    dw_router=torch.empty(shape.E, shape.H, device=dev),
                    db_router=torch.empty(shape.E, device=dev),
                    dw_gate=torch.empty_like(layer.w_gate), dw_up=torch.empty_like(layer.w_up),
                    dw_down=torch.empty_like(layer.w_down))

    def step(o, g):
        moe.moe_layer_forward(layer.cfg, layer.x, layer.w_router, layer.b_router, layer.packed,
                              layer.w_down, o, layer.ws)
        moe.moe_layer_backward(layer.cfg, layer.x, layer.w_router, layer.packed, layer.w_down,
                               dout, g["dx"], g["dw_router"], g["db_router"], g["dw_gate"],
                               g["dw_up"], g["dw_down"], layer.ws)

    step(out, grads())                     # sets the kernels up outside the capture
    torch.cuda.synchronize()
    gg = grads()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(out, gg)
    for seed in (43, 44):
        fresh = workloads.layer_inputs(shape, seed=seed, variant="perf")
        layer.x.copy_(fresh["x"].to(dev))
        dout.normal_()
        graph.replay()
        torch.cuda.synchronize()
        ref_out, ref = torch.empty_like(out), grads()
        step(ref_out, ref)
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out)
        for key in ref:
            assert torch.equal(gg[key], ref[key]), key
    assert layer.device_status() == 0
