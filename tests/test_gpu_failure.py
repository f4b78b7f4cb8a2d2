"""Failure detection without a GPU fault.

* A device-side wait that runs out: moe_check_wait_timeout makes one warp wait, with the
  library's bounded mbarrier wait, on a barrier nothing arrives at. The wait gives up
  after its limit, the status word carries MOE_DEV_TIMEOUT, moe_read_device_status
  reports it and clears it, and the context stays usable: a layer call afterwards still
  matches the oracle.
* A CUDA error reaches the caller as MOE_ERR_CUDA: moe_read_device_status synchronises
  its stream, which is illegal while the stream is being captured into a graph; the
  call returns MOE_ERR_CUDA with a reason, nothing runs on the GPU, and the next calls
  succeed (the library clears the reported error, so no later launch check sees it).
"""
import ctypes

import pytest
import torch

import expert_token_dispatch_gemm_b300 as moe
import workloads
from moe_gpu_harness import Layer, assert_close, oracle_layer, tol_for

pytestmark = pytest.mark.gpu

SHAPE = workloads.LayerShape("fail", N=300, H=128, I=64, E=8, top_k=2, ep_size=4)


def _layer_matches_oracle():
    inp = workloads.layer_inputs(SHAPE, seed=71, variant="exact")
    layer = Layer(SHAPE, inp)
    out, _ = layer.forward()
    assert layer.device_status() == 0
    assert_close(out, oracle_layer(SHAPE, inp)["out"], tol_for(SHAPE))


def test_device_wait_times_out_and_the_context_stays_usable():
    cfg = moe.config(SHAPE.N, SHAPE.H, SHAPE.I, SHAPE.E, SHAPE.top_k, SHAPE.ep_size)
    ws = moe.alloc_workspace(cfg)
    assert moe.moe_read_device_status(cfg, ws) == 0
    moe.moe_check_wait_timeout(cfg, ws)
    flags = moe.moe_read_device_status(cfg, ws, reset=True)     # waits for the kernel
    assert flags & moe.MOE_DEV_TIMEOUT
    status = moe.lib.moe_read_device_status(ctypes.byref(cfg), ctypes.c_void_p(ws.data_ptr()),
                                            ws.numel(), ctypes.byref(ctypes.c_int32()), 0,
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 0                                           # cleared by the reset
    _layer_matches_oracle()


def test_cuda_error_is_reported_as_moe_err_cuda():
    from cuda.bindings import runtime as cudart
    cfg = moe.config(SHAPE.N, SHAPE.H, SHAPE.I, SHAPE.E, SHAPE.top_k, SHAPE.ep_size)
    ws = moe.alloc_workspace(cfg)
    torch.cuda.synchronize()
    err, stream = cudart.cudaStreamCreate()
    assert err == cudart.cudaError_t.cudaSuccess
    try:
        # relaxed mode: the capture restricts nothing outside the captured stream
        err, = cudart.cudaStreamBeginCapture(
            stream, cudart.cudaStreamCaptureMode.cudaStreamCaptureModeRelaxed)
        assert err == cudart.cudaError_t.cudaSuccess
        flags = ctypes.c_int32(0)
        st = moe.lib.moe_read_device_status(ctypes.byref(cfg), ctypes.c_void_p(ws.data_ptr()),
                                            ws.numel(), ctypes.byref(flags), 0,
                                            ctypes.c_void_p(int(stream)))
        reason = moe.lib.moe_last_error().decode()
        err, _graph = cudart.cudaStreamEndCapture(stream)   # invalidated: no graph
        assert err != cudart.cudaError_t.cudaSuccess
        err, capturing = cudart.cudaStreamIsCapturing(stream)
        assert err == cudart.cudaError_t.cudaSuccess
        assert capturing == cudart.cudaStreamCaptureStatus.cudaStreamCaptureStatusNone
    finally:
        cudart.cudaStreamDestroy(stream)
    assert st == moe.binding.MOE_ERR_CUDA, reason
    assert reason
    _layer_matches_oracle()
