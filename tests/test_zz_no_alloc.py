"""qurl_w8a8_linear_static_scratch: the linear entry point that allocates
nothing and needs no workspace from its caller (its scratch is a buffer compiled
into the library), for callers that cannot allocate device memory -- e.g. an
engine that has already handed all of HBM to its own pools.

Checked through the C ABI against qurl_w8a8_linear given a workspace, on two
calls in a row (the second reuses the scratch the first left behind): the plan,
and so the summation order, is the same, so INT8 and FP8 outputs are
bit-identical.  After one warm-up call (which loads the library's modules on
the device), further calls leave the device's free memory and torch's reserved
memory unchanged.  This file is collected last, so that a failure here comes
after every other test has run."""
import ctypes

import pytest
import torch

import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu

# two different projections in a row: split K with the fp16 activation codes in
# the scratch (INT8), then another shape over the bytes the first one left there
SHAPES = ((64, 4608, 3584, "qkv64"), (256, 3584, 18944, "down256"))


def _quantized(qt, M, N, K, tag):
    X = synth.activations(f"noalloc/{tag}/X", M, K).cuda()
    W = synth.weights(f"noalloc/{tag}/W", N, K).cuda()
    Wq, sw, _, _ = q.prepare_weights(W, qt, s=1.5, keep_scaled=False)
    Xq, sx = q.quant_act(X, qt)
    return Xq, sx, Wq, sw


def _static_call(L, Xq, sx, Wq, sw, qt, Y):
    M, K = Xq.shape
    N = Wq.shape[0]
    return L.qurl_w8a8_linear_static_scratch(ctypes.c_void_p(Xq.data_ptr()), ctypes.c_void_p(sx.data_ptr()),
                                             ctypes.c_void_p(Wq.data_ptr()), ctypes.c_void_p(sw.data_ptr()), M, N, K,
                                             qt, ctypes.c_void_p(Y.data_ptr()), Y.stride(0),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("qt", [q.INT8, q.FP8_E4M3])
def test_static_scratch_matches_workspace_entry_twice(qt):
    assert torch.cuda.is_available()
    L = q.load()
    for M, N, K, tag in SHAPES:
        Xq, sx, Wq, sw = _quantized(qt, M, N, K, tag)
        ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        q.qurl_w8a8_linear(Xq, sx, Wq, sw, qt, ref, q.workspace(M, N, K, qt))
        Y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
        assert _static_call(L, Xq, sx, Wq, sw, qt, Y) == 0
        torch.cuda.synchronize()
        q.qurl_check_device_status()
        # same plan and summation order as the workspace entry: the same bits
        assert torch.equal(Y.view(torch.int16), ref.view(torch.int16)), (qt, M, N, K)


def test_static_scratch_allocates_nothing():
    L = q.load()
    inputs = {(qt, tag): _quantized(qt, M, N, K, tag) for qt in (q.INT8, q.FP8_E4M3) for M, N, K, tag in SHAPES}
    outs = {key: torch.empty((v[0].shape[0], v[2].shape[0]), dtype=torch.bfloat16, device="cuda")
            for key, v in inputs.items()}

    def calls():
        for key, (Xq, sx, Wq, sw) in inputs.items():
            assert _static_call(L, Xq, sx, Wq, sw, key[0], outs[key]) == 0

    calls()  # warm-up: loads the library's modules (and the scratch) on this device
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(3):
        calls()
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert torch.cuda.memory_reserved() == reserved0


def test_static_scratch_rejects_shapes_beyond_its_size():
    L = q.load()
    M, N, K = 256, 512, 70000  # the fp16 activation codes alone need 35.8 MB > 32 MiB
    assert q.qurl_workspace_size(M, N, K, q.INT8) > 32 * 1024 * 1024
    Xq = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    Wq = torch.zeros((N, K), dtype=torch.int8, device="cuda")
    sx = torch.ones(M, device="cuda")
    sw = torch.ones(N, device="cuda")
    Y = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
    assert _static_call(L, Xq, sx, Wq, sw, q.INT8, Y) == 4  # QURL_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(Y == 5.0)  # nothing was launched
