"""Failure detection on the GPU without a GPU fault: a GEMM told to skip its
first k-block load waits on a shared-memory stage that nothing fills; the wait
is bounded (~1 s), the kernel latches QURL_ERR_TIMEOUT and exits cleanly, the
host reads the status, and the context stays usable for the next call."""
import time

import pytest
import torch

import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("qt,M,N,K", [
    (q.INT8, 16, 512, 256),
    (q.FP8_E4M3, 16, 512, 256),
    (q.FP8_E4M3, 300, 512, 256),     # prefill: the CTA-pair kernel
    (q.FP8_E4M3, 256, 8192, 4096),   # decode shape that runs on CTA pairs
    (q.INT8, 1536, 8192, 4096),      # INT8 on CTA pairs, widened weights in TMEM
    (q.INT8, 2048, 512, 256),        # INT8 on CTA pairs, both operands widened in the workspace
])
def test_bounded_wait_times_out_and_context_survives(qt, M, N, K):
    X = synth.activations(f"fault/X/{M}/{K}", M, K).cuda()
    W = synth.weights(f"fault/W/{N}/{K}", N, K).cuda()
    Wq, sw, _, _ = q.prepare_weights(W, qt, s=1.5, keep_scaled=False)
    Xq, sx = q.quant_act(X, qt)
    ws = q.workspace(M, N, K, qt)
    if qt == q.INT8 and (M, N, K) == (1536, 8192, 4096):  # keep the CTA-pair kernel with weights in TMEM
        wide = q.plan(M, N, K, qt, torch.cuda.get_device_properties(0).multi_processor_count)["ws_bytes"]
        ws = torch.empty(wide - 1, dtype=torch.uint8, device="cuda")
    ref = q.linear(Xq, sx, Wq, sw, qt, ws)
    q.qurl_check_device_status()
    q.qurl_debug_inject_timeout()
    t0 = time.time()
    q.linear(Xq, sx, Wq, sw, qt, ws)
    with pytest.raises(q.QurlError) as e:
        q.qurl_check_device_status()
    assert e.value.status == 6  # QURL_ERR_TIMEOUT
    assert time.time() - t0 < 30
    q.qurl_check_device_status()  # cleared
    Y = q.linear(Xq, sx, Wq, sw, qt, ws)
    q.qurl_check_device_status()
    assert torch.equal(Y.view(torch.int16), ref.view(torch.int16))
