"""Launch chaining must never let a GEMM read weights that are still being
rewritten.

The decode GEMMs start loading weight tiles before their grid-dependency wait
when the kernel launched just before them is one of the library's quantizers
(or the INT8 widening kernel), which never write weights.  That is only safe if
the kernel two places back has completed by then -- in the per-RL-step flow it
is qurl_prepare_weights re-quantizing the very weights the next linear reads
(Paper-Notes "QuRL", section 方法详解 > 整体框架: the rollout actor is
re-quantized from the current weights every step).  Here re-quantization into
the same Wq / sw buffers is followed, on one stream and with no host
synchronisation, by the fused RMSNorm -> quant -> linear entry and by the plain
linear entry; the outputs must be bit-identical to those of a run with the
weights prepared and synchronised beforehand.  The weights span tens of
thousands of rows, so the preparation kernel runs many waves and its last ones
overlap whatever the stream launches next.
"""
import pytest
import torch

import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu

M, K, N = 64, 3584, 37888  # 7B gate_up at decode size: a prefetching GEMM, 37888 weight rows


def _bits(t):
    return t.view(torch.int16).clone()


@pytest.mark.parametrize("qt", [q.INT8, q.FP8_E4M3])
def test_requantize_then_linear_sees_new_weights(qt):
    assert torch.cuda.is_available()
    q.load()
    X = synth.activations("pdl/X", M, K).cuda()
    gamma = synth.gamma("pdl/g", K).cuda()
    Ws = [synth.weights(f"pdl/W{i}", N, K).cuda() for i in range(2)]
    ws = q.workspace(M, N, K, qt)
    # references: each weight set prepared in its own buffers, synchronised before use
    refs = []
    for W in Ws:
        Wq, sw, gf, _ = q.prepare_weights(W, qt, s=1.0, gamma=gamma, keep_scaled=False)
        torch.cuda.synchronize()
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        Xq = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        q.qurl_rmsnorm_quant_linear(X, gf, 1e-6, Wq, sw, qt, Y, Xq, sx, ws)
        torch.cuda.synchronize()
        Yl = q.linear(Xq, sx, Wq, sw, qt, ws)
        torch.cuda.synchronize()
        refs.append((_bits(Y), _bits(Yl), Xq.clone(), sx.clone()))
    assert not torch.equal(refs[0][0], refs[1][0])
    q.qurl_check_device_status()

    # one set of buffers, re-quantized in place and used at once, alternating the weight sets
    Wq = torch.empty((N, K), dtype=q.code_dtype(qt), device="cuda")
    sw = torch.empty(N, dtype=torch.float32, device="cuda")
    gf = torch.empty(K, dtype=torch.float32, device="cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Yl = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Xq = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    for rep in range(6):
        i = rep % 2
        # fused entry right behind the re-quantization
        q.qurl_prepare_weights(Ws[i], gamma, 1.0, qt, Wq, sw, gf)
        q.qurl_rmsnorm_quant_linear(X, gf, 1e-6, Wq, sw, qt, Y, Xq, sx, ws)
        torch.cuda.synchronize()
        assert torch.equal(_bits(Y), refs[i][0]), f"fused entry, repetition {rep}"
        # plain linear entry right behind the re-quantization of the other set
        j = 1 - i
        q.qurl_prepare_weights(Ws[j], gamma, 1.0, qt, Wq, sw, gf)
        q.qurl_w8a8_linear(refs[j][2], refs[j][3], Wq, sw, qt, Yl, ws)
        torch.cuda.synchronize()
        assert torch.equal(_bits(Yl), refs[j][1]), f"plain linear entry, repetition {rep}"
    q.qurl_check_device_status()
