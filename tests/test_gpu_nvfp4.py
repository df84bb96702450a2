"""The 4-bit (NVFP4, W4A4) variant on the GPU against the CPU oracle.

Quantization (E2M1 codes, E4M3 block scales, fp32 row scales) is bit-exact:
both sides decide every code on the IEEE quotient v / step.  The GEMM
multiplies the exactly widened fp16 values on the tensor cores and sums in
fp32, so its accumulators are held to the worst-case bound of any fp32
summation order, K * 2^-24 * sum_k |x_k w_k| (every product is exact), and its
bf16 outputs to the FP8 path's 1e-2 max-abs-rel (Paper-Notes "QuRL", section
局限与展望: 4-bit quantization; the format is a reading, see the oracle)."""
import os

import numpy as np
import pytest
import torch

import oracle
import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 1


def _np(t):
    return t.cpu().numpy()


def _bits(X):
    return synth.bf16_bits(X.cpu())


def _acc_bound(x, w, rows, cols):
    """K 2^-24 sum_k |x_k w_k| for the sampled outputs (exact dequantized operands)."""
    def deq(q4, sb):
        return oracle.e2m1_decode(oracle.nvfp4_unpack(q4)) * np.repeat(oracle.e4m3_decode(sb), 16, 1)
    xa = np.abs(deq(x[0][rows], x[1][rows]))
    wa = np.abs(deq(w[0][cols], w[1][cols]))
    K = xa.shape[1]
    return K * 2.0 ** -24 * (xa @ wa.T)


@pytest.mark.parametrize("M,K,pre", [(1, 16, 1.0), (33, 256, 1.5), (300, 1040, 1.5), (64, 5120, -0.75)])
def test_quant_act_rows_bit_exact(M, K, pre):
    X = synth.activations(f"nvfp4/act/{M}/{K}", M, K).cuda()
    X[min(2, M - 1), : min(K, 32)] = 0.0           # a zero block (a zero row when K <= 32)
    X[0, 16:32] = X[0, 16:32] * 1e-6 if K >= 32 else X[0, 16:32]  # a block far below the row's max
    q4, sb, g = q.nvfp4_quant(X, pre)
    torch.cuda.synchronize()
    r = oracle.nvfp4_quant_act(_bits(X), pre)
    np.testing.assert_array_equal(_np(q4), r[0])
    np.testing.assert_array_equal(_np(sb), r[1])
    np.testing.assert_array_equal(_np(g), r[2])


@pytest.mark.parametrize("N,K", [(7, 64), (512, 3584), (96, 27648)])
def test_quant_weight_rows_bit_exact(N, K):
    W = synth.weights(f"nvfp4/w/{N}/{K}", N, K).cuda()
    W[1 % N] = 0.0
    q4, sb, g = q.nvfp4_quant(W)
    torch.cuda.synchronize()
    r = oracle.nvfp4_quant_rows(_np(W))
    np.testing.assert_array_equal(_np(q4), r[0])
    np.testing.assert_array_equal(_np(sb), r[1])
    np.testing.assert_array_equal(_np(g), r[2])


def test_quant_golden_rows_and_signed_zero():
    """The hand-derived rows (every E2M1 tie, saturation, -0.1 -> code 8)."""
    import json
    rows = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_worked_examples.json")))["rows"]
    V = torch.tensor([r["v"] for r in rows], dtype=torch.float32, device="cuda")
    q4, sb, g = q.nvfp4_quant(V)
    torch.cuda.synchronize()
    codes = oracle.nvfp4_unpack(_np(q4))
    for i, r in enumerate(rows):
        np.testing.assert_array_equal(codes[i], np.array(r["codes"], np.uint8), err_msg=r["why"])
        np.testing.assert_array_equal(_np(sb)[i], np.array(r["block_scales"], np.uint8))


def _operands(M, N, K, tag):
    X = synth.activations(f"nvfp4/gemm/{tag}/X", M, K).cuda()
    W = synth.weights(f"nvfp4/gemm/{tag}/W", N, K).cuda()
    x = q.nvfp4_quant(X, 1.5)
    w = q.nvfp4_quant(W)
    return x, w


@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (300, 520, 1040), (64, 4608, 3584), (256, 256, 8192),
                                   (1024, 5120, 5120)])
def test_gemm_acc_and_linear(M, N, K):
    """Tiles, ragged M/N, a K tail (1040 = 16.25 k-blocks of 64), K split eight
    ways (one 256 x 256 tile), and 80 tiles on 76 SM pairs: 76 whole, the last
    4 split and reduced by their own kernel."""
    x, w = _operands(M, N, K, f"{M}/{N}/{K}")
    ws = q.nvfp4_workspace(M, N, K)
    acc = q.nvfp4_gemm_acc(x, w, ws)
    Y = q.nvfp4_linear(x, w, ws)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    xc = tuple(_np(t) for t in x)
    wc = tuple(_np(t) for t in w)
    ref = oracle.gemm_nvfp4(xc[0], xc[1], wc[0], wc[1], nthreads=NT)
    bound = _acc_bound(xc, wc, np.arange(M), np.arange(N))
    err = np.abs(_np(acc).astype(np.float64) - ref)
    assert np.all(err <= bound), float((err / np.maximum(bound, 1e-300)).max())
    Yo = oracle.bf16_decode(oracle.epilogue(ref, xc[2], wc[2]))
    Yg = _np(Y.float())
    assert np.max(np.abs(Yg - Yo)) <= 1e-2 * np.max(np.abs(Yo))


def test_linear_full_size_sampled():
    """The 32B-class gate_up at M = 2048: sampled outputs against the oracle."""
    M, (K, N) = 2048, synth.SHAPES_32B["gate_up"]
    x, w = _operands(M, N, K, "32b")
    ws = q.nvfp4_workspace(M, N, K)
    Y = q.nvfp4_linear(x, w, ws)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    g = np.random.Generator(np.random.PCG64(11))
    rows = np.unique(np.concatenate([g.choice(M, 24, replace=False), [0, 255, 256, M - 1]]))
    cols = np.unique(np.concatenate([g.choice(N, 160, replace=False), [0, 255, 256, N - 1]]))
    xc = tuple(_np(t) for t in x)
    wc = tuple(_np(t) for t in w)
    ref = oracle.gemm_nvfp4(xc[0][rows], xc[1][rows], wc[0][cols], wc[1][cols], nthreads=NT)
    Yo = oracle.bf16_decode(oracle.epilogue(ref, xc[2][rows], wc[2][cols]))
    Yg = _np(Y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].float())
    assert np.max(np.abs(Yg - Yo)) <= 1e-2 * np.max(np.abs(Yo))


def test_workspace_too_small_and_k_tail_rejected():
    x, w = _operands(64, 256, 512, "ws")
    ws = q.nvfp4_workspace(64, 256, 512)
    Y = torch.empty((64, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(q.QurlError) as e:
        q.qurl_nvfp4_linear(x, w, Y, ws[:-1])
    assert q.STATUS[e.value.status] == "QURL_ERR_WORKSPACE"
    lib = q.load()
    rc = lib.qurl_nvfp4_linear(q._ptr(x[0]), q._ptr(x[1]), q._ptr(x[2]), q._ptr(w[0]), q._ptr(w[1]), q._ptr(w[2]),
                               64, 256, 504, q._ptr(Y), 256, q._ptr(ws), ws.numel(), None)
    assert q.STATUS[rc] == "QURL_ERR_UNSUPPORTED"  # K not a multiple of 16


def test_attached_weight_copy_gives_identical_results_and_refreshes():
    """With the weights' fp16 copy attached (qurl_nvfp4_widen_weights) the
    linear launches one kernel fewer and gives the same bits; re-quantizing
    attached rows in place refreshes the copy; detached, calls widen again."""
    M, N, K = 512, 1024, 2048
    x, w = _operands(M, N, K, "attach")
    ws = q.nvfp4_workspace(M, N, K)

    def run():
        n0 = q.qurl_kernel_launches()
        Y = q.nvfp4_linear(x, w, ws)
        torch.cuda.synchronize()
        q.qurl_check_device_status()
        return Y.view(torch.int16).clone(), q.qurl_kernel_launches() - n0

    Y0, n0 = run()
    wide = q.nvfp4_wide_weights(w)
    Y1, n1 = run()
    assert n1 == n0 - 1 and torch.equal(Y0, Y1)
    W2 = synth.weights("nvfp4/gemm/attach/W2", N, K).cuda()
    q.qurl_nvfp4_quant(W2, 1.0, *w)  # new codes into the attached rows
    Y2, _ = run()
    q.qurl_detach_wide_weights(w[0])
    Y3, n3 = run()
    assert n3 == n0 and torch.equal(Y2, Y3) and not torch.equal(Y2, Y0)
    del wide
