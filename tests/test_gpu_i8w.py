"""INT8 prefill on CTA pairs with both operands widened to fp16 in the workspace
(qurl_debug_plan kernel 4): exact int32 accumulators and bit-exact bf16 outputs
against the CPU oracle in both accumulation modes.

A 256 x 256 x K-split unit is accumulated in one fp32 pass when every token's
sum of |code| is <= 2^17, or when max_t sum x^2 x max_n sum w^2 <= 2^48 (by
Cauchy-Schwarz no partial sum can then leave fp32's exact integer range 2^24),
and in 1024-deep chunks added in int32 otherwise.  The cases below put tiles of
each kind side by side, hit the Cauchy-Schwarz bound exactly, split K, ragged
edges, and more units per CTA pair than the kernel records modes for."""
import os

import numpy as np
import pytest
import torch

import oracle
import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 1


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a.view(np.uint8))).cuda().view(torch.int8)


def sampled(acc, rows, cols):
    return acc[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()


def edge_rows(M, tile=128):
    r = [x for t0 in range(0, M, tile) for x in (t0, t0 + 63, t0 + 64, t0 + tile - 1) if x < M] + [M - 1]
    return np.unique(np.array(r))


@pytest.mark.parametrize("M,N,K", [(2100, 1000, 4000), (2304, 768, 5120)])
def test_wide_modes_side_by_side(M, N, K):
    """Token tiles cycle through small codes (one pass by the sum of |code|),
    +-80 codes (sum |code| > 2^17: one pass by Cauchy-Schwarz against Gaussian-
    sized weight codes) and full-range codes; channel tiles alternate Gaussian-
    sized weight codes and full-range ones, so full-range tokens meet full-range
    weights in chunked units.  Ragged M, N and K (4000 is 62.5 k-blocks of 64)."""
    assert q.plan(M, N, K, q.INT8, sms())["kernel"] == 4
    g = np.random.Generator(np.random.PCG64(M + N + K))
    xq = np.empty((M, K), np.int8)
    for t in range(0, M, 256):
        lim = (10, 80, 127)[(t // 256) % 3]
        xq[t:t + 256] = g.integers(-lim, lim + 1, size=(min(256, M - t), K))
    wq = np.clip(np.rint(g.standard_normal((N, K)) * 28), -127, 127).astype(np.int8)
    for c in range(256, N, 512):
        wq[c:c + 256] = g.integers(-127, 128, size=(min(256, N - c), K))
    x16 = xq.astype(np.int64)
    w16 = wq.astype(np.int64)
    # the three kinds of unit are all present
    S = np.abs(x16).sum(1)
    Q = (x16 * x16).sum(1)
    Qn = (w16 * w16).sum(1)
    assert S[:256].max() <= 2 ** 17                                                   # one pass by S
    assert S[256:512].min() > 2 ** 17 and Q[256:512].max() * Qn[:256].max() <= 2 ** 48  # by Cauchy-Schwarz
    assert S[512:768].min() > 2 ** 17 and Q[512:768].min() * Qn[256:512].min() > 2 ** 48  # chunks
    ws = q.workspace(M, N, K, q.INT8)
    acc = q.gemm_acc(dev(xq), dev(wq), q.INT8, ws)
    sx = torch.rand(M, device="cuda") * 1e-2 + 1e-3
    sw = torch.rand(N, device="cuda") * 1e-2 + 1e-3
    Y = q.linear(dev(xq), sx, dev(wq), sw, q.INT8, ws)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    rows = edge_rows(M)
    cols = np.unique(np.concatenate([np.sort(g.choice(N, size=96, replace=False)), [0, 127, 128, 255, 256, N - 1]]))
    ref = oracle.gemm_i8(xq[rows].view(np.uint8), wq[cols].view(np.uint8), nthreads=NT)
    np.testing.assert_array_equal(sampled(acc, rows, cols), ref)
    Yo = oracle.epilogue(ref, sx.cpu().numpy()[rows], sw.cpu().numpy()[cols])
    np.testing.assert_array_equal(synth.bf16_bits(Y.cpu())[np.ix_(rows, cols)], Yo)


@pytest.mark.parametrize("n127,fast", [(1040, True), (1056, False)])
def test_wide_cauchy_schwarz_bound_is_tight(n127, fast):
    """x, w = +-127 over the first n127 codes, +-1 over the next four and 0 over
    the last twelve (K = n127 + 16).  n127 = 1040: sum x^2 x sum w^2 =
    (127^2 x 1040 + 4)^2 = 2.8137e14 <= 2^48 = 2.8147e14 (while sum |x| =
    132,084 > 2^17), one fp32 pass, and the sums reach 127^2 x 1040 =
    16,774,160, 3056 below 2^24, before +-1 terms that survive only if no low
    bit is dropped.  n127 = 1056 is over the bound (chunks).  Both exact."""
    M, N, K = 2048, 256, n127 + 16
    xq = np.zeros((M, K), np.int8)
    wq = np.zeros((N, K), np.int8)
    xq[:, :n127] = 127
    wq[:, :n127] = 127
    g = np.random.Generator(np.random.PCG64(n127))
    xq[:, n127:n127 + 4] = g.choice(np.array([-1, 1], np.int8), size=(M, 4))
    wq[:, n127:n127 + 4] = g.choice(np.array([-1, 1], np.int8), size=(N, 4))
    xq[1::2, :n127] = -127
    q2 = float((xq[0].astype(np.int64) ** 2).sum()) * float((wq[0].astype(np.int64) ** 2).sum())
    assert (q2 <= 2 ** 48) == fast and int(np.abs(xq[0].astype(np.int64)).sum()) > 2 ** 17
    acc = q.gemm_acc(dev(xq), dev(wq), q.INT8, q.workspace(M, N, K, q.INT8))
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    rows = np.array([0, 1, 2, 255, 256, 1023, M - 1])
    ref = oracle.gemm_i8(xq[rows].view(np.uint8), wq.view(np.uint8), nthreads=NT)
    assert np.abs(ref).max() >= 16_774_000
    np.testing.assert_array_equal(acc.cpu().numpy()[rows], ref)


def test_wide_split_k_chunks():
    """Few tiles (8 x 1), so K = 16384 is split eight ways (2048 k each): full-
    range codes make every split two 1024-deep chunks whose int32 running sum
    lives in the scratch, written as a partial and summed by the reduction."""
    M, N, K = 2048, 256, 16384
    p = q.plan(M, N, K, q.INT8, sms())
    assert p["kernel"] == 4 and p["splits"] > 1
    g = np.random.Generator(np.random.PCG64(3))
    xq = g.integers(-127, 128, size=(M, K)).astype(np.int8)
    wq = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    ws = q.workspace(M, N, K, q.INT8)
    acc = q.gemm_acc(dev(xq), dev(wq), q.INT8, ws)
    sx = torch.rand(M, device="cuda") * 1e-3 + 1e-4
    sw = torch.rand(N, device="cuda") * 1e-3 + 1e-4
    Y = q.linear(dev(xq), sx, dev(wq), sw, q.INT8, ws)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    rows = edge_rows(M, 256)
    ref = oracle.gemm_i8(xq[rows].view(np.uint8), wq.view(np.uint8), nthreads=NT)
    np.testing.assert_array_equal(acc.cpu().numpy()[rows], ref)
    Yo = oracle.epilogue(ref, sx.cpu().numpy()[rows], sw.cpu().numpy())
    np.testing.assert_array_equal(synth.bf16_bits(Y.cpu())[rows], Yo)


def test_wide_prefill_repeatable_on_normed_activations():
    """The 32B-class gate_up shape at M = 2048 with RMSNorm-quantized Gaussian
    activations (sum |code| ~ 1.6e5 > 2^17: one pass only by Cauchy-Schwarz):
    three runs agree bit for bit and a sample matches the oracle."""
    M, (K, N) = 2048, synth.SHAPES_32B["gate_up"]
    X = synth.activations("gpu/i8w/X", M, K, n_out=0).cuda()
    W = synth.weights("gpu/i8w/W", N, K).cuda()
    Wq, _, _, _ = q.prepare_weights(W, q.INT8, s=1.5, keep_scaled=False)
    del W
    Xq, _ = q.rmsnorm_quant(X, torch.ones(K, device="cuda"), q.INT8)
    assert int(Xq.to(torch.int64).abs().sum(1).max()) > 2 ** 17
    ws = q.workspace(M, N, K, q.INT8)
    runs = [q.gemm_acc(Xq, Wq, q.INT8, ws) for _ in range(3)]
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[0], runs[2])
    g = np.random.Generator(np.random.PCG64(29))
    rows = np.sort(g.choice(M, size=48, replace=False))
    cols = np.sort(g.choice(N, size=192, replace=False))
    xc = Xq.cpu().view(torch.uint8).numpy()
    wc = Wq.cpu().view(torch.uint8).numpy()
    ref = oracle.gemm_i8(xc[rows], wc[cols], nthreads=NT)
    np.testing.assert_array_equal(sampled(runs[0], rows, cols), ref)


def test_wide_more_units_than_mode_slots():
    """200 x 200 tiles of 256 x 256: ~526 units per CTA pair, beyond the 512
    whose accumulation mode the kernel records, so the last units take the
    chunked path (K = 2048: two chunks) without a recorded mode; small codes
    everywhere, so the recorded units take one pass.  bf16 outputs (5 GB)
    sampled from the last tiles."""
    M = N = 256 * 200
    K = 2048
    g = np.random.Generator(np.random.PCG64(31))
    xq = g.integers(-20, 21, size=(M, K)).astype(np.int8)
    wq = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    sx = torch.full((M,), 2.0 ** -10, device="cuda")
    sw = torch.full((N,), 2.0 ** -8, device="cuda")
    Y = q.linear(dev(xq), sx, dev(wq), sw, q.INT8, q.workspace(M, N, K, q.INT8))
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    rows = np.unique(np.concatenate([np.sort(g.choice(M, size=32, replace=False)), [M - 256, M - 1]]))
    cols = np.unique(np.concatenate([np.sort(g.choice(N, size=64, replace=False)), [N - 256, N - 1]]))
    got = synth.bf16_bits(Y[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu())
    del Y
    ref = oracle.gemm_i8(xq[rows].view(np.uint8), wq[cols].view(np.uint8), nthreads=NT)
    Yo = oracle.epilogue(ref, np.full(len(rows), 2.0 ** -10, np.float32), np.full(len(cols), 2.0 ** -8, np.float32))
    np.testing.assert_array_equal(got, Yo)


def test_attached_wide_weights_bit_identical_and_refreshed():
    """A call with the caller's persistent fp16 copy of the weights attached
    (qurl_widen_weights) launches one kernel fewer than one that widens Wq into
    its workspace and gives the same bits; re-quantizing the attached Wq in
    place through qurl_prepare_weights refreshes the copy; after detaching,
    calls widen again."""
    M, N, K = 2048, 1024, 2048
    X = synth.activations("gpu/i8w/att/X", M, K).cuda()
    W = synth.weights("gpu/i8w/att/W", N, K).cuda()
    Wq, sw, _, Wm = q.prepare_weights(W, q.INT8, s=1.5)
    Xq, sx = q.quant_act(X, q.INT8)
    ws = q.workspace(M, N, K, q.INT8)
    assert q.plan(M, N, K, q.INT8, sms())["kernel"] == 4

    def run():
        n0 = q.qurl_kernel_launches()
        Y = q.linear(Xq, sx, Wq, sw, q.INT8, ws)
        torch.cuda.synchronize()
        q.qurl_check_device_status()
        return Y, q.qurl_kernel_launches() - n0

    Y0, n_plain = run()
    wide = q.wide_weights(Wq)
    Y1, n_att = run()
    assert n_att == n_plain - 1 and torch.equal(Y0.view(torch.int16), Y1.view(torch.int16))
    # the per-step re-quantization of an updated master, into the same Wq buffer
    W2 = Wm + torch.randn_like(Wm) * 1e-3
    q.qurl_prepare_weights(W2, None, 1.0, q.INT8, Wq, sw)
    Y2, _ = run()
    q.qurl_detach_wide_weights(Wq)
    Y3, n_det = run()
    assert n_det == n_plain
    assert torch.equal(Y2.view(torch.int16), Y3.view(torch.int16))
    assert not torch.equal(Y2.view(torch.int16), Y0.view(torch.int16))
    del wide


@pytest.mark.parametrize("M,N,K", [(300, 4608, 3584), (264, 3584, 18944), (1024, 7168, 5120), (1024, 5120, 27648),
                                   (1024, 5120, 5120), (256, 4608, 3584), (256, 5120, 27648), (200, 55296, 5120)])
def test_attached_weights_take_the_pair_kernel_above_256_tokens(M, N, K):
    """With an attached fp16 copy of the weights, INT8 batches above 256 tokens
    run on the CTA-pair kernel (ragged M; K split at 264 x 3584 x 18944; at
    1024 x 5120 x 5120 and 1024 x 5120 x 27648 76 of the 80 tiles run whole and
    the last 4 split, reduced by their own kernel -- raw int32 sums through
    qurl_w8a8_gemm_acc too), and so do batches of 129 to 256 tokens on weights
    of 2^26 codes or more (one token tile, partly empty); all give the bits of
    the TMEM-weight kernel that runs without the copy, and of the oracle on a
    sample.  At 256 tokens on smaller weights the TMEM-weight kernel keeps the
    call."""
    big = M > 128 and N * K >= (1 << 26)
    assert q.plan(M, N, K, q.INT8, sms(), attached=True)["kernel"] == (4 if (M > 256 or big) else 1)
    X = synth.activations(f"gpu/i8w/mid/X/{M}", M, K).cuda()
    W = synth.weights(f"gpu/i8w/mid/W/{N}", N, K).cuda()
    Wq, sw, _, _ = q.prepare_weights(W, q.INT8, s=1.5, keep_scaled=False)
    del W
    Xq, sx = q.quant_act(X, q.INT8)
    ws = q.workspace(M, N, K, q.INT8)
    assert q.plan(M, N, K, q.INT8, sms())["kernel"] != 4
    Y0 = q.linear(Xq, sx, Wq, sw, q.INT8, ws)
    wide = q.wide_weights(Wq)
    n0 = q.qurl_kernel_launches()
    Y1 = q.linear(Xq, sx, Wq, sw, q.INT8, ws)
    launched = q.qurl_kernel_launches() - n0
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    assert launched >= 2  # the activations' widening, the pair GEMM (and a reduction where K is split)
    assert torch.equal(Y0.view(torch.int16), Y1.view(torch.int16))
    g = np.random.Generator(np.random.PCG64(M + N))
    rows = np.unique(np.concatenate([g.choice(M, 16, replace=False), [0, M - 1]]))
    cols = np.unique(np.concatenate([g.choice(N, 64, replace=False), [0, N - 1]]))
    xc = Xq.cpu().view(torch.uint8).numpy()
    wc = Wq.cpu().view(torch.uint8).numpy()
    ref = oracle.gemm_i8(xc[rows], wc[cols], nthreads=NT)
    Yo = oracle.epilogue(ref, sx.cpu().numpy()[rows], sw.cpu().numpy()[cols])
    np.testing.assert_array_equal(synth.bf16_bits(Y1.cpu())[np.ix_(rows, cols)], Yo)
    acc = q.gemm_acc(Xq, Wq, q.INT8, ws)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    np.testing.assert_array_equal(sampled(acc, rows, cols), ref)
    del wide
