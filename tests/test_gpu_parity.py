"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Bit-exact: quantized codes and scales (activation, weight, RMSNorm and SiLU
quantizers), INT8 int32 accumulators and INT8 bf16 outputs, flip counts.
FP8: fp32 accumulators within an accumulation-error bound, bf16 outputs within
max-abs-rel 1e-2 (the accumulation order differs from the exact fp64 oracle).

Sizes: small cases the oracle runs in seconds that still span several tiles,
K-splits and ragged tails; the full projection shapes of the 7B- and 32B-class
models in the launch configuration the benchmark uses, checked on a seeded
sample of output rows / channels.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 1
QTS = [q.INT8, q.FP8_E4M3]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    q.load()
    yield
    q.qurl_check_device_status()


def oqt(qt):
    return oracle.INT8 if qt == q.INT8 else oracle.FP8_E4M3


def codes(t):
    return t.contiguous().cpu().view(torch.uint8).numpy()


def f32(t):
    return t.cpu().numpy()


def bits(t):
    return synth.bf16_bits(t.cpu())


def max_abs_rel(y, ref):
    y = y.astype(np.float64)
    ref = ref.astype(np.float64)
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-30))


def sync_ok():
    torch.cuda.synchronize()
    q.qurl_check_device_status()


# ------------------------------------------------------------------ quantizers

ACT_SHAPES = [(16, 256), (1, 16), (17, 3584), (129, 5120), (3, 18944), (64, 27648), (2, 70000)]


@pytest.mark.parametrize("qt", QTS)
@pytest.mark.parametrize("M,K", ACT_SHAPES)
def test_quant_act_exact(qt, M, K):
    X = synth.activations(f"gpu/act/{M}/{K}", M, K)
    X[0, : K // 2] = 0  # a half-zero row
    if M > 2:
        X[2] = 0  # an all-zero row: scale 1, codes 0
    for pre in (1.0, 1.5):
        Xq, sx = q.quant_act(X.cuda(), qt, pre_scale=pre)
        sync_ok()
        qo, so = oracle.quant_act(bits(X), oqt(qt), pre_scale=pre)
        np.testing.assert_array_equal(codes(Xq), qo)
        np.testing.assert_array_equal(f32(sx), so)


def test_quant_act_fp8_midpoint_quotients():
    """FP8 codes round v / scale to the nearest e4m3 value, ties to even, with
    saturation.  With absmax 448 (scale exactly 1) or 672 at pre-scale 1.5
    (scale exactly 1.5) the quotients are every e4m3 rounding midpoint -- normal
    ones from 2^-6 to 448 and the subnormal ones below 2^-6 -- and one bf16 ulp
    either side of them: the kernel's reciprocal shortcut, which lands within a
    few fp32 ulps of the quotient, must hand each such code to the exact
    division."""
    mids = [(1 + (2 * k + 1) / 16) * 2.0 ** e for e in range(-6, 9) for k in range(8)]
    mids = [m for m in mids if m < 448] + [(j + 0.5) * 2.0 ** -9 for j in range(8)]
    b = torch.tensor(mids, dtype=torch.float32).to(torch.bfloat16)
    assert torch.equal(b.float(), torch.tensor(mids))  # every midpoint is a bf16 value
    up = (b.view(torch.int16) + 1).view(torch.bfloat16).float()
    dn = (b.view(torch.int16) - 1).view(torch.bfloat16).float()
    vals = torch.cat([b.float(), up, dn])
    row = torch.cat([torch.tensor([448.0]), vals, -vals])
    K = ((row.numel() + 15) // 16) * 16
    X = torch.zeros((1, K), dtype=torch.float32)
    X[0, : row.numel()] = row
    X = X.to(torch.bfloat16)
    for pre in (1.0, 1.5):
        Xq, sx = q.quant_act(X.cuda(), q.FP8_E4M3, pre_scale=pre)
        sync_ok()
        qo, so = oracle.quant_act(bits(X), oracle.FP8_E4M3, pre_scale=pre)
        np.testing.assert_array_equal(codes(Xq), qo)
        np.testing.assert_array_equal(f32(sx), so)
    assert mids[48] == 1.0625 and codes(Xq)[0, 1 + 48] == 0x38  # 1.0625 (between 1 and 1.125) -> 1.0 (even)


@pytest.mark.parametrize("qt", QTS)
@pytest.mark.parametrize("M,K,ldx", [(3000, 5120, 7168), (4100, 3584, 3584)])
def test_quantizers_on_streamed_rows(qt, M, K, ldx):
    """Prefill-sized batches (thousands of rows, several waves of row CTAs):
    per-token quant (rows strided as the q slice of a qkv output) and RMSNorm
    -> quant stay exact against the oracle, and the fp16 codes and code sums
    they leave for the INT8 GEMM give the bits of the separate quantizer +
    linear calls."""
    big = synth.activations(f"gpu/stream/{M}/{K}", M, ldx)
    X = big[:, :K].contiguous()
    g = synth.gamma(f"gpu/stream/g/{K}", K) * 1.5
    Xq, sx = q.quant_act(big.cuda()[:, :K], qt, pre_scale=1.5)
    Xr, sr, ms = q.rmsnorm_quant(X.cuda(), g.cuda(), qt, eps=1e-6, want_ms=True)
    sync_ok()
    qo, so = oracle.quant_act(bits(X), oqt(qt), pre_scale=1.5)
    np.testing.assert_array_equal(codes(Xq), qo)
    np.testing.assert_array_equal(f32(sx), so)
    ms_d = f32(ms)
    np.testing.assert_allclose(ms_d, oracle.rms_ms(bits(X)), rtol=2e-7)
    qo, so, _, _ = oracle.rmsnorm_quant(bits(X), g.numpy(), oqt(qt), eps=1e-6, ms_given=ms_d)
    np.testing.assert_array_equal(codes(Xr), qo)
    np.testing.assert_array_equal(f32(sr), so)
    N = 256
    Wq, sw, gf, _ = q.prepare_weights(synth.weights(f"gpu/stream/W/{K}", N, K).cuda(), qt, s=1.5,
                                      gamma=synth.gamma(f"gpu/stream/g/{K}", K).cuda())
    cd = q.code_dtype(qt)
    Y1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Y2 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    xs = torch.empty((M, K), dtype=cd, device="cuda")
    ss = torch.empty(M, dtype=torch.float32, device="cuda")
    q.qurl_quant_act_linear(big.cuda()[:, :K], 1.5, Wq, sw, qt, Y1, xs, ss, q.workspace(M, N, K, qt))
    R1 = q.linear(Xq, sx, Wq, sw, qt, q.workspace(M, N, K, qt))
    q.qurl_rmsnorm_quant_linear(X.cuda(), gf, 1e-6, Wq, sw, qt, Y2, xs, ss, q.workspace(M, N, K, qt))
    X2, s2 = q.rmsnorm_quant(X.cuda(), gf, qt, eps=1e-6)
    R2 = q.linear(X2, s2, Wq, sw, qt, q.workspace(M, N, K, qt))
    sync_ok()
    assert torch.equal(Y1.view(torch.int16), R1.view(torch.int16))
    assert torch.equal(Y2.view(torch.int16), R2.view(torch.int16))


@pytest.mark.parametrize("qt", QTS)
def test_quant_act_strided_rows(qt):
    """The o_proj input is a column slice of the qkv output (row stride 4608)."""
    big = synth.activations("gpu/act/strided", 37, 4608)
    X = big[:, :3584]
    Xq, sx = q.quant_act(big.cuda()[:, :3584], qt, pre_scale=1.5)
    sync_ok()
    qo, so = oracle.quant_act(bits(X.contiguous()), oqt(qt), pre_scale=1.5)
    np.testing.assert_array_equal(codes(Xq), qo)
    np.testing.assert_array_equal(f32(sx), so)


def test_quant_act_int8_half_integer_quotients():
    """INT8 codes round v / scale to the nearest integer, ties to even.  With
    absmax 127 (scale exactly 1) or 190.5 at pre-scale 1.5 (scale exactly 1.5)
    the quotients land exactly on half-integers, and one bf16 ulp either side of
    them: the kernel's reciprocal shortcut must hand every such code to the
    exact division."""
    K = 256
    row = np.zeros(K, np.float32)
    row[0] = 127.0
    halves = np.array([0.5, 1.5, 2.5, 3.5, 4.5, 10.5, 63.5, 64.5, 100.5, 126.5], np.float32)
    row[1:11] = halves
    row[11:21] = -halves
    b = torch.from_numpy(halves).to(torch.bfloat16)
    up = (b.view(torch.int16) + 1).view(torch.bfloat16).float().numpy()  # next bf16 above
    dn = (b.view(torch.int16) - 1).view(torch.bfloat16).float().numpy()  # next bf16 below
    row[21:31], row[31:41], row[41:51] = up, dn, -up
    g = np.random.Generator(np.random.PCG64(3))
    row[51:] = np.round(g.uniform(-126, 126, K - 51) * 2) / 2  # more halves and integers
    X = torch.from_numpy(np.stack([row, row * np.float32(0.75)])).to(torch.bfloat16)
    for pre in (1.0, 1.5):
        Xq, sx = q.quant_act(X.cuda(), q.INT8, pre_scale=pre)
        sync_ok()
        qo, so = oracle.quant_act(bits(X), oracle.INT8, pre_scale=pre)
        np.testing.assert_array_equal(codes(Xq), qo)
        np.testing.assert_array_equal(f32(sx), so)
    c = codes(Xq)[0].view(np.int8)
    assert list(c[1:6]) == [0, 2, 2, 4, 4]  # 0.5 -> 0, 1.5 -> 2, 2.5 -> 2, 3.5 -> 4, 4.5 -> 4 (ties to even)


@pytest.mark.parametrize("qt", QTS)
@pytest.mark.parametrize("M,K", [(16, 256), (33, 3584), (7, 5120), (4, 70000)])
def test_rmsnorm_quant(qt, M, K):
    X = synth.activations(f"gpu/rms/{M}/{K}", M, K)
    g = synth.gamma(f"gpu/rms/g/{K}", K) * 1.5
    Xq, sx, ms = q.rmsnorm_quant(X.cuda(), g.cuda(), qt, eps=1e-6, want_ms=True)
    sync_ok()
    ms_d = f32(ms)
    ms_o = oracle.rms_ms(bits(X))
    np.testing.assert_allclose(ms_d, ms_o, rtol=2e-7)
    # codes and scales are exact given the kernel's mean of squares
    qo, so, _, _ = oracle.rmsnorm_quant(bits(X), g.numpy(), oqt(qt), eps=1e-6, ms_given=ms_d)
    np.testing.assert_array_equal(codes(Xq), qo)
    np.testing.assert_array_equal(f32(sx), so)
    # the kernel's compensated mean of squares is the oracle's own fp32 value in (nearly) every
    # row; those rows are exact with no input from the kernel
    q2, s2, ms2, _ = oracle.rmsnorm_quant(bits(X), g.numpy(), oqt(qt), eps=1e-6)
    same = ms2 == ms_d
    assert same.mean() >= 0.9, same.mean()
    np.testing.assert_array_equal(codes(Xq)[same], q2[same])
    np.testing.assert_array_equal(f32(sx)[same], s2[same])


@pytest.mark.parametrize("qt", QTS)
@pytest.mark.parametrize("M,I", [(16, 256), (9, 18944), (3, 4096),
                                 # more rows than SMs, rows longer than 16384: the persistent kernel
                                 # that streams each row into shared memory (one row on most CTAs; six
                                 # or seven, both row buffers reused; the widest row it takes)
                                 (153, 16400), (1000, 18944), (300, 27648)])
def test_silu_mul_quant(qt, M, I):
    GU = synth.activations(f"gpu/silu/{M}/{I}", M, 2 * I, outlier_gain=4.0)
    GU[0, :4] = torch.tensor([0.0, -90.0, 60.0, -3.0])
    Xq, sx, h = q.silu_mul_quant(GU.cuda(), qt, pre_scale=1.5, want_h=True)
    sync_ok()
    _, _, ho = oracle.silu_mul_quant(bits(GU), oqt(qt), pre_scale=1.5)
    hd = f32(h)
    np.testing.assert_allclose(hd, ho, rtol=2e-6, atol=1e-35)
    qo, so, _ = oracle.silu_mul_quant(bits(GU), oqt(qt), pre_scale=1.5, h_given=hd)
    np.testing.assert_array_equal(codes(Xq), qo)
    np.testing.assert_array_equal(f32(sx), so)


@pytest.mark.parametrize("qt", QTS)
@pytest.mark.parametrize("wtype", ["fp32", "bf16"])
@pytest.mark.parametrize("N,K", [(512, 256), (136, 3584), (3, 27648), (5, 70000)])
def test_prepare_weights_exact(qt, wtype, N, K):
    W = synth.weights(f"gpu/w/{N}/{K}", N, K)
    W[1, :] = 0  # an all-zero output channel
    g = synth.gamma(f"gpu/w/g/{K}", K)
    Wi = W if wtype == "fp32" else W.to(torch.bfloat16)
    for s in (1.5, 1.0):
        Wq, sw, gf, Ws = q.prepare_weights(Wi.cuda(), qt, s=s, gamma=g.cuda())
        sync_ok()
        Wo, swo, gfo, Wso = oracle.prepare_weights(Wi.float().numpy(), oqt(qt), s=s, gamma=g.numpy())
        np.testing.assert_array_equal(codes(Wq), Wo)
        np.testing.assert_array_equal(f32(sw), swo)
        np.testing.assert_array_equal(f32(gf), gfo)
        np.testing.assert_array_equal(f32(Ws), Wso)


@pytest.mark.parametrize("qt", QTS)
def test_prepare_weights_in_place_master(qt):
    """W' may overwrite the fp32 master in place (the per-step re-quantization
    writes nothing new, but the set-up fold replaces W by W/s)."""
    W = synth.weights("gpu/w/inplace", 64, 3584)
    Wd = W.cuda()
    Wq = torch.empty((64, 3584), dtype=q.code_dtype(qt), device="cuda")
    sw = torch.empty(64, dtype=torch.float32, device="cuda")
    q.qurl_prepare_weights(Wd, None, 1.5, qt, Wq, sw, None, Wd)
    sync_ok()
    Wo, swo, _, Wso = oracle.prepare_weights(W.numpy(), oqt(qt), s=1.5)
    np.testing.assert_array_equal(codes(Wq), Wo)
    np.testing.assert_array_equal(f32(Wd), Wso)


# ------------------------------------------------------------------ GEMM

GEMM_SHAPES = [
    (16, 512, 256),     # the tiny layer
    (1, 136, 16),       # a single token, one k-block, ragged channel tile
    (17, 520, 4096),    # ragged tokens and channels, several INT8 chunks
    (64, 4608, 3584),   # 7B qkv decode: split-K
    (200, 1000, 1024),  # swap with two INT8 token tiles, ragged
    (300, 520, 2048),   # prefill orientation, ragged
    (129, 384, 1040),   # K not a multiple of the k-block (zero-filled tail)
    (512, 768, 3072),   # prefill, several tiles each way
]


def random_codes(qt, shape, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    if qt == q.INT8:
        return g.integers(-127, 128, size=shape).astype(np.int8).view(np.uint8)
    # codes of Gaussian values: the magnitudes a quantized layer sees
    v = g.standard_normal(shape).astype(np.float32) * np.float32(100.0)
    return oracle.e4m3_encode(np.clip(v, -448, 448))


def to_dev(codes_u8, qt):
    t = torch.from_numpy(np.ascontiguousarray(codes_u8)).cuda()
    return t.view(q.code_dtype(qt))


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("with_ws", [True, False])
def test_gemm_acc_int8_exact(M, N, K, with_ws):
    xq = random_codes(q.INT8, (M, K), M * 7 + K)
    wq = random_codes(q.INT8, (N, K), N * 13 + K)
    ws = q.workspace(M, N, K, q.INT8) if with_ws else None
    acc = q.gemm_acc(to_dev(xq, q.INT8), to_dev(wq, q.INT8), q.INT8, ws)
    sync_ok()
    ref = oracle.gemm_i8(xq, wq, nthreads=NT)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref)


def test_gemm_int8_worst_case_magnitude():
    """|acc| = 127^2 * 27648 = 445,934,592: far beyond fp32's 2^24 exact range,
    exact only through the chunked int32 accumulation."""
    K = 27648
    xq = np.full((3, K), 127, np.int8)
    xq[1] = -127
    xq[2, ::2] = -127
    wq = np.full((256, K), 127, np.int8)
    wq[1::2] = -127
    acc = q.gemm_acc(to_dev(xq.view(np.uint8), q.INT8), to_dev(wq.view(np.uint8), q.INT8), q.INT8,
                     q.workspace(3, 256, K, q.INT8))
    sync_ok()
    a = acc.cpu().numpy()
    assert a[0, 0] == 445_934_592 and a[0, 1] == -445_934_592 and a[1, 0] == -445_934_592
    assert a[2, 0] == 0
    np.testing.assert_array_equal(a, oracle.gemm_i8(xq.view(np.uint8), wq.view(np.uint8), nthreads=NT))


def test_gemm_int8_chunk_edge_exactness():
    """Partial sums of a 1024-deep chunk reach 1023 * 127^2 + 1 = 16,499,968 + 1, one
    below the fp32 integer limit 2^24 in magnitude, with +-1 terms that only survive
    if the tensor core's fp32 accumulation drops no low bit; more chunks follow
    with the opposite sign so the int32 sum also crosses zero."""
    K = 4096
    M, N = 8, 128
    xq = np.full((M, K), 127, np.int8)
    wq = np.full((N, K), 127, np.int8)
    g = np.random.Generator(np.random.PCG64(99))
    for c in range(K // 1024):
        lo, hi = c * 1024, (c + 1) * 1024
        sign = 1 if c % 2 == 0 else -1
        wq[:, lo:hi] *= sign
        # the last entries of each chunk: small +-1 products in varying places
        xq[:, hi - 8:hi] = g.choice(np.array([-1, 1], np.int8), size=(M, 8))
        wq[:, hi - 8:hi] = g.choice(np.array([-1, 1], np.int8), size=(N, 8))
    xq[1] = -xq[1]
    xq[2, ::3] = 0
    acc = q.gemm_acc(to_dev(xq.view(np.uint8), q.INT8), to_dev(wq.view(np.uint8), q.INT8), q.INT8)
    sync_ok()
    ref = oracle.gemm_i8(xq.view(np.uint8), wq.view(np.uint8), nthreads=NT)
    assert np.abs(ref).max() < 2 ** 24 * 2  # per chunk below 2^24; the total is exact in int32 anyway
    np.testing.assert_array_equal(acc.cpu().numpy(), ref)


@pytest.mark.parametrize("extra", [0, 1])
def test_gemm_int8_single_pass_limit(extra):
    """The decode INT8 kernel accumulates a token tile over all of K in one fp32
    pass when every token has sum_k |x| <= 2^24 / 128 = 131072, else in 1024-deep
    chunks.  Here sum |x| = 131042 (one pass) or 131073 (chunks), while the
    partial sums with w = -128 reach -16,773,120 = -(2^24 - 4096) or beyond, and
    +-1 terms follow that only survive if no low bit is dropped."""
    K, M, N = 8192, 16, 256
    xq = np.zeros((M, K), np.int8)
    xq[:, :8190] = 16
    xq[:, 8190:] = 1
    if extra:
        xq[:, :31] = 17  # sum |x| = 131042 + 31 = 131073: one over the single-pass limit
    xq[1] = -xq[1]
    wq = np.full((N, K), -128, np.int8)
    g = np.random.Generator(np.random.PCG64(5))
    wq[:, 8190:] = g.choice(np.array([-1, 0, 1], np.int8), size=(N, 2))
    wq[1::2, :8190] = 127
    assert int(np.abs(xq.astype(np.int64)).sum(1).max()) == (131073 if extra else 131042)
    acc = q.gemm_acc(to_dev(xq.view(np.uint8), q.INT8), to_dev(wq.view(np.uint8), q.INT8), q.INT8,
                     q.workspace(M, N, K, q.INT8))
    sync_ok()
    ref = oracle.gemm_i8(xq.view(np.uint8), wq.view(np.uint8), nthreads=NT)
    assert np.abs(ref).max() >= 16_773_120
    np.testing.assert_array_equal(acc.cpu().numpy(), ref)


@pytest.mark.parametrize("M", [8, 24, 48, 100, 128, 256])
@pytest.mark.parametrize("K", [1040, 3600])
@pytest.mark.parametrize("small", [True, False])
def test_gemm_int8_decode_tiles(M, K, small):
    """The decode kernel at every token-tile width (16 .. 128), K ragged against
    the 256-deep stage (1040 = 4 stages + 16, 3600 = 14 stages + 16) and split
    across CTAs, with small activation codes (one fp32 pass per split) and
    uniform ones (1024-deep chunks)."""
    N = 1160  # 9 channel tiles + 8 rows: few tiles, so K is split
    g = np.random.Generator(np.random.PCG64(M * 131 + K + small))
    lim = 10 if small else 127
    xq = g.integers(-lim, lim + 1, size=(M, K)).astype(np.int8)
    wq = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    acc = q.gemm_acc(to_dev(xq.view(np.uint8), q.INT8), to_dev(wq.view(np.uint8), q.INT8), q.INT8,
                     q.workspace(M, N, K, q.INT8))
    sync_ok()
    np.testing.assert_array_equal(acc.cpu().numpy(), oracle.gemm_i8(xq.view(np.uint8), wq.view(np.uint8), nthreads=NT))


@pytest.mark.parametrize("M", [16, 64, 256])
@pytest.mark.parametrize("small", [True, False])
def test_gemm_int8_decode_unsplit_long_k(M, small):
    """A workspace with room for the fp16 codes, their sums and the running sums
    of chunked units but not for split partials makes every unit run over all of
    K = 4352 (17 stages): uniform codes take five 1024-deep chunks (alternating
    the two accumulators) added into the int32 running sum (the last one
    ragged), small codes one fp32 pass."""
    N, K = 392, 4352
    g = np.random.Generator(np.random.PCG64(M + 7 * small))
    lim = 10 if small else 127
    xq = g.integers(-lim, lim + 1, size=(M, K)).astype(np.int8)
    wq = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # fp16 codes, their sums, the per-CTA running sums of chunked units (128 x 128 int32 each) and
    # the fused entries' handoff counters
    act = ((M * K * 2 + 255) // 256) * 256 + ((M * 4 + 255) // 256) * 256 + sms * 128 * 128 * 4 + 256
    assert q.qurl_workspace_size(M, N, K, q.INT8) > act  # the full-size plan would split K
    ws = torch.empty(act, dtype=torch.uint8, device="cuda")
    acc = q.gemm_acc(to_dev(xq.view(np.uint8), q.INT8), to_dev(wq.view(np.uint8), q.INT8), q.INT8, ws)
    sync_ok()
    np.testing.assert_array_equal(acc.cpu().numpy(), oracle.gemm_i8(xq.view(np.uint8), wq.view(np.uint8), nthreads=NT))


def test_gemm_int8_prefill_repeatable():
    """A prefill shape (on the CTA pairs) where every pair walks ~4 units of
    14 stages, so each shared-memory slot and TMEM stage is reused hundreds of
    times: three runs must agree bit for bit (a slot released before its reads
    had landed once corrupted ~1% of the outputs, differently on every run),
    and a sample matches the oracle."""
    M, N, K = 4096, 4608, 3584
    X = synth.activations("gpu/repeat/X", M, K)
    W = synth.weights("gpu/repeat/W", N, K)
    Wq, _, _, _ = q.prepare_weights(W.cuda(), q.INT8, s=1.5, keep_scaled=False)
    Xq, _ = q.quant_act(X.cuda(), q.INT8)
    ws = q.workspace(M, N, K, q.INT8)
    runs = [q.gemm_acc(Xq, Wq, q.INT8, ws) for _ in range(3)]
    sync_ok()
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[0], runs[2])
    g = np.random.Generator(np.random.PCG64(17))
    rows = np.sort(g.choice(M, size=64, replace=False))
    cols = np.sort(g.choice(N, size=256, replace=False))
    ref = oracle.gemm_i8(codes(Xq)[rows], codes(Wq)[cols], nthreads=NT)
    np.testing.assert_array_equal(runs[0].cpu().numpy()[np.ix_(rows, cols)], ref)


def pair_tmem_workspace(M, N, K):
    """A workspace one byte short of what the kernel with widened weights needs:
    the plan falls back to the CTA-pair kernel with the widened weights in TMEM."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wide = q.plan(M, N, K, q.INT8, sms)
    assert wide["kernel"] == 4
    p = q.plan(M, N, K, q.INT8, sms, ws_bytes=wide["ws_bytes"] - 1)
    assert p["kernel"] == 2
    return torch.empty(p["ws_bytes"], dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("M,N,K", [(1536, 8192, 4096), (2000, 4000, 4000)])
def test_gemm_int8_pair_modes(M, N, K):
    """Prefill shapes on the 256 x 256 CTA pairs (ragged in M, N and K in the
    second case: the last 256-deep stage reads 160 codes and zero fill):
    token tiles alternate between small codes (one fp32 pass, N = 256 MMAs) and
    full-range codes (chunked: two N = 128 half passes, each in 1024-deep chunks
    with the int32 running sum in the accumulator's upper half); exact int32
    against the oracle on rows from every tile edge."""
    g = np.random.Generator(np.random.PCG64(M + N))
    xq = g.integers(-10, 11, size=(M, K)).astype(np.int8)
    big = (np.arange(M) // 256) % 2 == 1
    xq[big] = g.integers(-127, 128, size=(int(big.sum()), K)).astype(np.int8)
    wq = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    acc = q.gemm_acc(to_dev(xq.view(np.uint8), q.INT8), to_dev(wq.view(np.uint8), q.INT8), q.INT8,
                     pair_tmem_workspace(M, N, K))
    sync_ok()
    edges = [r for t0 in range(0, M, 64) for r in (t0, t0 + 31, t0 + 63) if r < M] + [M - 1]
    rows = np.unique(np.array(edges))
    cols = np.unique(np.concatenate([np.sort(g.choice(N, size=96, replace=False)), [0, 127, 128, 255, N - 1]]))
    ref = oracle.gemm_i8(xq[rows].view(np.uint8), wq[cols].view(np.uint8), nthreads=NT)
    got = acc[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()
    np.testing.assert_array_equal(got, ref)


def test_fp8_pair_prefill_repeatable():
    """FP8 prefill on the CTA pairs: three runs of the fp32 accumulators agree
    bit for bit, and a sample lies within the fp32 accumulation bound of the
    oracle's exact sums."""
    M, N, K = 4096, 4608, 3584
    assert q.plan(M, N, K, q.FP8_E4M3, torch.cuda.get_device_properties(0).multi_processor_count)["kernel"] == 3
    xq = random_codes(q.FP8_E4M3, (M, K), 41)
    wq = random_codes(q.FP8_E4M3, (N, K), 43)
    Xd, Wd = to_dev(xq, q.FP8_E4M3), to_dev(wq, q.FP8_E4M3)
    ws = q.workspace(M, N, K, q.FP8_E4M3)
    runs = [q.gemm_acc(Xd, Wd, q.FP8_E4M3, ws) for _ in range(3)]
    sync_ok()
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[0], runs[2])
    g = np.random.Generator(np.random.PCG64(19))
    rows = np.unique(np.concatenate([np.sort(g.choice(M, size=48, replace=False)), [0, 255, 256, M - 1]]))
    cols = np.unique(np.concatenate([np.sort(g.choice(N, size=96, replace=False)), [0, 127, 128, 255, N - 1]]))
    ref = oracle.gemm_fp8(xq[rows], wq[cols], nthreads=NT)
    absref = oracle.gemm_fp8(xq[rows] & np.uint8(0x7F), wq[cols] & np.uint8(0x7F), nthreads=NT)
    got = runs[0].cpu().numpy()[np.ix_(rows, cols)].astype(np.float64)
    assert np.all(np.abs(got - ref) <= absref * (K * 2.0 ** -23) + 1e-30)


def test_gemm_int8_more_units_than_mode_slots():
    """7 x 1400 tiles of 256 x 256 on the CTA pairs with the widened weights in
    TMEM (the workspace leaves no room to widen the weights in it): every pair
    walks ~129 units, beyond the 128 whose accumulation mode the kernel records,
    so the last ones take the chunked path (two half passes) without a recorded
    mode."""
    M, N, K = 256 * 7, 256 * 1400, 256
    g = np.random.Generator(np.random.PCG64(23))
    xq = g.integers(-20, 21, size=(M, K)).astype(np.int8)
    wq = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    acc = q.gemm_acc(to_dev(xq.view(np.uint8), q.INT8), to_dev(wq.view(np.uint8), q.INT8), q.INT8,
                     pair_tmem_workspace(M, N, K))
    sync_ok()
    rows = np.sort(g.choice(M, size=96, replace=False))
    rows[-1] = M - 1  # a token of the last tile (the last units of their CTAs)
    cols = np.sort(g.choice(N, size=128, replace=False))
    ref = oracle.gemm_i8(xq[rows].view(np.uint8), wq[cols].view(np.uint8), nthreads=NT)
    got = acc[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()
    del acc
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("M", [200, 256])
def test_gemm_int8_mixed_token_tiles(M):
    """Two 128-token tiles: the first with small activation codes (one fp32 pass
    over K), the second with uniform codes whose sum |x| needs 1024-deep chunks;
    through the unfused linear (codes widened by a separate kernel) and the
    accumulator entry point."""
    N, K = 384, 4096
    g = np.random.Generator(np.random.PCG64(M))
    xq = g.integers(-127, 128, size=(M, K)).astype(np.int8)
    xq[:128] = g.integers(-20, 21, size=(128, K)).astype(np.int8)
    wq = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    xd, wd = to_dev(xq.view(np.uint8), q.INT8), to_dev(wq.view(np.uint8), q.INT8)
    ws = q.workspace(M, N, K, q.INT8)
    acc = q.gemm_acc(xd, wd, q.INT8, ws)
    sx = torch.rand(M, device="cuda") * 1e-2 + 1e-3
    sw = torch.rand(N, device="cuda") * 1e-2 + 1e-3
    Y = q.linear(xd, sx, wd, sw, q.INT8, ws)
    sync_ok()
    ref = oracle.gemm_i8(xq.view(np.uint8), wq.view(np.uint8), nthreads=NT)
    np.testing.assert_array_equal(acc.cpu().numpy(), ref)
    Yo = oracle.epilogue(ref, f32(sx), f32(sw))
    np.testing.assert_array_equal(bits(Y), Yo)


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_acc_fp8(M, N, K):
    xq = random_codes(q.FP8_E4M3, (M, K), M * 7 + K)
    wq = random_codes(q.FP8_E4M3, (N, K), N * 13 + K)
    acc = q.gemm_acc(to_dev(xq, q.FP8_E4M3), to_dev(wq, q.FP8_E4M3), q.FP8_E4M3, q.workspace(M, N, K, q.FP8_E4M3))
    sync_ok()
    ref = oracle.gemm_fp8(xq, wq, nthreads=NT)
    absref = oracle.gemm_fp8(xq & np.uint8(0x7F), wq & np.uint8(0x7F), nthreads=NT)  # sum_k |x w|, exact
    err = np.abs(acc.cpu().numpy().astype(np.float64) - ref)
    # fp32 accumulation: a few units of 2^-24 per term at worst, bounded by K
    bound = absref * (K * 2.0 ** -23) + 1e-30
    assert np.all(err <= bound), float((err / bound).max())
    assert float((err / (absref + 1e-30)).max()) < 1e-4


@pytest.mark.parametrize("M,N,K", [(1024, 5120, 27648), (1000, 5000, 12288), (2048, 5120, 27648)])
def test_fp8_pair_whole_units_and_split_tail(M, N, K):
    """FP8 prefill on CTA pairs with 80 tiles on 76 pairs: 76 tiles run over
    all of K and write their results themselves, the last 4 (the last channel
    tile of every token tile; ragged in both at 1000 x 5000) are split 18 and
    16 ways and reduced by their own kernel; at 2048 x 5120 x 27648 (160
    tiles: 152 whole, 8 split) the 56 MB of activations also put the tiles in
    groups of 7 token tiles (the last group short).  Raw accumulators
    (sampled, against the oracle within the fp32 summation bound) and the bf16
    linear (bits of the accumulators through the epilogue the oracle
    applies)."""
    xq = random_codes(q.FP8_E4M3, (M, K), M * 5 + K)
    wq = random_codes(q.FP8_E4M3, (N, K), N * 3 + K)
    ws = q.workspace(M, N, K, q.FP8_E4M3)
    X, W = to_dev(xq, q.FP8_E4M3), to_dev(wq, q.FP8_E4M3)
    acc = q.gemm_acc(X, W, q.FP8_E4M3, ws)
    sx = torch.rand(M, device="cuda") + 0.5
    sw = torch.rand(N, device="cuda") + 0.5
    Y = q.linear(X, sx, W, sw, q.FP8_E4M3, ws)
    sync_ok()
    g = np.random.Generator(np.random.PCG64(M + N + K))
    rows = np.unique(np.concatenate([g.choice(M, 24, replace=False), [0, 255, 256, M - 1]]))
    # columns of whole tiles and of the split tail (the last 256-channel tile)
    cols = np.unique(np.concatenate([g.choice(N, 96, replace=False), [0, 255, 256, 4863, 4864, N - 1]]))
    ref = oracle.gemm_fp8(xq[rows], wq[cols], nthreads=NT)
    absref = oracle.gemm_fp8(xq[rows] & np.uint8(0x7F), wq[cols] & np.uint8(0x7F), nthreads=NT)
    a = acc.cpu().numpy()[np.ix_(rows, cols)].astype(np.float64)
    assert np.all(np.abs(a - ref) <= absref * (K * 2.0 ** -23) + 1e-30)
    Yo = oracle.epilogue(acc.cpu().numpy()[np.ix_(rows, cols)], f32(sx)[rows], f32(sw)[cols])
    np.testing.assert_array_equal(bits(Y)[np.ix_(rows, cols)], Yo)


def _random_shapes(n, seed):
    """Seeded shapes across the decode and prefill ranges: any M and N, K a
    multiple of 16 (the row-stride rule of the codes), some with code
    magnitudes that force chunked INT8 accumulation."""
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(n):
        M = int(g.choice([g.integers(1, 65), g.integers(65, 300), g.integers(300, 1200)]))
        N = int(g.choice([g.integers(1, 200), g.integers(200, 3000)]))
        K = 16 * int(g.integers(1, 400))
        out.append((M, N, K, bool(g.integers(0, 2)), bool(g.integers(0, 2))))
    return out


@pytest.mark.parametrize("M,N,K,with_ws,big", _random_shapes(24, 2026))
@pytest.mark.parametrize("qt", QTS)
def test_gemm_random_shapes(qt, M, N, K, with_ws, big):
    """Accumulators of seeded random shapes, with the full workspace (split K,
    INT8 through the TMEM-operand kernel) or none (INT8 widened in shared
    memory): INT8 exact, FP8 within the fp32 accumulation bound."""
    g = np.random.Generator(np.random.PCG64(M * 1009 + N * 31 + K))
    if qt == q.INT8:
        lim = 127 if big else 12
        xq = g.integers(-lim, lim + 1, size=(M, K)).astype(np.int8).view(np.uint8)
        wq = g.integers(-127, 128, size=(N, K)).astype(np.int8).view(np.uint8)
    else:
        xq = random_codes(qt, (M, K), M * 7 + K + 1)
        wq = random_codes(qt, (N, K), N * 13 + K + 1)
    ws = q.workspace(M, N, K, qt) if with_ws else None
    acc = q.gemm_acc(to_dev(xq, qt), to_dev(wq, qt), qt, ws)
    sync_ok()
    if qt == q.INT8:
        np.testing.assert_array_equal(acc.cpu().numpy(), oracle.gemm_i8(xq, wq, nthreads=NT))
    else:
        ref = oracle.gemm_fp8(xq, wq, nthreads=NT)
        absref = oracle.gemm_fp8(xq & np.uint8(0x7F), wq & np.uint8(0x7F), nthreads=NT)
        err = np.abs(acc.cpu().numpy().astype(np.float64) - ref)
        assert np.all(err <= absref * (K * 2.0 ** -23) + 1e-30)


def _layer(qt, M, N, K, tag, s=1.0):
    """Oracle-quantized inputs of one projection (oracle computes every input)."""
    X = synth.activations(f"{tag}/X", M, K)
    W = synth.weights(f"{tag}/W", N, K)
    Xq, sx = oracle.quant_act(bits(X), oqt(qt))
    Wq, sw, _, _ = oracle.prepare_weights(W.numpy(), oqt(qt), s=s)
    return Xq, sx, Wq, sw


@pytest.mark.parametrize("qt", QTS)
@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_linear(qt, M, N, K):
    Xq, sx, Wq, sw = _layer(qt, M, N, K, f"gpu/lin/{M}/{N}/{K}")
    Y = q.linear(to_dev(Xq, qt), torch.from_numpy(sx).cuda(), to_dev(Wq, qt), torch.from_numpy(sw).cuda(), qt,
                 q.workspace(M, N, K, qt))
    sync_ok()
    Yo, _ = oracle.w8a8_linear(Xq, sx, Wq, sw, oqt(qt), nthreads=NT)
    yd = bits(Y)
    if qt == q.INT8:
        np.testing.assert_array_equal(yd, Yo)
    else:
        assert max_abs_rel(oracle.bf16_decode(yd), oracle.bf16_decode(Yo)) <= 1e-2


@pytest.mark.parametrize("qt", QTS)
def test_linear_output_row_stride(qt):
    """Y written into a wider buffer (row stride > N) leaves the gap untouched."""
    M, N, K = 40, 264, 512
    Xq, sx, Wq, sw = _layer(qt, M, N, K, "gpu/lin/ldy")
    Ybig = torch.full((M, N + 24), 7.0, dtype=torch.bfloat16, device="cuda")
    Y = Ybig[:, :N]
    q.qurl_w8a8_linear(to_dev(Xq, qt), torch.from_numpy(sx).cuda(), to_dev(Wq, qt), torch.from_numpy(sw).cuda(),
                       qt, Y, q.workspace(M, N, K, qt))
    sync_ok()
    Yo, _ = oracle.w8a8_linear(Xq, sx, Wq, sw, oqt(qt), nthreads=NT)
    assert torch.all(Ybig[:, N:] == 7.0)
    if qt == q.INT8:
        np.testing.assert_array_equal(bits(Y.contiguous()), Yo)
    else:
        assert max_abs_rel(oracle.bf16_decode(bits(Y.contiguous())), oracle.bf16_decode(Yo)) <= 1e-2


@pytest.mark.parametrize("qt", QTS)
def test_fused_rmsnorm_quant_linear(qt):
    M, N, K = 48, 4608, 3584
    X = synth.activations("gpu/fused/X", M, K)
    W = synth.weights("gpu/fused/W", N, K)
    g = synth.gamma("gpu/fused/g", K)
    Wq, sw, gf, _ = q.prepare_weights(W.cuda(), qt, s=1.5, gamma=g.cuda())
    Xd = X.cuda()
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Xqs = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
    sxs = torch.empty(M, dtype=torch.float32, device="cuda")
    q.qurl_rmsnorm_quant_linear(Xd, gf, 1e-6, Wq, sw, qt, Y, Xqs, sxs, q.workspace(M, N, K, qt))
    # the same steps as separate calls give the same bits
    Xq2, sx2, ms = q.rmsnorm_quant(Xd, gf, qt, eps=1e-6, want_ms=True)
    Y2 = q.linear(Xq2, sx2, Wq, sw, qt, q.workspace(M, N, K, qt))
    sync_ok()
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    # against the oracle: UAQ-folded weights and gain, layer output within 1e-2
    Wo, swo, gfo, _ = oracle.prepare_weights(W.numpy(), oqt(qt), s=1.5, gamma=g.numpy())
    qo, so, _, _ = oracle.rmsnorm_quant(bits(X), gfo, oqt(qt), eps=1e-6)
    Yo, _ = oracle.w8a8_linear(qo, so, Wo, swo, oqt(qt), nthreads=NT)
    assert max_abs_rel(oracle.bf16_decode(bits(Y)), oracle.bf16_decode(Yo)) <= 1e-2


def test_silu_over_every_bf16_gate():
    """h = silu(g) * u for every finite bf16 g in [-120, 120] (u = 1 and -3):
    within the relative 2e-6 the codes are decided on across the whole range of
    the exponential -- both tails, the reduction's boundaries at every multiple
    of ln 2 / 2, and the flush to 0 below g = -87.3."""
    v = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    g = v[torch.isfinite(v) & (v.abs() <= 120)]
    I = ((g.numel() + 15) // 16) * 16
    gate = torch.zeros(I)
    gate[: g.numel()] = g
    GU = torch.stack([torch.cat([gate, torch.ones(I)]), torch.cat([gate, torch.full((I,), -3.0)])])
    GU = GU.to(torch.bfloat16)
    _, _, h = q.silu_mul_quant(GU.cuda(), q.FP8_E4M3, pre_scale=1.0, want_h=True)
    sync_ok()
    _, _, ho = oracle.silu_mul_quant(bits(GU), oracle.FP8_E4M3, pre_scale=1.0)
    np.testing.assert_allclose(f32(h), ho, rtol=2e-6, atol=1e-35)


@pytest.mark.parametrize("qt", QTS)
def test_silu_stream_linear_matches_separate_calls(qt):
    """SiLU*mul -> quant -> linear at a streamed row width (I = 27648, 300
    rows): the fp16 codes and code sums the quantizer leaves for the INT8 GEMM
    give the bits of the quantizer + linear called apart, and the codes are the
    oracle's given the kernel's h."""
    M, N, I = 300, 512, 27648
    GU = synth.activations(f"gpu/fqs/GU/{M}", M, 2 * I, outlier_gain=4.0)
    W = synth.weights("gpu/fqs/W", N, I)
    Wq, sw, _, _ = q.prepare_weights(W.cuda(), qt, s=1.5)
    cd = q.code_dtype(qt)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    xs = torch.empty((M, I), dtype=cd, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    q.qurl_silu_mul_quant_linear(GU.cuda(), 1.5, Wq, sw, qt, Y, xs, sx, q.workspace(M, N, I, qt))
    Xq, s2, h = q.silu_mul_quant(GU.cuda(), qt, pre_scale=1.5, want_h=True)
    R = q.linear(Xq, s2, Wq, sw, qt, q.workspace(M, N, I, qt))
    sync_ok()
    assert torch.equal(xs.view(torch.uint8), Xq.view(torch.uint8)) and torch.equal(sx, s2)
    assert torch.equal(Y.view(torch.int16), R.view(torch.int16))
    qo, so, _ = oracle.silu_mul_quant(bits(GU), oqt(qt), pre_scale=1.5, h_given=f32(h))
    np.testing.assert_array_equal(codes(Xq), qo)
    np.testing.assert_array_equal(f32(s2), so)


@pytest.mark.parametrize("qt", QTS)
@pytest.mark.parametrize("M", [64, 200, 300])
def test_fused_quant_entries(qt, M):
    """quant_act -> linear and SiLU*mul -> quant -> linear, fused, give the bits
    of the separate calls (which the oracle checks above), and the layer output
    stays within 1e-2 of the oracle's chain."""
    K, N, I = 1024, 768, 2048
    X = synth.activations(f"gpu/fq/X/{M}", M, K)
    GU = synth.activations(f"gpu/fq/GU/{M}", M, 2 * I, outlier_gain=4.0)
    W1 = synth.weights("gpu/fq/W1", N, K)
    W2 = synth.weights("gpu/fq/W2", N, I)
    Wq1, sw1, _, _ = q.prepare_weights(W1.cuda(), qt, s=1.5)
    Wq2, sw2, _, _ = q.prepare_weights(W2.cuda(), qt, s=1.5)
    cd = q.code_dtype(qt)
    Y1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Y2 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    xs1 = torch.empty((M, K), dtype=cd, device="cuda")
    xs2 = torch.empty((M, I), dtype=cd, device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    sx2 = torch.empty(M, dtype=torch.float32, device="cuda")
    q.qurl_quant_act_linear(X.cuda(), 1.5, Wq1, sw1, qt, Y1, xs1, sx, q.workspace(M, N, K, qt))
    q.qurl_silu_mul_quant_linear(GU.cuda(), 1.5, Wq2, sw2, qt, Y2, xs2, sx2, q.workspace(M, N, I, qt))
    Xq1, s1 = q.quant_act(X.cuda(), qt, pre_scale=1.5)
    # INT8: no workspace runs the other INT8 kernel, with the same exact bits; FP8 sums in fp32, so
    # the comparison keeps the same plan (same K split, same summation order)
    R1 = q.linear(Xq1, s1, Wq1, sw1, qt, None if qt == q.INT8 else q.workspace(M, N, K, qt))
    Xq2, s2 = q.silu_mul_quant(GU.cuda(), qt, pre_scale=1.5)
    R2 = q.linear(Xq2, s2, Wq2, sw2, qt, q.workspace(M, N, I, qt))
    sync_ok()
    assert torch.equal(Y1.view(torch.int16), R1.view(torch.int16))
    assert torch.equal(Y2.view(torch.int16), R2.view(torch.int16))
    Wo, swo, _, _ = oracle.prepare_weights(W1.numpy(), oqt(qt), s=1.5)
    qo, so = oracle.quant_act(bits(X), oqt(qt), pre_scale=1.5)
    Yo, _ = oracle.w8a8_linear(qo, so, Wo, swo, oqt(qt), nthreads=NT)
    if qt == q.INT8:
        np.testing.assert_array_equal(bits(Y1), Yo)
    else:
        assert max_abs_rel(oracle.bf16_decode(bits(Y1)), oracle.bf16_decode(Yo)) <= 1e-2


@pytest.mark.parametrize("M,N,K", [(16, 512, 256), (64, 4608, 3584), (256, 1000, 2048)])
def test_linear_int8_with_and_without_workspace(M, N, K):
    """INT8 decode runs the TMEM-operand kernel with a workspace and the
    shared-memory widening kernel without one: the same exact bits."""
    Xq, sx, Wq, sw = _layer(q.INT8, M, N, K, f"gpu/lin/ws/{M}/{N}/{K}")
    args = (to_dev(Xq, q.INT8), torch.from_numpy(sx).cuda(), to_dev(Wq, q.INT8), torch.from_numpy(sw).cuda(), q.INT8)
    Ya = q.linear(*args, q.workspace(M, N, K, q.INT8))
    Yb = q.linear(*args, None)
    sync_ok()
    Yo, _ = oracle.w8a8_linear(Xq, sx, Wq, sw, oracle.INT8, nthreads=NT)
    np.testing.assert_array_equal(bits(Ya), Yo)
    np.testing.assert_array_equal(bits(Yb), Yo)


@pytest.mark.parametrize("qt", QTS)
def test_split_k_reduction(qt):
    """Decode shapes whose K is split across CTAs (4 to 300 channel tiles): each
    split writes its partial and a reduction kernel sums them in split order.
    Launches per call: the GEMM, the reduction when K is split, and for INT8 the
    widening of the activation codes."""
    M, K = 64, 2048
    for tiles in (4, 36, 75, 150, 300):
        N = tiles * 128
        Xq, sx, Wq, sw = _layer(qt, M, N, K, f"gpu/splitk/{tiles}")
        ws = q.workspace(M, N, K, qt)
        args = (to_dev(Xq, qt), torch.from_numpy(sx).cuda(), to_dev(Wq, qt), torch.from_numpy(sw).cuda(), qt)
        torch.cuda.synchronize()
        n0 = q.qurl_kernel_launches()
        Y = q.linear(*args, ws)
        launches = q.qurl_kernel_launches() - n0
        acc = q.gemm_acc(args[0], args[2], qt, ws)
        sync_ok()
        split = q.plan(M, N, K, qt, torch.cuda.get_device_properties(0).multi_processor_count)["splits"] > 1
        assert launches == 1 + int(split) + int(qt == q.INT8), (tiles, launches)
        Yo, acco = oracle.w8a8_linear(Xq, sx, Wq, sw, oqt(qt), nthreads=NT)
        if qt == q.INT8:
            np.testing.assert_array_equal(bits(Y), Yo)
            np.testing.assert_array_equal(acc.cpu().numpy(), acco)
        else:
            assert max_abs_rel(oracle.bf16_decode(bits(Y)), oracle.bf16_decode(Yo)) <= 1e-2


def test_split_workspace_reused_across_calls():
    """One workspace serves consecutive split-K calls of different shapes and
    kinds (linear, raw accumulators): nothing a call leaves behind -- fp16
    codes, code sums, partials of another shape -- changes the next result."""
    M, K = 64, 3584
    ws = q.workspace(M, 4608, K, q.INT8)
    for N, tag in ((4608, "a"), (3584, "b"), (4608, "a")):
        assert q.qurl_workspace_size(M, N, K, q.INT8) <= ws.numel()
        Xq, sx, Wq, sw = _layer(q.INT8, M, N, K, f"gpu/splitreuse/{tag}")
        args = (to_dev(Xq, q.INT8), torch.from_numpy(sx).cuda(), to_dev(Wq, q.INT8), torch.from_numpy(sw).cuda(),
                q.INT8)
        Y1 = q.linear(*args, ws)
        acc = q.gemm_acc(args[0], args[2], q.INT8, ws)
        Y2 = q.linear(*args, ws)
        sync_ok()
        Yo, acco = oracle.w8a8_linear(Xq, sx, Wq, sw, oracle.INT8, nthreads=NT)
        np.testing.assert_array_equal(bits(Y1), Yo)
        np.testing.assert_array_equal(bits(Y2), Yo)
        np.testing.assert_array_equal(acc.cpu().numpy(), acco)


# ------------------------------------------------------------------ full-size projections (sampled)

FULL = [
    # (model, proj, M, qtype): the 7B decode set is the benchmark workload
    ("7b", "qkv", 64, q.INT8), ("7b", "gate_up", 64, q.INT8), ("7b", "down", 64, q.INT8),
    ("7b", "qkv", 256, q.INT8), ("7b", "o_proj", 256, q.INT8), ("7b", "gate_up", 256, q.INT8),
    ("7b", "down", 256, q.INT8),
    ("7b", "gate_up", 256, q.FP8_E4M3), ("7b", "down", 64, q.FP8_E4M3), ("7b", "qkv", 4096, q.FP8_E4M3),
    ("32b", "gate_up", 1024, q.INT8), ("32b", "down", 256, q.FP8_E4M3), ("32b", "o_proj", 8192, q.FP8_E4M3),
    ("32b", "qkv", 8192, q.INT8),
    # shapes whose K is split to fill the last wave (320 and 160 tiles on 152 SMs; 80 tiles)
    ("32b", "down", 1024, q.INT8), ("32b", "down", 1024, q.FP8_E4M3), ("32b", "down", 256, q.INT8),
]


@pytest.mark.parametrize("model,proj,M,qt", FULL)
def test_full_size_projection_sampled(model, proj, M, qt):
    K, N = (synth.SHAPES_7B if model == "7b" else synth.SHAPES_32B)[proj]
    tag = f"gpu/full/{model}/{proj}/{M}"
    X = synth.activations(f"{tag}/X", M, K)
    W = synth.weights(f"{tag}/W", N, K)
    Wq, sw, _, _ = q.prepare_weights(W.cuda(), qt, s=1.5, keep_scaled=False)
    Xq, sx = q.quant_act(X.cuda(), qt)
    Y = q.linear(Xq, sx, Wq, sw, qt, q.workspace(M, N, K, qt))
    sync_ok()
    g = np.random.Generator(np.random.PCG64(M * 31 + N))
    rows = np.sort(g.choice(M, size=min(M, 96), replace=False))
    cols = np.sort(g.choice(N, size=160, replace=False))
    # oracle inputs from the oracle: the sampled weight rows and token rows
    Wo, swo, _, _ = oracle.prepare_weights(W.numpy()[cols], oqt(qt), s=1.5)
    Xo, sxo = oracle.quant_act(bits(X[rows]), oqt(qt))
    np.testing.assert_array_equal(codes(Wq)[cols], Wo)  # the GPU inputs equal the oracle's
    np.testing.assert_array_equal(codes(Xq)[rows], Xo)
    Yo, _ = oracle.w8a8_linear(Xo, sxo, Wo, swo, oqt(qt), nthreads=NT)
    yd = bits(Y)[np.ix_(rows, cols)]
    if qt == q.INT8:
        np.testing.assert_array_equal(yd, Yo)
    else:
        assert max_abs_rel(oracle.bf16_decode(yd), oracle.bf16_decode(Yo)) <= 1e-2


# ------------------------------------------------------------------ flip probe

@pytest.mark.parametrize("n", [16, 100_003, 1 << 22])
def test_count_diff_exact(n):
    g = np.random.Generator(np.random.PCG64(n))
    a = g.integers(0, 256, size=n, dtype=np.uint8)
    b = a.copy()
    idx = g.choice(n, size=max(1, n // 97), replace=False)
    b[idx] ^= np.uint8(0x41)
    c = q.count_diff(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda())
    sync_ok()
    assert int(c.item()) == oracle.count_diff(a, b) == len(idx)


@pytest.mark.parametrize("qt", QTS)
def test_flip_probe_matches_oracle(qt):
    """Re-quantize W' and W' + dW' on the GPU and count flipped codes: the count
    equals the oracle's, and UAQ (s = 1.5) flips more codes than s = 1."""
    N, K = 1024, 3584
    W = synth.weights("gpu/flip/W", N, K)
    dW = synth.update("gpu/flip/dW", N, K)
    counts = {}
    for s in (1.0, 1.5):
        Wq0, _, _, Ws = q.prepare_weights(W.cuda(), qt, s=s)
        Ws1 = Ws + float(s) * dW.cuda()  # SGD view: the update lands in W' space scaled by s
        Wq1, _, _, _ = q.prepare_weights(Ws1, qt, s=1.0, keep_scaled=False)
        c = int(q.count_diff(Wq0, Wq1).item())
        sync_ok()
        a0, _, _, Wso = oracle.prepare_weights(W.numpy(), oqt(qt), s=s)
        a1, _, _, _ = oracle.prepare_weights(Wso + np.float32(s) * dW.numpy(), oqt(qt), s=1.0)
        assert c == oracle.count_diff(a0, a1)
        counts[s] = c
    assert counts[1.5] > 1.5 * counts[1.0]
