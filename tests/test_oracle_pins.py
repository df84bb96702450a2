"""Pins of the CPU oracle against things other than itself.

Each test checks an oracle function against a library routine (torch CPU casts
and rounding, numpy integer / fp64 matmul), a closed form, an invariant, or a
hand-derived worked example (tests/golden/worked_examples.json).  A plausible
mistake in the oracle -- a dropped term, a wrong sign, a transposed operand, a
wrong rounding direction, a scale on the wrong axis -- fails one of them.

Source of the method: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement
Learning with Quantized Rollout": section "更新感知量化 (UAQ)" (W X = (W/s)(sX),
s folded into the norm gain; quantization error ~ |theta|/(s 2^b) falls by s,
update ~ s alpha G grows by s), section "损失函数 / 训练策略" (per-channel weight +
per-token activation INT8/FP8, s = 1.5), section "研究背景与动机" (updates ~1e-7
are masked by the quantization error).
"""
import json
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from w8a8_precision_gemm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def torch_e4m3(v: np.ndarray) -> np.ndarray:
    """Library special case: torch CPU fp32 -> float8_e4m3fn (RNE), after a clamp to +-448."""
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ----------------------------------------------------------------- e4m3 encode

def _check_chunk(bounds):
    a, b = bounds
    bits = np.arange(a, b, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    import oracle

    got = oracle.e4m3_encode(v)
    exp = torch_e4m3(v)
    bad = np.nonzero(got != exp)[0]
    return (len(bad), None if len(bad) == 0 else (hex(int(bits[bad[0]])), int(got[bad[0]]), int(exp[bad[0]])))


def test_e4m3_encode_exhaustive_all_fp32(orc):
    """Every one of the 2^32 fp32 bit patterns (both signs, zeros, subnormals,
    infinities and NaNs) against torch's cast; ~15 s on 8 cores."""
    step = 1 << 24
    chunks = [(a, a + step) for a in range(0, 1 << 32, step)]
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(_check_chunk, chunks))
    bad = [r for r in results if r[0]]
    assert not bad, bad[:3]


def test_e4m3_encode_edges(orc):
    """Rounding and saturation edges, by value."""
    edges = np.array([0.0, -0.0, 2.0 ** -10, -(2.0 ** -10), np.nextafter(np.float32(2.0 ** -10), np.float32(1)),
                      448.0, -448.0, 464.0, 463.99997, 465.0, 1e30, -1e30, np.inf, -np.inf,
                      2.0 ** -149, -(2.0 ** -149), 2.0 ** -126], dtype=np.float32)
    np.testing.assert_array_equal(orc.e4m3_encode(edges), torch_e4m3(edges))
    assert orc.e4m3_encode(edges[:5]).tolist() == [0x00, 0x80, 0x00, 0x80, 0x01]
    assert orc.e4m3_encode(edges[5:10]).tolist() == [0x7E, 0xFE, 0x7E, 0x7E, 0x7E]


def test_e4m3_decode_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    dec = orc.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(dec), nan)
    assert nan.sum() == 2  # S.1111.111
    np.testing.assert_array_equal(dec[~nan], lib[~nan])
    # closed-form special values of the format
    assert dec[0x7E] == 448.0 and dec[0xFE] == -448.0
    assert dec[0x01] == 2.0 ** -9 and dec[0x08] == 2.0 ** -6 and dec[0x38] == 1.0


def test_e4m3_roundtrip_is_identity_on_grid(orc):
    grid = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    ok = ~np.isnan(grid)
    codes = np.arange(256, dtype=np.uint8)[ok]
    np.testing.assert_array_equal(orc.e4m3_encode(grid[ok].astype(np.float32)), codes)


# ----------------------------------------------------------------- bf16

def test_bf16_encode_against_torch(orc):
    g = np.random.Generator(np.random.PCG64(7))
    bits = g.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    # exact ties (low 16 bits = 0x8000) with both parities, and carries into the exponent
    ties = (g.integers(0, 1 << 16, size=20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    v = np.concatenate([bits, ties, np.array([0x3F7FFFFF, 0x7F7FFFFF, 0x7F7F8000, 0x00008000], np.uint32)])
    v = v.view(np.float32)
    v = v[~np.isnan(v)]
    lib = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(orc.bf16_encode(v), lib)


# ----------------------------------------------------------------- row quantization

def _rows(seed, M, K):
    g = np.random.Generator(np.random.PCG64(seed))
    V = g.standard_normal((M, K), dtype=np.float32) * np.float32(0.02)
    V[:, :: max(1, K // 7)] *= np.float32(20.0)
    return V


def test_int8_quant_rows_against_torch_round(orc):
    """Library special case: torch fp32 division and torch.round (ties to even)."""
    V = _rows(1, 64, 1000)
    q, s = orc.quant_rows(V, orc.INT8)
    t = torch.from_numpy(V)
    a = t.abs().amax(dim=1)
    scale = a / torch.tensor(127.0)
    codes = torch.round(t / scale[:, None]).clamp(-127, 127).to(torch.int8)
    np.testing.assert_array_equal(s, scale.numpy())
    np.testing.assert_array_equal(q.view(np.int8), codes.numpy())


def test_fp8_quant_rows_against_torch_cast(orc):
    V = _rows(2, 64, 1000)
    q, s = orc.quant_rows(V, orc.FP8_E4M3)
    t = torch.from_numpy(V)
    scale = t.abs().amax(dim=1) / torch.tensor(448.0)
    np.testing.assert_array_equal(s, scale.numpy())
    np.testing.assert_array_equal(q, torch_e4m3((t / scale[:, None]).numpy()))


def test_int8_roundtrip_bound_and_range(orc):
    """|w - q*scale| <= scale/2 per element (one fp32 ulp of slack for the division)
    and every non-zero row reaches the code 127 in magnitude."""
    V = _rows(3, 128, 777)
    q, s = orc.quant_rows(V, orc.INT8)
    qi = q.view(np.int8).astype(np.float64)
    err = np.abs(V.astype(np.float64) - qi * s[:, None].astype(np.float64))
    bound = s[:, None].astype(np.float64) * (0.5 + 128 * 2.0 ** -23)
    assert np.all(err <= bound)
    assert np.all(np.abs(qi).max(axis=1) == 127)
    assert np.all(np.abs(qi) <= 127)


def test_fp8_roundtrip_bound(orc):
    """|w - dec(q)*scale| <= scale * ulp_e4m3(q) / 2 (+ an fp32 ulp), i.e. at most
    2^-4 |w| for normals and 2^-10 scale for subnormals; each row reaches 448."""
    V = _rows(4, 128, 777)
    q, s = orc.quant_rows(V, orc.FP8_E4M3)
    dec = orc.e4m3_decode(q)
    r = V.astype(np.float64) / s[:, None].astype(np.float64)
    ad = np.abs(dec)
    ulp = np.where(ad < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(ad, 2.0 ** -6))) - 3))
    # the rounding interval of a code is half an ulp on either side (at a binade
    # edge the lower side is half of the smaller ulp, which the larger bounds)
    assert np.all(np.abs(r - dec) <= ulp / 2 * (1 + 1e-6) + np.abs(r) * 2.0 ** -23)
    assert np.all(np.abs(dec).max(axis=1) == 448.0)


def test_zero_row_and_worked_examples(orc):
    gold = json.load(open(GOLDEN))
    for case in gold["int8_rows"]:
        q, s = orc.quant_rows(np.array([case["w"]], np.float32), orc.INT8)
        assert s[0] == np.float32(case["scale"]), case["cite"]
        assert q.view(np.int8)[0].tolist() == case["codes"], case["derivation"]
    for case in gold["fp8_rows"]:
        q, s = orc.quant_rows(np.array([case["w"]], np.float32), orc.FP8_E4M3)
        assert s[0] == np.float32(case["scale"])
        assert q[0].tolist() == case["codes"], case["derivation"]
    u = gold["uaq_int8"]
    Wq, sw, gf, Ws = orc.prepare_weights(np.array([u["w"]], np.float32), orc.INT8, s=u["s"],
                                         gamma=np.array(u["gamma"], np.float32))
    assert Ws[0].tolist() == u["w_scaled"]
    assert Wq.view(np.int8)[0].tolist() == u["codes"]
    assert gf.tolist() == u["gamma_folded"]
    assert sw[0] == np.float32(1.0) / np.float32(127.0)
    g = gold["gemm_int8"]
    acc = orc.gemm_i8(np.array(g["xq"], np.int8).view(np.uint8), np.array(g["wq"], np.int8).view(np.uint8))
    assert acc.tolist() == g["acc"]
    g = gold["gemm_fp8"]
    acc = orc.gemm_fp8(np.array(g["xq"], np.uint8), np.array(g["wq"], np.uint8))
    assert acc.tolist() == g["acc"]
    for e in gold["epilogue"]:
        Y = orc.epilogue(np.array(e["acc"], np.int32), np.array(e["sx"], np.float32), np.array(e["sw"], np.float32))
        assert Y.tolist() == e["y_bits"], e["derivation"]


def test_quant_act_matches_row_quant_of_bf16_values(orc):
    """a4 = per-token quantization of fp32(bf16 x) * pre_scale."""
    X = synth.activations("pin/act", 33, 512)
    xb = synth.bf16_bits(X)
    for qt in (orc.INT8, orc.FP8_E4M3):
        for pre in (1.0, 1.5):
            q, s = orc.quant_act(xb, qt, pre_scale=pre)
            v = X.float().numpy() * np.float32(pre)
            q2, s2 = orc.quant_rows(v, qt)
            np.testing.assert_array_equal(q, q2)
            np.testing.assert_array_equal(s, s2)
    # against torch directly for INT8
    q, s = orc.quant_act(xb, orc.INT8)
    t = X.float()
    scale = t.abs().amax(1) / 127.0
    np.testing.assert_array_equal(q.view(np.int8), torch.round(t / scale[:, None]).clamp(-127, 127).to(torch.int8).numpy())


# ----------------------------------------------------------------- GEMM + epilogue

@pytest.mark.parametrize("M,N,K", [(16, 512, 256), (5, 37, 96), (1, 1, 16)])
def test_gemm_int8_against_numpy(orc, M, N, K):
    g = np.random.Generator(np.random.PCG64(M * 1000 + N))
    Xq = g.integers(-127, 128, size=(M, K)).astype(np.int8)
    Wq = g.integers(-127, 128, size=(N, K)).astype(np.int8)
    acc = orc.gemm_i8(Xq.view(np.uint8), Wq.view(np.uint8), nthreads=3)
    ref = Xq.astype(np.int64) @ Wq.astype(np.int64).T
    np.testing.assert_array_equal(acc.astype(np.int64), ref)


def test_gemm_int8_worst_case_and_overflow(orc):
    """|acc| <= 127^2 K: K = 27648 (the largest in-feature count) gives 445,934,592 < 2^31."""
    K = 27648
    Xq = np.full((2, K), 127, np.int8)
    Wq = np.stack([np.full(K, 127, np.int8), np.full(K, -127, np.int8)])
    acc = orc.gemm_i8(Xq.view(np.uint8), Wq.view(np.uint8))
    assert acc[0, 0] == 127 * 127 * K == 445_934_592 and acc[0, 1] == -445_934_592
    Kbig = 133_200  # 127^2 * 133200 > 2^31 - 1
    with pytest.raises(RuntimeError):
        orc.gemm_i8(np.full((1, Kbig), 127, np.uint8), np.full((1, Kbig), 127, np.uint8))


def test_gemm_fp8_against_numpy_fp64(orc):
    g = np.random.Generator(np.random.PCG64(11))
    M, N, K = 9, 70, 320
    codes = np.arange(256, dtype=np.uint8)
    finite = codes[~np.isnan(torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy())]
    Xq = g.choice(finite, size=(M, K))
    Wq = g.choice(finite, size=(N, K))
    acc = orc.gemm_fp8(Xq, Wq, nthreads=2)
    dx = torch.from_numpy(Xq).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    dw = torch.from_numpy(Wq).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(acc, dx @ dw.T)  # every sum is exact in fp64


def test_epilogue_against_torch(orc):
    g = np.random.Generator(np.random.PCG64(12))
    M, N = 17, 300
    acc = g.integers(-(2 ** 28), 2 ** 28, size=(M, N)).astype(np.int32)
    sx = (g.random(M, dtype=np.float32) + np.float32(0.01)) * np.float32(0.1)
    sw = (g.random(N, dtype=np.float32) + np.float32(0.01)) * np.float32(1e-3)
    Y = orc.epilogue(acc, sx, sw)
    ref = ((torch.from_numpy(acc).float() * torch.from_numpy(sx)[:, None]) * torch.from_numpy(sw)[None, :])
    ref = ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(Y, ref)
    accf = g.standard_normal((M, N)) * 1e4
    Yf = orc.epilogue(accf, sx, sw)
    ref = ((torch.from_numpy(accf).float() * torch.from_numpy(sx)[:, None]) * torch.from_numpy(sw)[None, :])
    np.testing.assert_array_equal(Yf, ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_w8a8_linear_tracks_fp64_linear(orc):
    """End to end on the tiny layer (M=16, K=256, N=512): the quantized linear is
    close to the unquantized fp64 product (the quantization error bound), and the
    operands are not transposed (a transposition would make it unrelated)."""
    X = synth.activations("pin/tiny/X", 16, 256)
    W = synth.weights("pin/tiny/W", 512, 256)
    xb = synth.bf16_bits(X)
    exact = X.double().numpy() @ W.double().numpy().T
    for qt, tol in ((orc.INT8, 0.05), (orc.FP8_E4M3, 0.08)):
        Wq, sw, _, _ = orc.prepare_weights(W.numpy(), qt, s=1.0)
        Xq, sx = orc.quant_act(xb, qt)
        Y, _ = orc.w8a8_linear(Xq, sx, Wq, sw, qt)
        y = orc.bf16_decode(Y).astype(np.float64)
        rel = np.abs(y - exact).max() / np.abs(exact).max()
        assert rel < tol, (qt, rel)


# ----------------------------------------------------------------- UAQ

def test_uaq_invariance_fp64_identity():
    """(W/s)(sX) = WX in fp64, the identity UAQ rests on (max-rel <= 1e-14)."""
    X = synth.activations("pin/uaq/X", 16, 256).double().numpy()
    W = synth.weights("pin/uaq/W", 512, 256).double().numpy()
    s = 1.5
    lhs = (W / s) @ (s * X).T
    rhs = W @ X.T
    assert np.abs(lhs - rhs).max() / np.abs(rhs).max() <= 1e-14


def test_uaq_fold_axes(orc):
    """The oracle's fold keeps the layer's function: W'(gamma'-normed x) equals
    W(gamma-normed x) up to fp32 rounding -- W is divided column-wise and the gain
    multiplied, so scaling W's rows or forgetting the gain would be O(1) off."""
    K, N, M = 256, 384, 8
    W = synth.weights("pin/fold/W", N, K).numpy()
    gam = synth.gamma("pin/fold/g", K).numpy()
    X = synth.activations("pin/fold/X", M, K)
    xb = synth.bf16_bits(X)
    for s in (1.5, 2.0, 0.75):
        _, _, gf, Ws = orc.prepare_weights(W, orc.INT8, s=s, gamma=gam)
        # RMSNorm outputs with each gain (the oracle's own normalisation)
        _, _, ms, v_folded = orc.rmsnorm_quant(xb, gf, orc.INT8)
        _, _, _, v_plain = orc.rmsnorm_quant(xb, gam, orc.INT8)
        y_folded = v_folded.astype(np.float64) @ Ws.astype(np.float64).T
        y_plain = v_plain.astype(np.float64) @ W.astype(np.float64).T
        rel = np.abs(y_folded - y_plain).max() / np.abs(y_plain).max()
        assert rel < 1e-6, (s, rel)
        np.testing.assert_array_equal(gf, gam * np.float32(s))


def test_uaq_leaves_codes_nearly_unchanged(orc):
    """With absmax scaling q(W/s) = q(W) in exact arithmetic; in fp32 a code moves
    only when w/scale sits within a few ulps of a rounding midpoint (expected
    fraction ~1e-5), and the dequantized layer output is unchanged to bf16."""
    W = synth.weights("pin/uaqcodes/W", 1024, 1024).numpy()
    for qt in (orc.INT8, orc.FP8_E4M3):
        q1, sw1, _, _ = orc.prepare_weights(W, qt, s=1.0)
        q2, sw2, _, _ = orc.prepare_weights(W, qt, s=1.5)
        frac = orc.count_diff(q1, q2) / q1.size
        assert frac <= 1e-4, frac
        np.testing.assert_allclose(sw2 * np.float32(1.5), sw1, rtol=3e-7)


# ----------------------------------------------------------------- RMSNorm, SiLU

def test_rms_ms_against_numpy(orc):
    X = synth.activations("pin/ms", 40, 3584)
    ms = orc.rms_ms(synth.bf16_bits(X))
    ref = np.mean(X.double().numpy() ** 2, axis=1)
    np.testing.assert_allclose(ms, ref, rtol=1e-13)


def test_rmsnorm_against_torch_and_constant_row(orc):
    X = synth.activations("pin/rms", 12, 1024)
    gam = synth.gamma("pin/rms/g", 1024).numpy()
    q, s, ms, v = orc.rmsnorm_quant(synth.bf16_bits(X), gam, orc.INT8, eps=1e-6)
    ref = torch.nn.functional.rms_norm(X.float(), (1024,), weight=torch.from_numpy(gam), eps=1e-6).numpy()
    np.testing.assert_allclose(v, ref, rtol=2e-6, atol=1e-6)
    # ms_given = the oracle's own fp32 ms reproduces the same codes
    q2, s2, _, _ = orc.rmsnorm_quant(synth.bf16_bits(X), gam, orc.INT8, eps=1e-6, ms_given=ms)
    np.testing.assert_array_equal(q, q2)
    np.testing.assert_array_equal(s, s2)
    # a constant row c with unit gain normalises to ~sign(c): every code is +-127
    c = torch.full((2, 64), 3.0, dtype=torch.bfloat16)
    c[1] = -0.5
    qc, sc, _, vc = orc.rmsnorm_quant(synth.bf16_bits(c), np.ones(64, np.float32), orc.INT8)
    assert qc.view(np.int8)[0].tolist() == [127] * 64 and qc.view(np.int8)[1].tolist() == [-127] * 64
    for row, cval in ((0, 3.0), (1, 0.5)):
        np.testing.assert_allclose(np.abs(vc[row]), cval / math.sqrt(cval * cval + 1e-6), rtol=1e-6)


def test_silu_mul_against_torch(orc):
    I = 700
    GU = synth.activations("pin/silu", 9, 2 * I, outlier_gain=5.0)
    GU[0, :3] = torch.tensor([0.0, -100.0, 60.0], dtype=torch.bfloat16)
    q, s, h = orc.silu_mul_quant(synth.bf16_bits(GU), orc.INT8)
    g = GU[:, :I].float()
    u = GU[:, I:].float()
    ref = (torch.nn.functional.silu(g) * u).numpy()
    np.testing.assert_allclose(h, ref, rtol=4e-6, atol=1e-30)
    assert h[0, 0] == 0.0 and abs(h[0, 1]) < 1e-30
    # codes are the per-token quantization of h * pre_scale
    q2, s2, _ = orc.silu_mul_quant(synth.bf16_bits(GU), orc.FP8_E4M3, pre_scale=1.5)
    q3, s3 = orc.quant_rows(h * np.float32(1.5), orc.FP8_E4M3)
    np.testing.assert_array_equal(q2, q3)
    np.testing.assert_array_equal(s2, s3)


# ----------------------------------------------------------------- flip probe

def test_count_diff_against_numpy(orc):
    g = np.random.Generator(np.random.PCG64(5))
    a = g.integers(0, 256, size=100_003, dtype=np.uint8)
    b = a.copy()
    idx = g.choice(a.size, size=1234, replace=False)
    b[idx] ^= np.uint8(0x10)
    assert orc.count_diff(a, b) == 1234 == int((a != b).sum())


def _expected_int8_flips(Ws, sw, sigma):
    """Closed form for a Gaussian update far smaller than the step: a code flips
    when the update carries w across a rounding midpoint, P ~ E|dw| / step with
    E|dw| = sigma sqrt(2/pi) and step = the channel scale."""
    K = Ws.shape[1]
    return float(np.sum(K * sigma * math.sqrt(2.0 / math.pi) / sw.astype(np.float64)))


def test_flip_probe_closed_form_and_s_squared(orc):
    """A ~1e-7 update flips ~1e-4 of the INT8 codes at s = 1 (the update is
    nearly masked), and UAQ with s = 1.5 flips s^2 = 2.25 times as many when the
    update is taken in W' space (SGD: dW' = s dW), s = 1.5 times as many when
    its size does not scale (Adam-like: dW' = dW)."""
    N, K = 1024, 3584
    W = synth.weights("pin/flip/W", N, K).numpy()
    dW = synth.update("pin/flip/dW", N, K).numpy()
    s = 1.5
    # s = 1: requantize W and W + dW
    q0, sw0, _, _ = orc.prepare_weights(W, orc.INT8, s=1.0)
    q1, _, _, _ = orc.prepare_weights(W + dW, orc.INT8, s=1.0)
    f1 = orc.count_diff(q0, q1)
    e1 = _expected_int8_flips(W, sw0, 1e-7)
    # UAQ: W' = W/s is the master; one update in W' space
    qa, swa, _, Ws = orc.prepare_weights(W, orc.INT8, s=s)
    qb, _, _, _ = orc.prepare_weights(Ws + np.float32(s) * dW, orc.INT8, s=1.0)
    qc, _, _, _ = orc.prepare_weights(Ws + dW, orc.INT8, s=1.0)
    f_sgd = orc.count_diff(qa, qb)
    f_adam = orc.count_diff(qa, qc)
    frac = f1 / W.size
    assert 5e-5 < frac < 3e-4, frac
    assert abs(f1 - e1) / e1 < 0.15, (f1, e1)
    assert 1.9 <= f_sgd / f1 <= 2.6, f_sgd / f1
    assert 1.3 <= f_adam / f1 <= 1.7, f_adam / f1
