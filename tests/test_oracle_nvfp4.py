"""Pins of the oracle's 4-bit (NVFP4) row quantization and GEMM (CPU only).

The pages name 4-bit quantization as the next, unexplored speedup (Paper-Notes
"QuRL", section 局限与展望; the QeRL entry of the related-papers list on the
fugumt page uses NVFP4) without defining the format; the oracle takes NVIDIA's
published NVFP4 layout with a per-row fp32 second-level scale.  Pinned against:
  * hand-derived worked examples (tests/golden/nvfp4_worked_examples.json):
    every E2M1 tie, saturation, the sign of zero, a zero row, a block scale
    that rounds, a block whose scale underflows to zero;
  * E2M1 by brute force: the nearest of the 8 magnitudes, ties to the even
    code, over a dense grid and every midpoint;
  * the block scales against torch's float8_e4m3fn cast of the same quotient,
    and the codes against the brute-force rounding of torch's fp32 division;
  * the exact GEMM against numpy's fp64 matmul of the dequantized operands
    (exact at these sizes: every product is a multiple of 2^-20 and every
    partial sum stays below 2^33 of those units);
  * the round-trip bound |v - dec(code) e_b| <= e_b h below saturation, h
    half the E2M1 gap at that magnitude (1/4 up to 2, 1/2 up to 4, 1 up to 6).
A dropped block scale, nibbles in the wrong order, ties to away, or the block
maximum taken over the row would each fail the golden or torch cases."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_worked_examples.json")
MAGS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def brute_e2m1(r):
    """Nearest E2M1 code of each r (fp64 distances to all 8 magnitudes, ties
    to the even code, saturation above 6, sign kept)."""
    r = np.asarray(r, np.float64)
    a = np.minimum(np.abs(r), 6.0)
    d = np.abs(a[..., None] - MAGS)
    best = d.min(-1, keepdims=True)
    cand = d == best
    # among tied candidates take the even code (only two can tie)
    idx = np.where(cand & (np.arange(8) % 2 == 0), np.arange(8), 99).min(-1)
    idx = np.where(idx == 99, cand.argmax(-1), idx)
    return (np.signbit(r).astype(np.uint8) * 8 + idx).astype(np.uint8)


def test_golden_worked_examples():
    g = json.load(open(GOLDEN))
    V = np.array([r["v"] for r in g["rows"]], np.float32)
    q4, sb, gs = oracle.nvfp4_quant_rows(V)
    codes = oracle.nvfp4_unpack(q4)
    for i, r in enumerate(g["rows"]):
        np.testing.assert_array_equal(codes[i], np.array(r["codes"], np.uint8), err_msg=r["why"])
        np.testing.assert_array_equal(sb[i], np.array(r["block_scales"], np.uint8), err_msg=r["why"])
        assert gs[i] == np.float32(r["g"])
    # packing: value 2j in the low nibble of byte j
    assert q4[0, 0] == (codes[0, 0] | (codes[0, 1] << 4))


def test_e2m1_brute_force_and_midpoints():
    grid = np.concatenate([np.linspace(-8, 8, 20001), (MAGS[:-1] + MAGS[1:]) / 2, -(MAGS[:-1] + MAGS[1:]) / 2,
                           MAGS, -MAGS, [1e-30, -1e-30, 6.0001, 100.0, -100.0]]).astype(np.float32)
    np.testing.assert_array_equal(oracle.e2m1_encode(grid), brute_e2m1(grid))
    # decode: sign x magnitude table
    np.testing.assert_array_equal(oracle.e2m1_decode(np.arange(16)), np.concatenate([MAGS, -MAGS]))


@pytest.mark.parametrize("seed,K", [(0, 64), (1, 256), (2, 1040)])
def test_rows_against_torch_division_and_cast(seed, K):
    g = np.random.Generator(np.random.PCG64(seed))
    V = (g.standard_normal((24, K)) * np.exp(g.uniform(-6, 6, (24, 1)))).astype(np.float32)
    V[:, g.integers(0, K, 3)] *= 20.0  # outlier columns
    V[3, 16:32] = 0.0                   # a zero block
    V[5] = 0.0                          # a zero row
    q4, sb, gs = oracle.nvfp4_quant_rows(V)
    codes = oracle.nvfp4_unpack(q4)
    t = torch.from_numpy(V)
    A = t.abs().amax(1)
    gt = torch.where(A == 0, torch.ones_like(A), A / 2688.0)
    np.testing.assert_array_equal(gs, gt.numpy())
    d6 = 6.0 * gt
    ab = t.view(24, K // 16, 16).abs().amax(2)
    s_ref = (ab / d6[:, None]).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(sb, s_ref.view(torch.uint8).numpy())
    e = s_ref.to(torch.float32) * gt[:, None]                     # step per block, fp32
    q = t.view(24, K // 16, 16) / torch.where(e == 0, torch.ones_like(e), e)[:, :, None]
    ref = brute_e2m1(q.reshape(24, K).numpy())
    ref[(e == 0).repeat_interleave(16, 1).numpy()] = 0
    np.testing.assert_array_equal(codes, ref)
    # round trip below saturation: within half the grid gap at that magnitude
    qa = np.abs(q.reshape(24, K).numpy().astype(np.float64))
    eb = np.repeat(e.numpy(), 16, 1).astype(np.float64)
    val = oracle.e2m1_decode(codes) * eb
    h = np.where(qa <= 2, 0.25, np.where(qa <= 4, 0.5, 1.0))
    inside = qa <= 6.0
    assert np.all((np.abs(val - V) <= eb * (h + 1e-6))[inside])


def test_act_rows_apply_the_pre_scale_in_fp32():
    g = np.random.Generator(np.random.PCG64(5))
    X = torch.from_numpy(g.standard_normal((8, 128)).astype(np.float32)).to(torch.bfloat16)
    bits = X.view(torch.int16).numpy().view(np.uint16)
    v = X.float() * torch.tensor(1.5, dtype=torch.float32)
    a = oracle.nvfp4_quant_act(bits, 1.5)
    b = oracle.nvfp4_quant_rows(v.numpy())
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("M,N,K", [(5, 7, 64), (16, 24, 256), (3, 4, 2048)])
def test_gemm_exact_against_numpy(M, N, K):
    g = np.random.Generator(np.random.PCG64(M * N + K))
    x = oracle.nvfp4_quant_rows((g.standard_normal((M, K)) * 3).astype(np.float32))
    w = oracle.nvfp4_quant_rows((g.standard_normal((N, K)) * 0.02).astype(np.float32))
    acc = oracle.gemm_nvfp4(x[0], x[1], w[0], w[1], nthreads=2)

    def deq(q4, sb):
        return oracle.e2m1_decode(oracle.nvfp4_unpack(q4)) * np.repeat(oracle.e4m3_decode(sb), 16, 1)

    ref = deq(x[0], x[1]) @ deq(w[0], w[1]).T
    np.testing.assert_array_equal(acc, ref)
    # the epilogue with the row scales gives the dequantized product within bf16 rounding
    Y = oracle.bf16_decode(oracle.epilogue(acc, x[2], w[2]))
    full = ref * x[2][:, None].astype(np.float64) * w[2][None, :].astype(np.float64)
    assert np.max(np.abs(Y - full)) <= 2 ** -7 * np.max(np.abs(full)) + 1e-30
