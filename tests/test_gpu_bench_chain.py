"""Parity of the benchmark's own chains with the CPU oracle, at their full sizes.

Three configurations, each run through the fused quantize -> linear entry
points of the C ABI and replayed from the CUDA graph the benchmark captures
(the same weights, buffers and launch configuration):
  * the headline step's passes: the 32B-class chain (qkv 5120->7168, o_proj
    5120->5120, gate_up 5120->55296, down 27648->5120) at M = 256, 1024 and
    8192 on one weight set;
  * the 7B-class decode chain (qkv 3584->4608, o_proj 3584->3584, gate_up
    3584->37888, down 18944->3584) at M = 64 and 256;
  * the 7B-class chain at M = 512 and 4096;
the 7B batches alternating two weight sets (the second row-rotated).

Each stage is checked on a seeded sample of token rows and output channels,
with the oracle computing that stage from the GPU's own stage input (the
previous projection's bf16 output), so every stage is held to its own bar:
  * weight codes, scales and folded gains: bit-exact (per-channel quantization
    of the UAQ-folded W' = W / 1.5, gamma' = 1.5 gamma);
  * INT8 bf16 outputs of every stage: bit-exact, the RMSNorm stages given the
    kernel's mean of squares and the down stage given the kernel's SiLU*mul h
    (both from the standalone quantizer on the same rows; the fused entries
    give the same bits), against which the down GEMM's codes left in the
    scratch are also exact;
  * every stage's bf16 output within max-abs-rel 1e-2 of the oracle on its own
    mean of squares and h (FP8 outputs: always this bar, the fp32 accumulation
    order differs).
Two replays of the graph give the same bits.
"""
import os

import numpy as np
import pytest
import torch

import bench
import oracle
import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 1

CONFIGS = {"32b_headline": (bench.HEADLINE[0], bench.HEADLINE[1], 1),
           "7b_decode": (bench.DECODE_7B[0], bench.DECODE_7B[1], 2),
           "7b_chain": (bench.CHAIN_7B[0], bench.CHAIN_7B[1], 2)}


def bits(t):
    return synth.bf16_bits(t.contiguous().cpu())


def codes(t):
    return t.contiguous().cpu().view(torch.uint8).numpy()


def max_abs_rel(y_bits, ref_bits):
    y = oracle.bf16_decode(y_bits).astype(np.float64)
    ref = oracle.bf16_decode(ref_bits).astype(np.float64)
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-30))


def sample(g, n, k):
    """k sorted indices of range(n), always including the first and the last."""
    mid = g.choice(np.arange(1, n - 1), size=k - 2, replace=False)
    return np.sort(np.concatenate([[0, n - 1], mid]))


_weights = {}


def weights(model):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    q.load()
    if model not in _weights:
        _weights.clear()  # one model's fp32 masters at a time
        _weights[model] = bench.make_weights(model)
    return _weights[model]


@pytest.mark.parametrize("qt", [q.INT8, q.FP8_E4M3])
@pytest.mark.parametrize("cfg", list(CONFIGS))
def test_bench_chain_matches_oracle(cfg, qt):
    model, Ms, nsets = CONFIGS[cfg]
    hid, inter = bench.MODELS[model]["hidden"], bench.MODELS[model]["inter"]
    W, gammas = weights(model)
    oq = oracle.INT8 if qt == q.INT8 else oracle.FP8_E4M3
    layers = [bench.Layer(q, qt, model, W, gammas, rotate=r) for r in range(nsets)]
    bufs = [bench.Buffers(q, qt, model, M) for M in Ms]
    for B in bufs:
        B.x.copy_(synth.activations(bench.input_name(model, B.M), B.M, hid))

    def step():
        for i, B in enumerate(bufs):
            bench.chain(q, qt, layers[i % nsets], B)

    graph, launches = bench.graph_of(step, q)
    assert launches >= len(Ms) * len(bench.PROJ)  # at least one GEMM per projection and batch
    graph.replay()
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    first = {(B.M, name): bits(B.y[name]) for B in bufs for name in bench.PROJ}
    graph.replay()
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    for B in bufs:
        for name in bench.PROJ:
            np.testing.assert_array_equal(bits(B.y[name]), first[(B.M, name)])

    for i, B in enumerate(bufs):
        rot = i % nsets
        L = layers[rot]
        M = B.M
        g = np.random.Generator(np.random.PCG64(1000 + M + 7 * qt + 13 * hid))
        rows = sample(g, M, min(M, 24))
        ref = {}
        for name, K, N in bench.chain_shapes(model):
            cols = sample(g, N, 64)
            src = (cols - (N // 2 if rot else 0)) % N  # the rotated set's row n is W[n - N/2]
            gam = gammas.get(name)
            Wo, swo, gfo, _ = oracle.prepare_weights(W[name].numpy()[src], oq, s=bench.S_UAQ,
                                                     gamma=None if gam is None else gam.numpy())
            Wq, sw, gf = L.w[name]
            np.testing.assert_array_equal(codes(Wq)[cols], Wo)
            np.testing.assert_array_equal(sw.cpu().numpy()[cols], swo)
            if gfo is not None:
                np.testing.assert_array_equal(gf.cpu().numpy(), gfo)
            ref[name] = (cols, Wo, swo, gfo)

        def check(name, xq, sx, exact):
            cols, Wo, swo, _ = ref[name]
            Yo, _ = oracle.w8a8_linear(xq, sx, Wo, swo, oq, nthreads=NT)
            yd = bits(B.y[name])[np.ix_(rows, cols)]
            if exact and qt == q.INT8:
                np.testing.assert_array_equal(yd, Yo)
            assert max_abs_rel(yd, Yo) <= 1e-2, name

        ridx = torch.as_tensor(rows, device="cuda")

        def rms_stage(name, inp):
            """RMSNorm -> quant -> linear of the GPU's stage input: exact given the
            kernel's mean of squares, within 1e-2 on the oracle's own."""
            gfo = ref[name][3]
            _, _, ms = q.rmsnorm_quant(inp[ridx], torch.from_numpy(gfo).cuda(), qt, eps=bench.EPS, want_ms=True)
            xo, so, _, _ = oracle.rmsnorm_quant(bits(inp)[rows], gfo, oq, eps=bench.EPS, ms_given=ms.cpu().numpy())
            check(name, xo, so, exact=True)
            xo, so, _, _ = oracle.rmsnorm_quant(bits(inp)[rows], gfo, oq, eps=bench.EPS)
            check(name, xo, so, exact=False)

        # qkv: RMSNorm (gain gamma' = 1.5 gamma) -> quant -> linear, from the batch's input
        rms_stage("qkv", B.x)
        # o_proj: the q slice of the GPU's qkv output, quantized with pre-scale s
        xo, so = oracle.quant_act(bits(B.y["qkv"][:, :hid])[rows], oq, pre_scale=bench.S_UAQ)
        check("o_proj", xo, so, exact=True)
        # gate_up: RMSNorm -> quant of the GPU's o_proj output
        rms_stage("gate_up", B.y["o_proj"])
        # down: SiLU(gate) * up of the GPU's gate_up output -> quant (pre-scale s) -> linear.  The
        # codes the down GEMM consumed are still in the scratch; they equal the oracle's given the
        # kernel's h, and the GEMM + epilogue from them is exact
        gu = B.y["gate_up"]
        _, _, h = q.silu_mul_quant(gu[ridx], qt, pre_scale=bench.S_UAQ, want_h=True)
        hd = h.cpu().numpy()
        xo, so, ho = oracle.silu_mul_quant(bits(gu)[rows], oq, pre_scale=bench.S_UAQ)
        np.testing.assert_allclose(hd, ho, rtol=2e-6, atol=1e-35)
        check("down", xo, so, exact=False)
        xo, so, _ = oracle.silu_mul_quant(bits(gu)[rows], oq, pre_scale=bench.S_UAQ, h_given=hd)
        np.testing.assert_array_equal(codes(bench.dense(B.xq, M, inter))[rows], xo)
        np.testing.assert_array_equal(B.sx.cpu().numpy()[rows], so)
        check("down", xo, so, exact=True)
        torch.cuda.synchronize()
        q.qurl_check_device_status()
    del graph, bufs, layers
    torch.cuda.empty_cache()


def test_flip_probe_at_chain_sizes_matches_oracle():
    """The benchmark's weight-update probe on the 7B qkv projection (full size):
    the GPU's count equals the oracle's for both 8-bit types, both readings of
    the update and s in {1, 1.5}, and s = 1.5 flips more codes."""
    q.load()
    model = "7b"
    K, N = bench.MODELS[model]["shapes"]["qkv"]
    W = synth.weights(f"bench/{model}/qkv/W", N, K)
    dW = synth.update(f"bench/{model}/qkv/dW", N, K)
    for qt, oq in ((q.INT8, oracle.INT8), (q.FP8_E4M3, oracle.FP8_E4M3)):
        got = {}
        for s in (1.0, bench.S_UAQ):
            Wq0, _, _, Wp = q.prepare_weights(W.cuda(), qt, s=s, keep_scaled=True)
            Wo0, _, _, Wpo = oracle.prepare_weights(W.numpy(), oq, s=s)
            np.testing.assert_array_equal(Wp.cpu().numpy(), Wpo)
            for reading, f in (("sgd", s), ("same_size", 1.0)):
                upd = dW * f  # one fp32 product (exact for f = 1), then one fp32 sum: the same roundings
                Wn = Wp + upd.cuda()  # as the numpy update below
                Wq1, _, _, _ = q.prepare_weights(Wn, qt, s=1.0, keep_scaled=False)
                n_gpu = int(q.count_diff(Wq0, Wq1).item())
                Wo1, _, _, _ = oracle.prepare_weights(Wpo + dW.numpy() * np.float32(f), oq, s=1.0)
                assert n_gpu == oracle.count_diff(Wo0, Wo1), (qt, s, reading)
                got[(reading, s)] = n_gpu
        for reading in ("sgd", "same_size"):
            assert got[(reading, bench.S_UAQ)] > got[(reading, 1.0)], (qt, reading)
