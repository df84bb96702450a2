"""Pins of the oracle's FP8 key/value cache quantization (CPU only).

The oracle applies the per-token FP8 rule to each attention head's key and
value vectors of the fused qkv output and scatters the codes into a paged
cache by slot (Paper-Notes "QuRL", section 局限与展望: FP8 KV-cache
quantization; the granularity is a reading, see the oracle).  Pinned against:
  * hand-derived worked examples (tests/golden/kv_cache_worked_examples.json):
    ties to even in the normal and subnormal ranges, saturation, zero heads,
    scale 2, a padding token that must write nothing;
  * torch's own fp32 division and float8_e4m3fn cast, head by head, on
    random data with outlier columns and shuffled slots;
  * the e4m3 round-trip bound |x - dec(code) scale| <= scale ulp(code) / 2;
  * the cache read-back against torch's float8 decode, product and bf16 cast.
A slip in the slicing (k and v swapped, a head offset by one, q not skipped)
or the scatter (slot ignored, padding written) fails the golden and torch
cases."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from w8a8_precision_gemm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_cache_worked_examples.json")


def _bits(x):
    return synth.bf16_bits(torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16))


def _caches(S, H, D, fill=0xAA, sfill=-7.0):
    return (np.full((S, H, D), fill, np.uint8), np.full((S, H), sfill, np.float32),
            np.full((S, H, D), fill, np.uint8), np.full((S, H), sfill, np.float32))


def test_golden_worked_examples(orc):
    g = json.load(open(GOLDEN))
    q_dim, H, D = 16, 2, 16
    rows, slots = [], []
    for t in g["tokens"]:
        q = np.zeros(q_dim, np.float32)
        rows.append(np.concatenate([q] + [np.asarray(h, np.float32) for h in t["k"]] +
                                   [np.asarray(h, np.float32) for h in t["v"]]))
        slots.append(t["slot"])
    X = _bits(np.stack(rows))
    assert np.array_equal(oracle.bf16_decode(X), np.stack(rows))  # every value is a bf16
    kc, ks, vc, vs = oracle.kv_cache_quant(X, q_dim, H, D, np.array(slots), _caches(3, H, D))
    for t in g["tokens"]:
        s = t["slot"]
        if s < 0:
            continue
        np.testing.assert_array_equal(kc[s], np.array(t["k_codes"], np.uint8))
        np.testing.assert_array_equal(vc[s], np.array(t["v_codes"], np.uint8))
        np.testing.assert_array_equal(ks[s], np.array(t["k_scales"], np.float32))
        np.testing.assert_array_equal(vs[s], np.array(t["v_scales"], np.float32))
    # the padding token's slot (1) is untouched
    assert np.all(kc[1] == 0xAA) and np.all(vc[1] == 0xAA) and np.all(ks[1] == -7.0) and np.all(vs[1] == -7.0)


@pytest.mark.parametrize("M,q_dim,H,D", [(37, 64, 4, 128), (5, 0, 1, 16), (9, 5120, 8, 128)])
def test_matches_torch_per_head(orc, M, q_dim, H, D):
    g = np.random.Generator(np.random.PCG64(M * 7 + H))
    ld = q_dim + 2 * H * D + 8  # a wider row stride than the three parts
    X = g.standard_normal((M, ld)).astype(np.float32)
    X[:, q_dim + 3] *= 40  # an outlier column in key head 0
    X[0, q_dim:q_dim + D] = 0  # a zero head
    Xb = _bits(X)
    S = M + 3
    slots = g.permutation(S)[:M].astype(np.int64)
    slots[M // 2] = -1
    kc, ks, vc, vs = oracle.kv_cache_quant(Xb, q_dim, H, D, slots, _caches(S, H, D))
    xt = torch.from_numpy(oracle.bf16_decode(Xb).copy())
    for m in range(M):
        s = slots[m]
        for part, (codes, scales) in enumerate(((kc, ks), (vc, vs))):
            v = xt[m, q_dim + part * H * D: q_dim + (part + 1) * H * D].reshape(H, D)
            if s < 0:
                continue
            amax = v.abs().amax(1)
            scale = torch.where(amax == 0, torch.ones_like(amax), amax / 448.0)
            ref = (v / scale[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(codes[s], ref)
            np.testing.assert_array_equal(scales[s], scale.numpy())
    for s in set(range(S)) - set(int(x) for x in slots if x >= 0):
        assert np.all(kc[s] == 0xAA) and np.all(vs[s] == -7.0)


def test_round_trip_bound_and_readback(orc):
    g = np.random.Generator(np.random.PCG64(11))
    M, q_dim, H, D = 64, 128, 4, 128
    X = (g.standard_normal((M, q_dim + 2 * H * D)) * np.exp(g.uniform(-3, 3, (M, 1)))).astype(np.float32)
    Xb = _bits(X)
    slots = np.arange(M, dtype=np.int64)[::-1].copy()
    kc, ks, vc, vs = oracle.kv_cache_quant(Xb, q_dim, H, D, slots, _caches(M, H, D))
    x = oracle.bf16_decode(Xb).astype(np.float64)
    for part, (codes, scales) in enumerate(((kc, ks), (vc, vs))):
        v = x[:, q_dim + part * H * D: q_dim + (part + 1) * H * D].reshape(M, H, D)[np.argsort(slots)]
        dec = oracle.e4m3_decode(codes)
        # half an e4m3 ulp of the code's binade (subnormal spacing 2^-9 below 2^-6), in units of the scale
        mag = np.maximum(np.abs(dec), 2.0 ** -6)
        ulp = 2.0 ** (np.floor(np.log2(mag)) - 3)
        err = np.abs(v - dec * scales[..., None].astype(np.float64))
        assert np.all(err <= scales[..., None] * ulp / 2 * (1 + 2 ** -20) + 1e-45)
        # read back: torch's float8 decode, one fp32 product, one bf16 rounding
        back = oracle.kv_cache_dequant(codes, scales, np.arange(M), H, D)
        t = (torch.from_numpy(codes.reshape(M, H * D)).view(torch.float8_e4m3fn).float() *
             torch.from_numpy(np.repeat(scales, D, axis=1)))
        np.testing.assert_array_equal(back, synth.bf16_bits(t.to(torch.bfloat16)))
