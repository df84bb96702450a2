"""FP8 key/value cache quantization on the GPU (qurl_kv_cache_quant,
qurl_kv_cache_dequant) against the CPU oracle: codes and scales bit-exact,
read-back bit-exact, padding slots untouched, an out-of-range slot reported.
Layouts of the 7B- and 32B-class fused qkv outputs (q | k | v; 4 or 8 KV heads
of 128)."""
import numpy as np
import pytest
import torch

import oracle
import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu


def _fill(caches):
    for c in caches:
        c.view(torch.uint8).fill_(0xAA) if c.dtype == torch.float8_e4m3fn else c.fill_(-7.0)


def _np(c):
    return c.cpu().view(torch.uint8).numpy() if c.dtype == torch.float8_e4m3fn else c.cpu().numpy()


@pytest.mark.parametrize("model,M", [("7b", 300), ("32b", 77), ("32b", 8192)])
def test_kv_cache_quant_matches_oracle(model, M):
    hid, kvh, hd = (3584, 4, 128) if model == "7b" else (5120, 8, 128)
    N = hid + 2 * kvh * hd
    assert N == (synth.SHAPES_7B if model == "7b" else synth.SHAPES_32B)["qkv"][1]
    Y = synth.activations(f"gpu/kv/{model}/{M}", M, N)  # the qkv output (bf16), outlier columns included
    g = np.random.Generator(np.random.PCG64(M))
    S = M + 64
    slots = g.permutation(S)[:M].astype(np.int64)
    slots[::7] = -1  # padding tokens
    caches = q.kv_cache(S, kvh, hd)
    _fill(caches)
    q.qurl_kv_cache_quant(Y.cuda(), hid, kvh, hd, torch.from_numpy(slots).cuda(), *caches)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    ref = (np.full((S, kvh, hd), 0xAA, np.uint8), np.full((S, kvh), -7.0, np.float32),
           np.full((S, kvh, hd), 0xAA, np.uint8), np.full((S, kvh), -7.0, np.float32))
    rows = np.arange(M) if M <= 400 else np.sort(g.choice(M, 256, replace=False))
    oracle.kv_cache_quant(synth.bf16_bits(Y)[rows], hid, kvh, hd, slots[rows], ref)
    got = [_np(c) for c in caches]
    used = slots[rows][slots[rows] >= 0]
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a[used], b[used])
    untouched = np.setdiff1d(np.arange(S), slots[slots >= 0])
    assert np.all(got[0][untouched] == 0xAA) and np.all(got[3][untouched] == -7.0)
    # read-back of the written slots, against the oracle's
    rs = torch.from_numpy(used.copy()).cuda()
    for cache, scale, oc, os_ in ((caches[0], caches[1], ref[0], ref[1]), (caches[2], caches[3], ref[2], ref[3])):
        out = torch.empty((used.size, kvh * hd), dtype=torch.bfloat16, device="cuda")
        q.qurl_kv_cache_dequant(cache, scale, rs, out)
        torch.cuda.synchronize()
        q.qurl_check_device_status()
        np.testing.assert_array_equal(synth.bf16_bits(out.cpu()), oracle.kv_cache_dequant(oc, os_, used, kvh, hd))


def test_kv_cache_quant_strided_and_bad_slot():
    """The k | v columns read out of a wider row (the whole qkv output of a
    batch that also carries other columns), and a slot beyond the cache:
    nothing is written for that token and the status word reports it."""
    hid, kvh, hd, M = 64, 2, 16, 5
    wide = synth.activations("gpu/kv/strided", M, hid + 2 * kvh * hd + 24)
    Y = wide[:, : hid + 2 * kvh * hd]
    S = 4
    slots = np.array([3, 0, 9, -1, 1], np.int64)  # 9 >= S
    caches = q.kv_cache(S, kvh, hd)
    _fill(caches)
    q.qurl_kv_cache_quant(wide.cuda()[:, : hid + 2 * kvh * hd], hid, kvh, hd, torch.from_numpy(slots).cuda(), *caches)
    with pytest.raises(q.QurlError) as e:
        q.qurl_check_device_status()
    assert e.value.status == 1  # QURL_ERR_INVALID_ARG
    q.qurl_check_device_status()  # cleared
    ref = (np.full((S, kvh, hd), 0xAA, np.uint8), np.full((S, kvh), -7.0, np.float32),
           np.full((S, kvh, hd), 0xAA, np.uint8), np.full((S, kvh), -7.0, np.float32))
    ok = slots < S
    oracle.kv_cache_quant(synth.bf16_bits(Y.contiguous())[ok], hid, kvh, hd, slots[ok], ref)
    for a, b in zip((_np(c) for c in caches), ref):
        np.testing.assert_array_equal(a, b)  # slot 2 keeps the sentinel (its token was padding)
