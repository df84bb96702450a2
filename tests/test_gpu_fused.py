"""The fused entry points as one kernel at decode sizes (§ single-kernel
fusion): the decode GEMM's CTAs quantize the input rows between them (RMSNorm
-> quant, quant with the UAQ pre-scale, SiLU * up -> quant), hand over through
two counters in the workspace's last 256 bytes, then run the product.

Against the two-kernel path (the standalone quantizer, then qurl_w8a8_linear
on its codes with the same workspace): codes, scales and bf16 outputs
bit-identical, for INT8 (widened weights in TMEM) and FP8 (single-CTA and
CTA-pair decode kernels), K split or not.  The call launches one kernel (two
with a split-K reduction), leaves the counters zero, replays from a CUDA graph,
and a handoff that runs out is reported without faulting (Paper-Notes "QuRL",
sections 更新感知量化 (UAQ) and 系统集成与工程实现: the quantized rollout's
linear layers)."""
import time

import pytest
import torch

import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu
S = 1.5

# (M, N, K): decode shapes covering the kernels and split-K
SHAPES = [(64, 4608, 3584), (16, 512, 256), (200, 3584, 3584), (256, 37888, 3584), (256, 3584, 18944)]


@pytest.fixture(autouse=True)
def fused_decode_on():
    """These tests exercise the in-kernel quantizer wherever a plan allows it
    (mode 2), then restore the previous mode."""
    prev = q.qurl_set_fused_decode(2)
    yield
    q.qurl_set_fused_decode(prev)


def _bits(t):
    return t.contiguous().view(torch.int16).clone()


def _setup(qt, kind, M, N, K, tag):
    W = synth.weights(f"fused/{tag}/W", N, K).cuda()
    g = synth.gamma(f"fused/{tag}/g", K).cuda() if kind == "rms" else None
    Wq, sw, gf, _ = q.prepare_weights(W, qt, s=S, gamma=g, keep_scaled=False)
    cols = 2 * K if kind == "silu" else K
    X = synth.activations(f"fused/{tag}/X", M, cols).cuda()
    return X, Wq, sw, gf


def _fused(kind, X, gf, Wq, sw, qt, Y, Xq, sx, ws):
    if kind == "rms":
        q.qurl_rmsnorm_quant_linear(X, gf, 1e-6, Wq, sw, qt, Y, Xq, sx, ws)
    elif kind == "act":
        q.qurl_quant_act_linear(X, S, Wq, sw, qt, Y, Xq, sx, ws)
    else:
        q.qurl_silu_mul_quant_linear(X, S, Wq, sw, qt, Y, Xq, sx, ws)


def _two_kernel(kind, X, gf, Wq, sw, qt, ws):
    if kind == "rms":
        Xq, sx = q.rmsnorm_quant(X, gf, qt, eps=1e-6)
    elif kind == "act":
        Xq, sx = q.quant_act(X, qt, pre_scale=S)
    else:
        Xq, sx = q.silu_mul_quant(X, qt, pre_scale=S)
    return Xq, sx, q.linear(Xq, sx, Wq, sw, qt, ws)


@pytest.mark.parametrize("qt", [q.INT8, q.FP8_E4M3])
@pytest.mark.parametrize("kind", ["rms", "act", "silu"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fused_decode_is_one_kernel_and_matches_two_kernel_path(qt, kind, M, N, K):
    X, Wq, sw, gf = _setup(qt, kind, M, N, K, f"{kind}/{M}/{N}/{K}")
    ws = q.workspace(M, N, K, qt)
    Xq0, sx0, Y0 = _two_kernel(kind, X, gf, Wq, sw, qt, ws)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Xq = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    plan = q.plan(M, N, K, qt, torch.cuda.get_device_properties(0).multi_processor_count)
    for rep in range(2):  # the second call finds the counters the first one left
        n0 = q.qurl_kernel_launches()
        _fused(kind, X, gf, Wq, sw, qt, Y, Xq, sx, ws)
        launched = q.qurl_kernel_launches() - n0
        torch.cuda.synchronize()
        q.qurl_check_device_status()
        assert launched == (2 if plan["splits"] > 1 else 1), (rep, launched, plan)
        assert torch.equal(Xq.view(torch.uint8), Xq0.view(torch.uint8))
        assert torch.equal(sx, sx0)
        assert torch.equal(_bits(Y), _bits(Y0)), rep
        assert int(ws[-256:].count_nonzero()) == 0  # the handoff counters are left zero


@pytest.mark.parametrize("qt", [q.INT8, q.FP8_E4M3])
def test_fused_decode_replays_from_a_graph(qt):
    M, N, K = 64, 4608, 3584
    X, Wq, sw, gf = _setup(qt, "rms", M, N, K, "graph")
    ws = q.workspace(M, N, K, qt)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Xq = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    _, _, Y0 = _two_kernel("rms", X, gf, Wq, sw, qt, q.workspace(M, N, K, qt))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _fused("rms", X, gf, Wq, sw, qt, Y, Xq, sx, ws)  # first use outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _fused("rms", X, gf, Wq, sw, qt, Y, Xq, sx, ws)
    for _ in range(3):
        Y.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        q.qurl_check_device_status()
        assert torch.equal(_bits(Y), _bits(Y0))


@pytest.mark.parametrize("qt,M,N,K", [(q.INT8, 64, 4608, 3584), (q.FP8_E4M3, 64, 4608, 3584),
                                      (q.FP8_E4M3, 256, 37888, 3584)])
def test_fused_handoff_timeout_is_reported(qt, M, N, K):
    """The first CTA skips its arrival at the handoff (test hook): every CTA's
    bounded wait runs out, the kernel reports QURL_ERR_TIMEOUT and skips its
    main loop; once the counters are zeroed again the next call is exact."""
    X, Wq, sw, gf = _setup(qt, "act", M, N, K, f"timeout/{qt}/{M}")
    ws = q.workspace(M, N, K, qt)
    _, _, Y0 = _two_kernel("act", X, gf, Wq, sw, qt, q.workspace(M, N, K, qt))
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Xq = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
    sx = torch.empty(M, dtype=torch.float32, device="cuda")
    q.qurl_check_device_status()
    q.qurl_debug_inject_timeout()
    t0 = time.time()
    _fused("act", X, gf, Wq, sw, qt, Y, Xq, sx, ws)
    with pytest.raises(q.QurlError) as e:
        q.qurl_check_device_status()
    assert e.value.status == 6  # QURL_ERR_TIMEOUT
    assert time.time() - t0 < 30
    ws[-256:].zero_()
    _fused("act", X, gf, Wq, sw, qt, Y, Xq, sx, ws)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    assert torch.equal(_bits(Y), _bits(Y0))


@pytest.mark.parametrize("qt", [q.INT8, q.FP8_E4M3])
@pytest.mark.parametrize("kind", ["rms", "act", "silu"])
@pytest.mark.parametrize("M,N,K", [(64, 4608, 3584), (256, 3584, 18944)])
def test_fused_entry_switch_gives_identical_results(qt, kind, M, N, K):
    """The same fused entry with the quantizer inside the GEMM kernel and as
    its own kernel before it: one launch fewer in the first case, and codes,
    scales and bf16 outputs bit-identical."""
    X, Wq, sw, gf = _setup(qt, kind, M, N, K, f"switch/{kind}/{M}")
    ws = q.workspace(M, N, K, qt)
    res = {}
    for on in (True, False):
        q.qurl_set_fused_decode(2 if on else 0)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        Xq = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        n0 = q.qurl_kernel_launches()
        _fused(kind, X, gf, Wq, sw, qt, Y, Xq, sx, ws)
        res[on] = (q.qurl_kernel_launches() - n0, Xq.view(torch.uint8).clone(), sx.clone(), _bits(Y))
        torch.cuda.synchronize()
        q.qurl_check_device_status()
    assert res[False][0] == res[True][0] + 1
    for a, b in zip(res[True][1:], res[False][1:]):
        assert torch.equal(a, b)


def test_fused_decode_switch_rejects_other_values():
    lib = q.load()
    assert lib.qurl_set_fused_decode(3, None) == 1  # QURL_ERR_INVALID_ARG
    assert lib.qurl_set_fused_decode(-1, None) == 1


@pytest.mark.parametrize("qt", [q.INT8, q.FP8_E4M3])
@pytest.mark.parametrize("kind,M", [("rms", 64), ("rms", 256), ("act", 64), ("act", 256), ("silu", 64)])
def test_fused_decode_default_routing(qt, kind, M):
    """Mode 1 (the default) quantizes inside the GEMM only where that measured
    faster: RMSNorm rows for INT8 and for FP8 at M <= 64, per-token rows for
    INT8 at M <= 64, SiLU * up rows never.  Same outputs as mode 0."""
    N, K = 4608, 3584
    X, Wq, sw, gf = _setup(qt, kind, M, N, K, f"route/{kind}/{M}")
    ws = q.workspace(M, N, K, qt)
    plan = q.plan(M, N, K, qt, torch.cuda.get_device_properties(0).multi_processor_count)
    expect = {"rms": qt == q.INT8 or M <= 64, "act": qt == q.INT8 and M <= 64, "silu": False}[kind]
    got = {}
    for mode in (2, 1, 0):
        q.qurl_set_fused_decode(mode)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        Xq = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        n0 = q.qurl_kernel_launches()
        _fused(kind, X, gf, Wq, sw, qt, Y, Xq, sx, ws)
        got[mode] = (q.qurl_kernel_launches() - n0, _bits(Y))
        torch.cuda.synchronize()
        q.qurl_check_device_status()
    assert got[2][0] == got[0][0] - 1, plan  # the plan can take the quantizer
    assert got[1][0] == (got[2][0] if expect else got[0][0]), (plan, got)
    assert torch.equal(got[1][1], got[0][1]) and torch.equal(got[2][1], got[0][1])
