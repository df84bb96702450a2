"""Parity of the ACR token objective kernel (through the C ABI) with the CPU oracle.

The objective: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement Learning
with Quantized Rollout", section "方法详解 > 关键设计 > 自适应裁剪范围 (ACR)"
(decoupled PPO with the truncated weight min(pi_prox / pi_behav, C) and the
clipping range [1 - eps, (1 + eps) / r]) and section "损失函数 / 训练策略" (a
token-level mean).

Tolerances, from the arithmetic: per token the kernel evaluates two expf (at
most 2 ulp each) and a few rounded products with no cancellation, so term and
dterm are within rel 2e-6 of the fp64 oracle; the sums run in fp32 per thread
(a few dozen tokens) and fp64 beyond, so the objective and the means are within
1e-5 of the sum of magnitudes.  A token whose oracle ratio lies within 2e-5 of
a clip bound or of the cap C may fall on either side in fp32: both branches are
right there, so those tokens are excluded from the per-token comparison and
bound the difference of the clipped / capped counts.  The valid-token count is
exact.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import synth

pytestmark = pytest.mark.gpu
KEYS = ("logp", "logp_prox", "logp_behav", "adv", "mask")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    q.load()
    yield
    q.qurl_check_device_status()


def _dev(r):
    return {k: torch.from_numpy(np.ascontiguousarray(r[k])).cuda() for k in KEYS}


def _run(r, **kw):
    d = _dev(r)
    stats, dterm, term = q.acr_objective(*(d[k] for k in KEYS), want_term=True, **kw)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    return stats.cpu().numpy(), dterm.cpu().numpy(), term.cpu().numpy()


def _ambiguous(r, eps, C, adaptive, rel=2e-5):
    lpp = r["logp_prox"].astype(np.float64)
    ratio = np.exp(lpp - r["logp_behav"])
    w = np.minimum(ratio, C)
    R = np.exp(r["logp"] - lpp)
    upper = (1 + eps) / w if adaptive else np.full_like(w, 1 + eps)
    near = lambda x, b: np.abs(x / b - 1) < rel
    return r["mask"].astype(bool) & (near(R, 1 - eps) | near(R, upper) | near(ratio, C))


def _check(r, eps=0.2, C=2.0, adaptive=True):
    sd, dd, td = _run(r, eps=eps, C=C, adaptive=adaptive)
    so, to, do = oracle.acr_objective(*(r[k] for k in KEYS), eps=eps, C=C, adaptive=adaptive)
    valid = r["mask"].astype(bool)
    amb = _ambiguous(r, eps, C, adaptive)
    n = so[1]
    assert sd[1] == n
    assert np.all(td[~valid] == 0) and np.all(dd[~valid] == 0)
    ok = valid & ~amb
    np.testing.assert_allclose(td[ok], to[ok], rtol=2e-6, atol=0)
    np.testing.assert_allclose(dd[ok], do[ok], rtol=2e-6, atol=0)
    np.testing.assert_array_equal(dd[ok] == 0, do[ok] == 0)  # the same branch wherever it is decided
    if n:
        tol = 1e-5 * np.abs(to).sum() / n
        assert abs(sd[0] - so[0]) <= tol, (sd[0], so[0], tol)
        assert abs(sd[2] - so[2]) * n <= amb.sum()
        assert abs(sd[4] - so[4]) * n <= amb.sum()
        assert sd[3] == pytest.approx(so[3], rel=1e-5)
        dkl = np.abs(r["logp_behav"].astype(np.float64) - r["logp_prox"])[valid].sum() / n
        assert abs(sd[5] - so[5]) <= 1e-5 * dkl
    else:
        assert np.all(sd == 0)
    return sd, dd, td, amb


@pytest.mark.parametrize("adaptive", [True, False])
@pytest.mark.parametrize("n_seq,max_len", [(64, 1024), (37, 999), (1, 3), (3, 1), (152 * 4, 2048)])
def test_objective_matches_oracle(adaptive, n_seq, max_len):
    """Several CTAs' strides, a ragged T mod 4 tail (36963 = 4 * 9240 + 3),
    tails alone (T = 3), and more 4-token groups than one pass of the grid."""
    r = synth.rollout(f"gpu/acr/{n_seq}/{max_len}", n_seq, max_len)
    sd, dd, _, amb = _check(r, adaptive=adaptive)
    assert amb.sum() <= max(2, 1e-3 * r["mask"].sum())


def test_worked_examples_on_the_gpu():
    """The hand-derived cases (tests/golden/acr_worked_examples.json) on the kernel."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "acr_worked_examples.json")))
    toks = g["tokens"]
    r = {k: np.array([t[k] for t in toks], np.uint8 if k == "mask" else np.float32) for k in KEYS}
    for mode in ("acr", "tis"):
        sd, dd, td = _run(r, eps=g["eps"], C=g["C"], adaptive=(mode == "acr"))
        ev = lambda e: float(eval(e, {"__builtins__": {}}, {"exp": math.exp}))
        for t, tok in enumerate(toks):
            assert td[t] == pytest.approx(ev(tok[mode]["term"]), rel=2e-6, abs=0), (mode, t, tok["why"])
            assert dd[t] == pytest.approx(ev(tok[mode]["dterm"]), rel=2e-6, abs=0), (mode, t, tok["why"])
        assert sd[1] == g["stats"]["n_valid"]
        assert round(sd[2] * sd[1]) == sum(tok[mode]["clipped"] for tok in toks)


def test_empty_masked_and_padding_nan():
    r = synth.rollout("gpu/acr/pad", 16, 500)
    clean = _run(r)
    junk = {k: v.copy() for k, v in r.items()}
    pad = r["mask"] == 0
    for k in ("logp", "logp_prox", "logp_behav", "adv"):
        junk[k][pad] = np.float32("nan")
    dirty = _run(junk)
    for a, b in zip(clean, dirty):
        np.testing.assert_array_equal(a, b)  # padding values never reach a result
    allpad = {k: v.copy() for k, v in r.items()}
    allpad["mask"][:] = 0
    sd, dd, td = _run(allpad)
    assert np.all(sd == 0) and np.all(dd == 0) and np.all(td == 0)
    empty = {k: v[:0] for k, v in r.items()}
    sd, dd, td = _run(empty)
    assert np.all(sd == 0) and dd.size == 0 and td.size == 0


def test_repeatable_and_optional_outputs():
    """One kernel a call; a reused workspace (its ticket counter is left at
    zero) and fresh ones give the same bits; the optional outputs change
    nothing else."""
    r = synth.rollout("gpu/acr/rep", 128, 1024)
    d = _dev(r)
    args = [d[k] for k in KEYS]
    ws = q.acr_workspace()
    n0 = q.qurl_kernel_launches()
    a = q.acr_objective(*args, want_term=True, workspace=ws)
    b = q.acr_objective(*args, want_term=True, workspace=ws)
    c = q.acr_objective(*args, want_term=False, want_dterm=False)
    e = q.acr_objective(*[x[: 4 * 999 + 1] for x in args], workspace=ws)  # another grid on the same workspace
    f = q.acr_objective(*args, want_term=True, workspace=ws)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    assert q.qurl_kernel_launches() - n0 == 5
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert torch.equal(a[0], c[0]) and c[1] is None and c[2] is None
    assert torch.equal(a[0], f[0]) and torch.equal(a[1], f[1])
    assert int(ws[-256:].count_nonzero()) == 0  # the ticket counter is back at zero
    so, _, _ = oracle.acr_objective(*(r[k][: 4 * 999 + 1] for k in KEYS))
    assert e[0][1].item() == so[1]


def test_full_size_minibatch():
    """The benchmark's mini-batch: 512 responses x 8192 token slots (4.2 M)."""
    r = synth.rollout("bench/acr/0", 512, 8192)
    sd, _, _, amb = _check(r, adaptive=True)
    assert sd[1] > 0.5 * 512 * 8192 * 0.5
