"""Pins of the oracle's ACR token objective (CPU, no GPU).

Source: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement Learning with
Quantized Rollout", section "方法详解 > 关键设计 > 自适应裁剪范围 (ACR)": the
decoupled-PPO objective of a quantized rollout,
    J = E~[ min(pi_prox / pi_behav, C) * min(R A, clip(R, 1 - eps, (1 + eps) / r) A) ],
with the truncated importance weight of TIS and ACR's upper bound (1 + eps) / r;
section "损失函数 / 训练策略": the GRPO/DAPO decoupled variant (a token-level mean).

What pins it, other than the formula itself:
  * hand-derived worked examples (tests/golden/acr_worked_examples.json);
  * without quantization (pi_behav = pi_prox) both modes reduce to the textbook
    PPO clipped surrogate, computed with torch ops, whose autograd gradient the
    oracle's per-token derivative must match;
  * the per-token derivative against central finite differences of the
    oracle's own per-token term, in both modes;
  * invariants the definition fixes: ACR caps every positive-advantage token's
    weighted ratio at exactly 1 + eps and reaches it where it clips; ACR and
    plain TIS agree on negative advantages wherever the clip range is not
    empty; padding slots never matter; the KL estimate of a constant log-ratio
    shift is that shift.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from w8a8_precision_gemm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "acr_worked_examples.json")


def _ev(expr):
    return float(eval(expr, {"__builtins__": {}}, {"exp": math.exp}))  # expressions of exp() and numbers only


def _arrays(toks):
    f = lambda k: np.array([t[k] for t in toks], np.float32)
    return f("logp"), f("logp_prox"), f("logp_behav"), f("adv"), np.array([t["mask"] for t in toks], np.uint8)


@pytest.mark.parametrize("mode", ["acr", "tis"])
def test_worked_examples(orc, mode):
    g = json.load(open(GOLDEN))
    toks = g["tokens"]
    lp, lpp, lpb, a, m = _arrays(toks)
    stats, term, dterm = orc.acr_objective(lp, lpp, lpb, a, m, eps=g["eps"], C=g["C"], adaptive=(mode == "acr"))
    for t, tok in enumerate(toks):
        exp_t, exp_d = _ev(tok[mode]["term"]), _ev(tok[mode]["dterm"])
        assert term[t] == pytest.approx(exp_t, rel=1e-12, abs=1e-300), (t, tok["why"])
        assert dterm[t] == pytest.approx(exp_d, rel=1e-12, abs=1e-300), (t, tok["why"])
    st = dict(zip(orc.ACR_STATS, stats))
    n = g["stats"]["n_valid"]
    assert st["n_valid"] == n
    assert st["objective"] == pytest.approx(sum(_ev(tok[mode]["term"]) for tok in toks) / n, rel=1e-12)
    assert st["clipped_frac"] == sum(tok[mode]["clipped"] for tok in toks) / n
    assert st["capped_frac"] == _ev(g["stats"]["capped_frac"])
    assert st["mean_tis_weight"] == pytest.approx(_ev(g["stats"]["mean_tis_weight"]), rel=1e-14)
    assert st["kl_behav_prox"] == pytest.approx(_ev(g["stats"]["kl_behav_prox"]), rel=1e-14)


def _ppo_clip_torch(lp, lpp, a, m, eps):
    """Textbook PPO clipped surrogate (mean over valid tokens) and its autograd
    gradient with respect to logp, in fp64 torch ops."""
    x = torch.tensor(lp, dtype=torch.float64, requires_grad=True)
    ratio = torch.exp(x - torch.tensor(lpp, dtype=torch.float64))
    A = torch.tensor(a, dtype=torch.float64)
    valid = torch.tensor(m, dtype=torch.bool)
    surr = torch.min(ratio * A, torch.clamp(ratio, 1 - eps, 1 + eps) * A)
    J = surr[valid].mean()
    J.backward()
    return float(J.detach()), x.grad.numpy()


@pytest.mark.parametrize("adaptive", [True, False])
def test_without_quantization_is_ppo_clip(orc, adaptive):
    r = synth.rollout("pin/acr/ppo", 16, 512)
    lpb = r["logp_prox"].copy()  # the rollout policy is the full-precision one: w = 1
    stats, term, dterm = orc.acr_objective(r["logp"], r["logp_prox"], lpb, r["adv"], r["mask"], eps=0.2,
                                           adaptive=adaptive)
    J, grad = _ppo_clip_torch(r["logp"], r["logp_prox"], r["adv"], r["mask"], 0.2)
    n = stats[1]
    assert n == r["mask"].sum()
    assert stats[0] == pytest.approx(J, rel=1e-12)
    np.testing.assert_allclose(dterm / n, grad, rtol=1e-12, atol=1e-18)
    assert stats[3] == 1.0 and stats[4] == 0.0 and stats[5] == 0.0
    assert 0.0 < stats[2] < 0.2  # some tokens clip, most do not


@pytest.mark.parametrize("adaptive", [True, False])
def test_derivative_against_finite_differences(orc, adaptive):
    r = synth.rollout("pin/acr/fd", 8, 256)
    eps, C = 0.2, 2.0
    lp = r["logp"]
    h = np.float32(2.0 ** -12)
    lp_hi, lp_lo = (lp + h).astype(np.float32), (lp - h).astype(np.float32)
    args = (r["logp_prox"], r["logp_behav"], r["adv"], r["mask"])
    _, t_hi, _ = orc.acr_objective(lp_hi, *args, eps=eps, C=C, adaptive=adaptive)
    _, t_lo, _ = orc.acr_objective(lp_lo, *args, eps=eps, C=C, adaptive=adaptive)
    _, _, dterm = orc.acr_objective(lp, *args, eps=eps, C=C, adaptive=adaptive)
    fd = (t_hi - t_lo) / (lp_hi.astype(np.float64) - lp_lo.astype(np.float64))
    # away from the kinks of min / clip (R within 1e-3 of either bound in log terms)
    lR = lp.astype(np.float64) - r["logp_prox"]
    w = np.minimum(np.exp(r["logp_prox"].astype(np.float64) - r["logp_behav"]), C)
    upper = (1 + eps) / w if adaptive else np.full_like(w, 1 + eps)
    smooth = (np.abs(lR - np.log(1 - eps)) > 1e-3) & (np.abs(lR - np.log(upper)) > 1e-3)
    valid = r["mask"].astype(bool) & smooth
    assert valid.sum() > 0.9 * r["mask"].sum()
    np.testing.assert_allclose(dterm[valid], fd[valid], rtol=1e-5, atol=1e-9)
    assert (dterm == 0).sum() > 0 and (dterm != 0).sum() > 0  # both branches are exercised


def test_acr_caps_the_weighted_ratio(orc):
    r = synth.rollout("pin/acr/cap", 16, 512)
    eps = 0.2
    _, term_acr, dterm_acr = orc.acr_objective(**r, eps=eps, adaptive=True)
    _, term_tis, _ = orc.acr_objective(**r, eps=eps, adaptive=False)
    pos = r["mask"].astype(bool) & (r["adv"] > 0)
    A = r["adv"].astype(np.float64)
    # ACR: w * min(R, c) <= 1 + eps for every positive-advantage token, with equality where it clips
    assert np.all(term_acr[pos] <= (1 + eps) * A[pos] * (1 + 1e-15))
    clipped = pos & (dterm_acr == 0)
    assert clipped.sum() > 0
    np.testing.assert_allclose(term_acr[clipped], (1 + eps) * A[clipped], rtol=1e-15)
    # plain TIS lets the weighted ratio reach w (1 + eps): above 1 + eps where w > 1
    w = np.minimum(np.exp(r["logp_prox"].astype(np.float64) - r["logp_behav"]), 2.0)
    assert np.any(term_tis[pos & (w > 1.05)] > (1 + eps) * A[pos & (w > 1.05)] * 1.01)


def test_acr_and_tis_agree_on_negative_advantages(orc):
    r = synth.rollout("pin/acr/neg", 16, 512)
    eps = 0.2
    _, ta, da = orc.acr_objective(**r, eps=eps, adaptive=True)
    _, tt, dt = orc.acr_objective(**r, eps=eps, adaptive=False)
    w = np.minimum(np.exp(r["logp_prox"].astype(np.float64) - r["logp_behav"]), 2.0)
    # the lower bound decides negative advantages; the two modes share it while the adaptive
    # range [1 - eps, (1 + eps) / w] is not empty
    neg = r["mask"].astype(bool) & (r["adv"] < 0) & (w <= (1 + eps) / (1 - eps))
    assert neg.sum() > 1000
    np.testing.assert_array_equal(ta[neg], tt[neg])
    np.testing.assert_array_equal(da[neg], dt[neg])
    pos = r["mask"].astype(bool) & (r["adv"] > 0)
    assert np.any(ta[pos] != tt[pos])  # and differ on positive ones


def test_padding_and_empty_batches(orc):
    r = synth.rollout("pin/acr/pad", 8, 256)
    s0, t0, d0 = orc.acr_objective(**r)
    pad = r["mask"] == 0
    assert pad.sum() > 0
    junk = {k: v.copy() for k, v in r.items()}
    for k in ("logp", "logp_prox", "logp_behav", "adv"):
        junk[k][pad] = np.float32("nan")
    s1, t1, d1 = orc.acr_objective(**junk)
    np.testing.assert_array_equal(s0, s1)
    np.testing.assert_array_equal(t0, t1)
    np.testing.assert_array_equal(d0, d1)
    assert np.all(t1[pad] == 0) and np.all(d1[pad] == 0)
    empty = {k: v.copy() for k, v in r.items()}
    empty["mask"][:] = 0
    s2, t2, d2 = orc.acr_objective(**empty)
    assert np.all(s2 == 0) and np.all(t2 == 0) and np.all(d2 == 0)
    s3, _, _ = orc.acr_objective(*(r[k][:0] for k in ("logp", "logp_prox", "logp_behav", "adv", "mask")))
    assert np.all(s3 == 0)


def test_kl_estimate_and_cap_of_a_constant_shift(orc):
    T = 1000
    lpp = np.full(T, -1.0, np.float32)
    lpb = np.full(T, -1.5, np.float32)  # log(pi_behav / pi_prox) = -0.5 on every token
    args = (lpp, lpp, lpb, np.ones(T, np.float32), np.ones(T, np.uint8))
    st, _, _ = orc.acr_objective(*args, C=2.0)
    assert st[5] == -0.5 and st[4] == 0.0 and st[3] == pytest.approx(math.exp(0.5), rel=1e-15)
    st, _, _ = orc.acr_objective(*args, C=1.5)  # e^0.5 = 1.65 > 1.5: every weight capped
    assert st[4] == 1.0 and st[3] == 1.5
