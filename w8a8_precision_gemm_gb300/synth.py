"""Seeded synthetic inputs for the W8A8 linear layer.

Random numbers only -- this module holds none of the method's arithmetic (no
scaling, quantization, normalisation or matmul), so the CUDA path and the CPU
oracle can both be fed from it without sharing any of the computation.

Distributions (the workloads of the QuRL rollout actor's projections):
  * activations X ~ N(0, 1), with round(1% of K) input channels (at least one;
    4 for K = 256) multiplied by 20 -- the outlier channels of LLM activations;
    cast to bf16 (the activation dtype of the layer);
  * weights W ~ N(0, 0.02) in fp32 (the training master copy);
  * RMSNorm gain gamma ~ 1 + N(0, 0.1) in fp32;
  * weight update dW ~ N(0, 1e-7) in fp32 (the size of one RL update: lr ~1e-6
    times gradients ~0.1-1);
  * rollout token log-probabilities for the ACR objective (``rollout``).
Standard deviations, not variances.  Generator: numpy PCG64 seeded per tensor
from a stable name, so every run and every machine draws the same numbers.
"""
from __future__ import annotations

import zlib

import numpy as np
import torch


def seed_of(name: str, base: int = 20260215) -> int:
    """Stable 64-bit seed for a named tensor."""
    return (base << 32) ^ zlib.crc32(name.encode())


def rng(name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed_of(name)))


def n_outliers(K: int) -> int:
    if K == 256:
        return 4
    return max(1, int(round(0.01 * K)))


def activations(name: str, M: int, K: int, outlier_gain: float = 20.0, n_out: int | None = None) -> torch.Tensor:
    """bf16 [M, K] on the CPU: N(0,1) with seeded outlier channels x outlier_gain."""
    g = rng(name)
    x = g.standard_normal((M, K), dtype=np.float32)
    n_out = n_outliers(K) if n_out is None else n_out
    if n_out > 0:
        idx = g.permutation(K)[:n_out]
        x[:, idx] *= np.float32(outlier_gain)
    return torch.from_numpy(x).to(torch.bfloat16)


def weights(name: str, N: int, K: int, std: float = 0.02) -> torch.Tensor:
    """fp32 [N, K] on the CPU, N(0, std)."""
    g = rng(name)
    return torch.from_numpy(g.standard_normal((N, K), dtype=np.float32) * np.float32(std))


def gamma(name: str, K: int, std: float = 0.1) -> torch.Tensor:
    """fp32 [K] RMSNorm gain 1 + N(0, std)."""
    g = rng(name)
    return torch.from_numpy(np.float32(1.0) + g.standard_normal(K, dtype=np.float32) * np.float32(std))


def update(name: str, N: int, K: int, std: float = 1e-7) -> torch.Tensor:
    """fp32 [N, K] weight update N(0, std)."""
    return weights(name, N, K, std)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor (the oracle's input format)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# Projection shapes of the two model classes (K = in-features, N = out-features),
# fused qkv rows ordered q|k|v and fused gate_up rows ordered gate|up.
SHAPES_7B = {
    "qkv": (3584, 4608),
    "o_proj": (3584, 3584),
    "gate_up": (3584, 37888),
    "down": (18944, 3584),
}
SHAPES_32B = {
    "qkv": (5120, 7168),
    "o_proj": (5120, 5120),
    "gate_up": (5120, 55296),
    "down": (27648, 5120),
}


def rollout(name: str, n_seq: int, max_len: int, kl: float = 0.025, step_std: float = 0.1,
            mean_nll: float = 0.3) -> dict:
    """One mini-batch of quantized rollouts, token slots flattened response by
    response ([n_seq * max_len]; slots past a response's length are padding):
      * logp_prox:  the full-precision old actor's log-probability of each
        sampled token, -Exponential(mean_nll) (mostly confident tokens, a tail);
      * logp_behav: the quantized actor that sampled the tokens, logp_prox +
        N(kl, sqrt(2 kl)) -- for a small perturbation the log-ratio of the
        sampled token has mean KL(behav || prox) and variance 2 KL; kl = 0.025
        is the late-training divergence the pages report (0.002 early);
      * logp:       the policy being trained, a few updates on, logp_prox +
        N(0, step_std);
      * adv:        one N(0, 1) advantage per response (group-normalised
        rewards), repeated over its tokens;
      * mask:       1 on the first len_i slots of response i, len_i uniform in
        [max_len / 8, max_len].
    float32 arrays and a uint8 mask, on the CPU."""
    g = rng(name)
    T = n_seq * max_len
    lpp = -g.exponential(mean_nll, size=T).astype(np.float32)
    lpb = (lpp + g.normal(kl, np.sqrt(2.0 * kl), size=T)).astype(np.float32)
    lp = (lpp + g.normal(0.0, step_std, size=T)).astype(np.float32)
    adv = np.repeat(g.standard_normal(n_seq).astype(np.float32), max_len)
    lens = g.integers(max(1, max_len // 8), max_len + 1, size=n_seq)
    mask = (np.arange(max_len)[None, :] < lens[:, None]).astype(np.uint8).reshape(T)
    return {"logp": lp, "logp_prox": lpp, "logp_behav": lpb, "adv": adv, "mask": mask}
