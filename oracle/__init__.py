"""CPU oracle of the QuRL W8A8 linear layer -- TEST INFRASTRUCTURE ONLY.

Plain C (``qurl_oracle.c``) behind ctypes, numpy in and out.  Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package; the product library never links or calls it, and this package
imports nothing from the product package.

What each function computes, and which passage of the source pages it restates,
is written in ``qurl_oracle.c``.  Pages: Paper-Notes ICLR2026, "QuRL: Efficient
Reinforcement Learning with Quantized Rollout" -- sections "更新感知量化 (UAQ)"
(invariant scaling), "损失函数 / 训练策略" (per-channel / per-token INT8 or FP8,
s = 1.5; the GRPO/DAPO decoupled objective), "系统集成与工程实现" (one-time UAQ
preprocessing, INT8/FP8 matmul) and "自适应裁剪范围 (ACR)" (the token objective
of the quantized rollout).

Parity pinning: every function here is pinned by tests under ``tests/`` that
check it against library routines (torch CPU casts and rounding, numpy integer
and fp64 matmul), closed forms and invariants -- see test_oracle_pins.py and
test_oracle_acr.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

INT8 = 0
FP8_E4M3 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qurl_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (no fast-math, no FMA
    contraction, so x86-64 and aarch64 agree bit for bit)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["cc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i, f, z = ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [f]
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_bf16_encode.restype = ctypes.c_uint16
            L.orc_bf16_encode.argtypes = [f]
            L.orc_e4m3_encode_array.argtypes = [P, z, P]
            L.orc_bf16_encode_array.argtypes = [P, z, P]
            L.orc_quant_rows_f32.argtypes = [P, i, i, i, i, P, P]
            L.orc_quant_act.argtypes = [P, i, i, i, f, i, P, P]
            L.orc_prepare_weights.argtypes = [P, i, i, i, P, f, i, P, P, P, P]
            L.orc_rms_ms.argtypes = [P, i, i, i, P]
            L.orc_rmsnorm_quant.argtypes = [P, i, i, i, P, f, P, i, P, P, P, P]
            L.orc_silu_mul_quant.argtypes = [P, i, i, i, f, P, i, P, P, P]
            L.orc_gemm_i8.argtypes = [P, P, i, i, i, P, i]
            L.orc_gemm_fp8.argtypes = [P, P, i, i, i, P, i]
            L.orc_epilogue_i32.argtypes = [P, P, P, i, i, P, i]
            L.orc_epilogue_f64.argtypes = [P, P, P, i, i, P, i]
            L.orc_count_diff.restype = ctypes.c_uint64
            L.orc_count_diff.argtypes = [P, P, z]
            L.orc_acr_objective.argtypes = [P, P, P, P, P, ctypes.c_int64, ctypes.c_double, ctypes.c_double, i,
                                            P, P, P]
            L.orc_kv_cache_quant.argtypes = [P, i, i, i, i, i, P, P, P, P, P]
            L.orc_kv_cache_dequant.argtypes = [P, P, P, i, i, i, P]
            L.orc_e2m1_encode.restype = ctypes.c_uint8
            L.orc_e2m1_encode.argtypes = [f]
            L.orc_e2m1_decode.restype = ctypes.c_double
            L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            L.orc_nvfp4_quant_rows_f32.argtypes = [P, i, i, i, P, P, P]
            L.orc_nvfp4_quant_act.argtypes = [P, i, i, i, f, P, P, P]
            L.orc_gemm_nvfp4.argtypes = [P, P, P, P, i, i, i, P, i]
            for name in ("orc_quant_rows_f32", "orc_quant_act", "orc_prepare_weights", "orc_rmsnorm_quant",
                         "orc_silu_mul_quant", "orc_gemm_i8", "orc_gemm_fp8", "orc_acr_objective",
                         "orc_kv_cache_quant", "orc_kv_cache_dequant", "orc_nvfp4_quant_rows_f32",
                         "orc_nvfp4_quant_act", "orc_gemm_nvfp4"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


# ---------------------------------------------------------------- formats

def e4m3_encode(v) -> np.ndarray:
    """fp32 -> e4m3 code bytes (RNE, saturating to +-448, sign kept)."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(_p(v), v.size, _p(out))
    return out


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 code bytes -> exact float64 values."""
    L = lib()
    table = np.array([L.orc_e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def bf16_encode(v) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_encode_array(_p(v), v.size, _p(out))
    return out


def bf16_decode(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- method steps

def quant_rows(V, qtype):
    """Per-row symmetric absmax quantization of fp32 rows -> (codes u8, scales f32)."""
    V = _c(V, np.float32)
    M, K = V.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty(M, np.float32)
    _check(lib().orc_quant_rows_f32(_p(V), M, K, K, qtype, _p(q), _p(s)), "quant_rows")
    return q, s


def quant_act(X_bits, qtype, pre_scale=1.0):
    """Per-token quantization of bf16 activations (uint16 bits [M, K])."""
    X = _c(X_bits, np.uint16)
    M, K = X.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty(M, np.float32)
    _check(lib().orc_quant_act(_p(X), M, K, K, float(pre_scale), qtype, _p(q), _p(s)), "quant_act")
    return q, s


def prepare_weights(W, qtype, s=1.5, gamma=None):
    """UAQ fold W' = W/s (column-wise), gamma' = gamma*s, then per-channel
    quantization of W'.  Returns (Wq u8 [N,K], sw f32 [N], gamma' or None, W' f32)."""
    W = _c(W, np.float32)
    N, K = W.shape
    Wq = np.empty((N, K), np.uint8)
    sw = np.empty(N, np.float32)
    Ws = np.empty((N, K), np.float32)
    g = None if gamma is None else _c(gamma, np.float32)
    gf = None if gamma is None else np.empty(K, np.float32)
    _check(lib().orc_prepare_weights(_p(W), N, K, K, _p(g), float(s), qtype, _p(Wq), _p(sw), _p(gf), _p(Ws)),
           "prepare_weights")
    return Wq, sw, gf, Ws


def rms_ms(X_bits) -> np.ndarray:
    X = _c(X_bits, np.uint16)
    M, K = X.shape
    ms = np.empty(M, np.float64)
    lib().orc_rms_ms(_p(X), M, K, K, _p(ms))
    return ms


def rmsnorm_quant(X_bits, gamma_folded, qtype, eps=1e-6, ms_given=None):
    """RMSNorm(gain gamma') -> per-token quantization.
    Returns (codes, scales, ms used (f32), v (f32 normalised rows))."""
    X = _c(X_bits, np.uint16)
    M, K = X.shape
    g = _c(gamma_folded, np.float32)
    msg = None if ms_given is None else _c(ms_given, np.float32)
    q = np.empty((M, K), np.uint8)
    s = np.empty(M, np.float32)
    mso = np.empty(M, np.float32)
    v = np.empty((M, K), np.float32)
    _check(lib().orc_rmsnorm_quant(_p(X), M, K, K, _p(g), float(eps), _p(msg), qtype, _p(q), _p(s), _p(mso),
                                   _p(v)), "rmsnorm_quant")
    return q, s, mso, v


def silu_mul_quant(GU_bits, qtype, pre_scale=1.0, h_given=None):
    """h = silu(gate) * up over GU [M, 2I] (gate first), v = h * pre_scale, then
    per-token quantization.  Returns (codes, scales, h)."""
    GU = _c(GU_bits, np.uint16)
    M, I2 = GU.shape
    I = I2 // 2
    hg = None if h_given is None else _c(h_given, np.float32)
    q = np.empty((M, I), np.uint8)
    s = np.empty(M, np.float32)
    h = np.empty((M, I), np.float32)
    _check(lib().orc_silu_mul_quant(_p(GU), M, I, I2, float(pre_scale), _p(hg), qtype, _p(q), _p(s), _p(h)),
           "silu_mul_quant")
    return q, s, h


def kv_cache_quant(QKV_bits, q_dim, kv_heads, head_dim, slot_mapping, caches):
    """FP8 quantization of the keys and values of the qkv output QKV (uint16
    bf16 bits [M, >= q_dim + 2 kv_heads head_dim]) per token and head, into
    slot slot_mapping[m] of the caches (kc u8 [S, kv_heads, head_dim], ks f32
    [S, kv_heads], vc, vs), which are updated in place; negative slots skip."""
    X = _c(QKV_bits, np.uint16)
    M, ldq = X.shape
    slots = _c(slot_mapping, np.int64)
    kc, ks, vc, vs = caches
    for a in caches:
        assert a.flags["C_CONTIGUOUS"]
    _check(lib().orc_kv_cache_quant(_p(X), M, ldq, q_dim, kv_heads, head_dim, _p(slots), _p(kc), _p(ks), _p(vc),
                                    _p(vs)), "kv_cache_quant")
    return caches


def kv_cache_dequant(cache, scale, slots, kv_heads, head_dim):
    """bf16 bits [n, kv_heads * head_dim] of the cached values of the given slots."""
    s = _c(slots, np.int64)
    out = np.empty((s.size, kv_heads * head_dim), np.uint16)
    _check(lib().orc_kv_cache_dequant(_p(_c(cache, np.uint8)), _p(_c(scale, np.float32)), _p(s), s.size, kv_heads,
                                      head_dim, _p(out)), "kv_cache_dequant")
    return out


def gemm_i8(Xq, Wq, nthreads=1):
    """int32 acc[m,n] = sum_k Xq[m,k]*Wq[n,k] (int64 accumulation, range-checked)."""
    Xq = _c(Xq, np.uint8)
    Wq = _c(Wq, np.uint8)
    M, K = Xq.shape
    N = Wq.shape[0]
    acc = np.empty((M, N), np.int32)
    _check(lib().orc_gemm_i8(_p(Xq), _p(Wq), M, N, K, _p(acc), int(nthreads)), "gemm_i8")
    return acc


def gemm_fp8(Xq, Wq, nthreads=1):
    """fp64 acc[m,n] = sum_k dec(Xq[m,k])*dec(Wq[n,k]) (exact)."""
    Xq = _c(Xq, np.uint8)
    Wq = _c(Wq, np.uint8)
    M, K = Xq.shape
    N = Wq.shape[0]
    acc = np.empty((M, N), np.float64)
    _check(lib().orc_gemm_fp8(_p(Xq), _p(Wq), M, N, K, _p(acc), int(nthreads)), "gemm_fp8")
    return acc


def epilogue(acc, sx, sw):
    """bf16 bits y = bf16((fp32(acc) * sx[m]) * sw[n])."""
    sx = _c(sx, np.float32)
    sw = _c(sw, np.float32)
    M, N = acc.shape
    Y = np.empty((M, N), np.uint16)
    if acc.dtype == np.int32:
        a = _c(acc, np.int32)
        lib().orc_epilogue_i32(_p(a), _p(sx), _p(sw), M, N, _p(Y), N)
    else:
        a = _c(acc, np.float64)
        lib().orc_epilogue_f64(_p(a), _p(sx), _p(sw), M, N, _p(Y), N)
    return Y


def w8a8_linear(Xq, sx, Wq, sw, qtype, nthreads=1):
    """Full W8A8 linear: exact 8-bit GEMM then the dequantizing epilogue.
    Returns (Y bf16 bits [M,N], acc)."""
    acc = gemm_i8(Xq, Wq, nthreads) if qtype == INT8 else gemm_fp8(Xq, Wq, nthreads)
    return epilogue(acc, sx, sw), acc


# ---------------------------------------------------------------- 4-bit variant (NVFP4)

def e2m1_encode(v) -> np.ndarray:
    """fp32 -> E2M1 codes (0..15; RNE, saturating at 6, sign kept)."""
    L = lib()
    v = _c(v, np.float32)
    return np.array([L.orc_e2m1_encode(float(x)) for x in v.ravel()], np.uint8).reshape(v.shape)


def e2m1_decode(codes) -> np.ndarray:
    L = lib()
    table = np.array([L.orc_e2m1_decode(c) for c in range(16)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8) & 15]


def nvfp4_quant_rows(V):
    """fp32 rows [R, K] -> (packed codes u8 [R, K/2], block scales e4m3 u8 [R, K/16], row scales f32 [R])."""
    V = _c(V, np.float32)
    R, K = V.shape
    q4 = np.empty((R, K // 2), np.uint8)
    sb = np.empty((R, K // 16), np.uint8)
    g = np.empty(R, np.float32)
    _check(lib().orc_nvfp4_quant_rows_f32(_p(V), R, K, K, _p(q4), _p(sb), _p(g)), "nvfp4_quant_rows")
    return q4, sb, g


def nvfp4_quant_act(X_bits, pre_scale=1.0):
    """bf16 rows (uint16 bits) [M, K], v = x * pre_scale -> (codes, block scales, row scales)."""
    X = _c(X_bits, np.uint16)
    M, K = X.shape
    q4 = np.empty((M, K // 2), np.uint8)
    sb = np.empty((M, K // 16), np.uint8)
    g = np.empty(M, np.float32)
    _check(lib().orc_nvfp4_quant_act(_p(X), M, K, K, float(pre_scale), _p(q4), _p(sb), _p(g)), "nvfp4_quant_act")
    return q4, sb, g


def nvfp4_unpack(q4) -> np.ndarray:
    """Packed codes [R, K/2] -> one code per value [R, K] (value 2j in the low nibble)."""
    q4 = np.asarray(q4, np.uint8)
    out = np.empty((q4.shape[0], q4.shape[1] * 2), np.uint8)
    out[:, 0::2] = q4 & 15
    out[:, 1::2] = q4 >> 4
    return out


def gemm_nvfp4(q4x, sbx, q4w, sbw, nthreads=1) -> np.ndarray:
    """Exact acc[m, n] = sum_k x value * w value (block scales applied, row scales not), fp64."""
    q4x, sbx, q4w, sbw = (_c(a, np.uint8) for a in (q4x, sbx, q4w, sbw))
    M, N, K = q4x.shape[0], q4w.shape[0], q4x.shape[1] * 2
    acc = np.empty((M, N), np.float64)
    _check(lib().orc_gemm_nvfp4(_p(q4x), _p(sbx), _p(q4w), _p(sbw), M, N, K, _p(acc), nthreads), "gemm_nvfp4")
    return acc


def count_diff(a, b) -> int:
    a = _c(a, np.uint8)
    b = _c(b, np.uint8)
    assert a.size == b.size
    return int(lib().orc_count_diff(_p(a), _p(b), a.size))


# ---------------------------------------------------------------- ACR objective

ACR_NSTATS = 6
ACR_STATS = ("objective", "n_valid", "clipped_frac", "mean_tis_weight", "capped_frac", "kl_behav_prox")


def acr_objective(logp, logp_prox, logp_behav, adv, mask, eps=0.2, C=2.0, adaptive=True):
    """The decoupled-PPO token objective with truncated importance weights and
    ACR's clipping range (qurl_oracle.c, orc_acr_objective).  Inputs: [T]
    float32 log-probabilities and advantages, [T] uint8 mask.  Returns
    (stats float64 [6] in ACR_STATS order, term float64 [T], dterm float64 [T])."""
    lp, lpp, lpb, a = (_c(x, np.float32) for x in (logp, logp_prox, logp_behav, adv))
    m = _c(mask, np.uint8)
    T = lp.size
    assert lpp.size == lpb.size == a.size == m.size == T
    term = np.empty(T, np.float64)
    dterm = np.empty(T, np.float64)
    stats = np.empty(ACR_NSTATS, np.float64)
    _check(lib().orc_acr_objective(_p(lp), _p(lpp), _p(lpb), _p(a), _p(m), T, float(eps), float(C),
                                   1 if adaptive else 0, _p(term), _p(dterm), _p(stats)), "acr_objective")
    return stats, term, dterm
