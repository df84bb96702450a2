"""W8A8 linear layer of QuRL's quantized rollout actor on one GB300 (sm_103a).

A thin binding over the C ABI of ``libqurl.so`` (``include/qurl.h``).  Every
function named ``qurl_*`` has the C entry point's name and arguments, with
torch tensors in place of device pointers; it only marshals arguments -- every
step of the computation runs in the library's CUDA kernels.  The convenience
helpers at the bottom allocate outputs with torch and call those functions.

There is no CPU fallback: if the CUDA library has not been built, or no CUDA
device is present, the calls raise.

Method: Paper-Notes ICLR2026, "QuRL: Efficient Reinforcement Learning with
Quantized Rollout" -- UAQ invariant scaling W X = (W/s)(sX) with s folded into
the preceding norm gain (section "更新感知量化 (UAQ)"), per-channel weight and
per-token activation INT8 / FP8 quantization, s = 1.5 (section "损失函数 /
训练策略"), INT8/FP8 matmul in the rollout (section "系统集成与工程实现").
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
import weakref

import torch

from . import _build

INT8 = 0
FP8_E4M3 = 1
BF16 = 0
FP32 = 1

STATUS = {0: "QURL_OK", 1: "QURL_ERR_INVALID_ARG", 2: "QURL_ERR_UNSUPPORTED", 3: "QURL_ERR_ALIGNMENT",
          4: "QURL_ERR_WORKSPACE", 5: "QURL_ERR_CUDA", 6: "QURL_ERR_TIMEOUT"}

HEADER = os.path.join(_build.ROOT, "include", "qurl.h")

_lock = threading.Lock()
_lib = None


class QurlError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


def lib_path() -> str:
    return _build.LIB


def exported_names() -> list[str]:
    """Entry points declared in include/qurl.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(qurl_[a-z0-9_]+)\s*\(", text)))


def load() -> ctypes.CDLL:
    """Load libqurl.so (built by ``_build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is not built; run `python -m w8a8_precision_gemm_gb300._build` "
                               "(or __graft_entry__.build()) first -- this package has no CPU fallback")
        L = ctypes.CDLL(_build.LIB)
        P, i, f, z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sig = {
            "qurl_prepare_weights": [P, i, i, i, i, P, f, i, P, P, P, P, P],
            "qurl_quant_act": [P, i, i, i, f, i, P, P, P],
            "qurl_rmsnorm_quant": [P, i, i, i, P, f, i, P, P, P, P],
            "qurl_silu_mul_quant": [P, i, i, i, f, i, P, P, P, P],
            "qurl_w8a8_linear": [P, P, P, P, i, i, i, i, P, i, P, z, P],
            "qurl_w8a8_gemm_acc": [P, P, i, i, i, i, P, P, z, P],
            "qurl_w8a8_linear_static_scratch": [P, P, P, P, i, i, i, i, P, i, P],
            "qurl_rmsnorm_quant_linear": [P, i, P, f, P, P, i, i, i, i, P, i, P, P, P, z, P],
            "qurl_quant_act_linear": [P, i, f, P, P, i, i, i, i, P, i, P, P, P, z, P],
            "qurl_silu_mul_quant_linear": [P, i, f, P, P, i, i, i, i, P, i, P, P, P, z, P],
            "qurl_count_diff": [P, P, z, P, P],
            "qurl_check_device_status": [P],
            "qurl_debug_inject_timeout": [],
            "qurl_set_fused_decode": [i, P],
            "qurl_widen_weights": [P, i, i, P, P],
            "qurl_detach_wide_weights": [P],
            "qurl_nvfp4_quant": [P, i, i, i, i, f, P, P, P, P],
            "qurl_nvfp4_widen_weights": [P, P, i, i, P, P],
            "qurl_nvfp4_linear": [P, P, P, P, P, P, i, i, i, P, i, P, z, P],
            "qurl_nvfp4_gemm_acc": [P, P, P, P, i, i, i, P, P, z, P],
            "qurl_debug_plan": [i, i, i, i, i, z, P],
            "qurl_debug_plan_ex": [i, i, i, i, i, z, i, P],
            "qurl_debug_mma_probe": [i, i, i, P, P],
            "qurl_acr_objective": [P, P, P, P, P, ctypes.c_longlong, f, f, i, P, P, P, P, z, P],
            "qurl_kv_cache_quant": [P, i, i, i, i, i, P, ctypes.c_longlong, P, P, P, P, P],
            "qurl_kv_cache_dequant": [P, P, P, i, i, i, ctypes.c_longlong, P, P],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.qurl_workspace_size.argtypes = [i, i, i, i]
        L.qurl_workspace_size.restype = ctypes.c_size_t
        L.qurl_wide_weights_size.argtypes = [i, i]
        L.qurl_wide_weights_size.restype = ctypes.c_size_t
        L.qurl_nvfp4_workspace_size.argtypes = [i, i, i]
        L.qurl_nvfp4_workspace_size.restype = ctypes.c_size_t
        L.qurl_acr_workspace_size.argtypes = []
        L.qurl_acr_workspace_size.restype = ctypes.c_size_t
        L.qurl_status_string.argtypes = [ctypes.c_int]
        L.qurl_status_string.restype = ctypes.c_char_p
        L.qurl_version.argtypes = []
        L.qurl_version.restype = ctypes.c_int
        L.qurl_kernel_launches.argtypes = []
        L.qurl_kernel_launches.restype = ctypes.c_ulonglong
        _lib = L
        return L


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libqurl takes device tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ok(rc: int, where: str):
    if rc != 0:
        raise QurlError(rc, where)


def _ld(t) -> int:
    """Row stride of a row-major matrix whose rows may be strided (X, GU, W, Y)."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D tensor with unit column stride")
    return t.stride(0)


def _dense(*ts):
    """Code, scale and accumulator buffers are dense (row stride = row length)."""
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("code / scale / accumulator tensors must be contiguous")


# ---------------------------------------------------------------- the C ABI, by name

def qurl_prepare_weights(W, gamma, s, qt, Wq, sw, gamma_folded=None, W_scaled=None, stream=None):
    _dense(gamma, Wq, sw, gamma_folded, W_scaled)
    wt = FP32 if W.dtype == torch.float32 else BF16
    N, K = W.shape
    _ok(load().qurl_prepare_weights(_ptr(W), wt, N, K, _ld(W), _ptr(gamma), float(s), qt, _ptr(Wq), _ptr(sw),
                                    _ptr(gamma_folded), _ptr(W_scaled), _stream(stream)), "qurl_prepare_weights")


def qurl_quant_act(X, pre_scale, qt, Xq, sx, stream=None):
    _dense(Xq, sx)
    M, K = X.shape
    _ok(load().qurl_quant_act(_ptr(X), M, K, _ld(X), float(pre_scale), qt, _ptr(Xq), _ptr(sx), _stream(stream)),
        "qurl_quant_act")


def qurl_rmsnorm_quant(X, gamma_folded, eps, qt, Xq, sx, ms_out=None, stream=None):
    _dense(gamma_folded, Xq, sx, ms_out)
    M, K = X.shape
    _ok(load().qurl_rmsnorm_quant(_ptr(X), M, K, _ld(X), _ptr(gamma_folded), float(eps), qt, _ptr(Xq), _ptr(sx),
                                  _ptr(ms_out), _stream(stream)), "qurl_rmsnorm_quant")


def qurl_silu_mul_quant(GU, pre_scale, qt, Xq, sx, h_out=None, stream=None):
    _dense(Xq, sx, h_out)
    M, I2 = GU.shape
    _ok(load().qurl_silu_mul_quant(_ptr(GU), M, I2 // 2, _ld(GU), float(pre_scale), qt, _ptr(Xq), _ptr(sx),
                                   _ptr(h_out), _stream(stream)), "qurl_silu_mul_quant")


def qurl_workspace_size(M, N, K, qt) -> int:
    return int(load().qurl_workspace_size(M, N, K, qt))


def qurl_w8a8_linear(Xq, sx, Wq, sw, qt, Y, workspace=None, stream=None):
    _dense(Xq, sx, Wq, sw, workspace)
    M, K = Xq.shape
    N = Wq.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(load().qurl_w8a8_linear(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), M, N, K, qt, _ptr(Y), _ld(Y),
                                _ptr(workspace), ws_bytes, _stream(stream)), "qurl_w8a8_linear")


def qurl_w8a8_linear_static_scratch(Xq, sx, Wq, sw, qt, Y, stream=None):
    """qurl_w8a8_linear with the library's built-in scratch buffer instead of a
    workspace: for callers that cannot allocate device memory."""
    _dense(Xq, sx, Wq, sw)
    M, K = Xq.shape
    N = Wq.shape[0]
    _ok(load().qurl_w8a8_linear_static_scratch(_ptr(Xq), _ptr(sx), _ptr(Wq), _ptr(sw), M, N, K, qt, _ptr(Y), _ld(Y),
                                               _stream(stream)), "qurl_w8a8_linear_static_scratch")


def qurl_w8a8_gemm_acc(Xq, Wq, qt, acc, workspace=None, stream=None):
    _dense(Xq, Wq, acc, workspace)
    M, K = Xq.shape
    N = Wq.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(load().qurl_w8a8_gemm_acc(_ptr(Xq), _ptr(Wq), M, N, K, qt, _ptr(acc), _ptr(workspace), ws_bytes,
                                  _stream(stream)), "qurl_w8a8_gemm_acc")


def qurl_rmsnorm_quant_linear(X, gamma_folded, eps, Wq, sw, qt, Y, Xq_scratch, sx_scratch, workspace=None,
                              stream=None):
    _dense(gamma_folded, Wq, sw, Xq_scratch, sx_scratch, workspace)
    M, K = X.shape
    N = Wq.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(load().qurl_rmsnorm_quant_linear(_ptr(X), _ld(X), _ptr(gamma_folded), float(eps), _ptr(Wq), _ptr(sw), M, N,
                                         K, qt, _ptr(Y), _ld(Y), _ptr(Xq_scratch), _ptr(sx_scratch),
                                         _ptr(workspace), ws_bytes, _stream(stream)), "qurl_rmsnorm_quant_linear")


def qurl_quant_act_linear(X, pre_scale, Wq, sw, qt, Y, Xq_scratch, sx_scratch, workspace=None, stream=None):
    _dense(Wq, sw, Xq_scratch, sx_scratch, workspace)
    M, K = X.shape
    N = Wq.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(load().qurl_quant_act_linear(_ptr(X), _ld(X), float(pre_scale), _ptr(Wq), _ptr(sw), M, N, K, qt, _ptr(Y),
                                     _ld(Y), _ptr(Xq_scratch), _ptr(sx_scratch), _ptr(workspace), ws_bytes,
                                     _stream(stream)), "qurl_quant_act_linear")


def qurl_silu_mul_quant_linear(GU, pre_scale, Wq, sw, qt, Y, Xq_scratch, sx_scratch, workspace=None, stream=None):
    _dense(Wq, sw, Xq_scratch, sx_scratch, workspace)
    M, I2 = GU.shape
    N = Wq.shape[0]
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _ok(load().qurl_silu_mul_quant_linear(_ptr(GU), _ld(GU), float(pre_scale), _ptr(Wq), _ptr(sw), M, N, I2 // 2,
                                          qt, _ptr(Y), _ld(Y), _ptr(Xq_scratch), _ptr(sx_scratch), _ptr(workspace),
                                          ws_bytes, _stream(stream)), "qurl_silu_mul_quant_linear")


def qurl_count_diff(a, b, count, stream=None):
    _dense(a, b, count)
    n = a.numel() * a.element_size()
    assert b.numel() * b.element_size() == n
    _ok(load().qurl_count_diff(_ptr(a), _ptr(b), n, _ptr(count), _stream(stream)), "qurl_count_diff")


def qurl_acr_objective(logp, logp_prox, logp_behav, adv, mask, eps, C, adaptive, term, dterm, stats, workspace,
                       stream=None):
    ins = (logp, logp_prox, logp_behav, adv)
    _dense(*ins, mask, term, dterm, stats, workspace)
    T = logp.numel()
    for t in ins + tuple(x for x in (term, dterm) if x is not None):
        if t.dtype != torch.float32 or t.numel() != T:
            raise ValueError("log-probabilities, advantages, term and dterm are fp32 [T]")
    if mask.dtype not in (torch.uint8, torch.bool) or mask.numel() != T:
        raise ValueError("mask is uint8 / bool [T]")
    if stats.dtype != torch.float64 or stats.numel() < ACR_NSTATS:
        raise ValueError("stats is fp64 [6]")
    _ok(load().qurl_acr_objective(*(_ptr(t) for t in ins), _ptr(mask), T, float(eps), float(C), 1 if adaptive else 0,
                                  _ptr(term), _ptr(dterm), _ptr(stats), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream(stream)),
        "qurl_acr_objective")


def qurl_kv_cache_quant(qkv, q_dim, kv_heads, head_dim, slot_mapping, k_cache, k_scale, v_cache, v_scale,
                        stream=None):
    _dense(slot_mapping, k_cache, k_scale, v_cache, v_scale)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping is int64")
    M = qkv.shape[0]
    _ok(load().qurl_kv_cache_quant(_ptr(qkv), M, _ld(qkv), q_dim, kv_heads, head_dim, _ptr(slot_mapping),
                                   k_cache.shape[0], _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale),
                                   _stream(stream)), "qurl_kv_cache_quant")


def qurl_kv_cache_dequant(cache, scale, slots, out, stream=None):
    _dense(cache, scale, slots, out)
    num_slots, kv_heads, head_dim = cache.shape
    _ok(load().qurl_kv_cache_dequant(_ptr(cache), _ptr(scale), _ptr(slots), slots.numel(), kv_heads, head_dim,
                                     num_slots, _ptr(out), _stream(stream)), "qurl_kv_cache_dequant")


def kv_cache(num_slots, kv_heads, head_dim, device="cuda"):
    """Empty FP8 key and value caches with their scales: (k_cache, k_scale, v_cache, v_scale)."""
    return (torch.empty((num_slots, kv_heads, head_dim), dtype=torch.float8_e4m3fn, device=device),
            torch.empty((num_slots, kv_heads), dtype=torch.float32, device=device),
            torch.empty((num_slots, kv_heads, head_dim), dtype=torch.float8_e4m3fn, device=device),
            torch.empty((num_slots, kv_heads), dtype=torch.float32, device=device))


def qurl_check_device_status(stream=None):
    _ok(load().qurl_check_device_status(_stream(stream)), "qurl_check_device_status")


def plan(M, N, K, qt, num_sms, ws_bytes=None, attached=False):
    """The GEMM plan for a shape (host-side; see qurl_debug_plan_ex): with
    `attached`, the INT8 plan of weights that carry an fp16 copy;
    "whole_units" counts the tiles that run unsplit before a split tail."""
    out = (ctypes.c_longlong * 9)()
    ws = ctypes.c_size_t(-1).value if ws_bytes is None else ws_bytes
    _ok(load().qurl_debug_plan_ex(M, N, K, qt, num_sms, ws, 1 if attached else 0, out), "qurl_debug_plan_ex")
    keys = ("kernel", "swap", "bn", "tiles_tok", "tiles_ch", "splits", "kb_per_split", "ws_bytes", "whole_units")
    return dict(zip(keys, list(out)))


def qurl_debug_mma_probe(route, ctas, iters, stream=None) -> float:
    """Launch a tensor-rate probe (see include/qurl.h); returns the operations it performs."""
    ops = ctypes.c_double(0.0)
    _ok(load().qurl_debug_mma_probe(route, ctas, iters, ctypes.byref(ops), _stream(stream)), "qurl_debug_mma_probe")
    return ops.value


def qurl_debug_inject_timeout():
    """Test hook: the next GEMM launch stalls on purpose and times out (~1 s)."""
    _ok(load().qurl_debug_inject_timeout(), "qurl_debug_inject_timeout")


def qurl_set_fused_decode(mode: int) -> int:
    """Where the fused entries quantize a decode batch: 0 its own kernel, 1 inside
    the GEMM kernel where that is faster (default), 2 inside it wherever possible.
    Returns the previous mode."""
    prev = ctypes.c_int(0)
    _ok(load().qurl_set_fused_decode(int(mode), ctypes.byref(prev)), "qurl_set_fused_decode")
    return prev.value


def qurl_status_string(s: int) -> str:
    return load().qurl_status_string(s).decode()


def qurl_version() -> int:
    return int(load().qurl_version())


def qurl_kernel_launches() -> int:
    return int(load().qurl_kernel_launches())


# ---------------------------------------------------------------- allocating helpers

def code_dtype(qt):
    return torch.int8 if qt == INT8 else torch.float8_e4m3fn


def prepare_weights(W, qt, s=1.5, gamma=None, keep_scaled=True, stream=None):
    """UAQ fold + per-channel quantization.  Returns (Wq, sw, gamma', W')."""
    N, K = W.shape
    dev = W.device
    Wq = torch.empty((N, K), dtype=code_dtype(qt), device=dev)
    sw = torch.empty(N, dtype=torch.float32, device=dev)
    gf = None if gamma is None else torch.empty(K, dtype=torch.float32, device=dev)
    Ws = torch.empty((N, K), dtype=torch.float32, device=dev) if keep_scaled else None
    qurl_prepare_weights(W, gamma, s, qt, Wq, sw, gf, Ws, stream)
    return Wq, sw, gf, Ws


def quant_act(X, qt, pre_scale=1.0, stream=None):
    M, K = X.shape
    Xq = torch.empty((M, K), dtype=code_dtype(qt), device=X.device)
    sx = torch.empty(M, dtype=torch.float32, device=X.device)
    qurl_quant_act(X, pre_scale, qt, Xq, sx, stream)
    return Xq, sx


def rmsnorm_quant(X, gamma_folded, qt, eps=1e-6, want_ms=False, stream=None):
    M, K = X.shape
    Xq = torch.empty((M, K), dtype=code_dtype(qt), device=X.device)
    sx = torch.empty(M, dtype=torch.float32, device=X.device)
    ms = torch.empty(M, dtype=torch.float32, device=X.device) if want_ms else None
    qurl_rmsnorm_quant(X, gamma_folded, eps, qt, Xq, sx, ms, stream)
    return (Xq, sx, ms) if want_ms else (Xq, sx)


def silu_mul_quant(GU, qt, pre_scale=1.0, want_h=False, stream=None):
    M, I2 = GU.shape
    Xq = torch.empty((M, I2 // 2), dtype=code_dtype(qt), device=GU.device)
    sx = torch.empty(M, dtype=torch.float32, device=GU.device)
    h = torch.empty((M, I2 // 2), dtype=torch.float32, device=GU.device) if want_h else None
    qurl_silu_mul_quant(GU, pre_scale, qt, Xq, sx, h, stream)
    return (Xq, sx, h) if want_h else (Xq, sx)


def workspace(M, N, K, qt, device="cuda"):
    """Workspace for a linear call of this shape, zero-filled: its last 256 bytes
    hold the fused entry points' handoff counters, which must start at zero (and
    which every call leaves at zero)."""
    nbytes = qurl_workspace_size(M, N, K, qt)
    return torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device) if nbytes else None


def linear(Xq, sx, Wq, sw, qt, ws=None, stream=None):
    M, N = Xq.shape[0], Wq.shape[0]
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=Xq.device)
    qurl_w8a8_linear(Xq, sx, Wq, sw, qt, Y, ws, stream)
    return Y


def gemm_acc(Xq, Wq, qt, ws=None, stream=None):
    M, N = Xq.shape[0], Wq.shape[0]
    acc = torch.empty((M, N), dtype=torch.int32 if qt == INT8 else torch.float32, device=Xq.device)
    qurl_w8a8_gemm_acc(Xq, Wq, qt, acc, ws, stream)
    return acc


def count_diff(a, b, stream=None) -> torch.Tensor:
    c = torch.empty(1, dtype=torch.int64, device=a.device)
    qurl_count_diff(a, b, c, stream)
    return c


# ---------------------------------------------------------------- attached fp16 weight copies

def qurl_widen_weights(Wq, wide, stream=None):
    """Write the fp16 copy of INT8 codes Wq [N, K] (and their per-channel sums
    of squares) into `wide` and attach it to Wq (see include/qurl.h)."""
    _dense(Wq, wide)
    N, K = Wq.shape
    _ok(load().qurl_widen_weights(_ptr(Wq), N, K, _ptr(wide), _stream(stream)), "qurl_widen_weights")


def qurl_detach_wide_weights(Wq):
    _ok(load().qurl_detach_wide_weights(_ptr(Wq)), "qurl_detach_wide_weights")


def wide_weights(Wq, stream=None) -> torch.Tensor:
    """Allocate, fill and attach the fp16 copy of INT8 codes Wq.  The returned
    tensor holds a reference to Wq and detaches the copy when it is freed, so
    neither buffer can be reused at its address while attached."""
    N, K = Wq.shape
    wide = torch.empty(int(load().qurl_wide_weights_size(N, K)), dtype=torch.uint8, device=Wq.device)
    qurl_widen_weights(Wq, wide, stream)
    wide._qurl_wq = Wq  # Wq outlives the attachment
    weakref.finalize(wide, load().qurl_detach_wide_weights, ctypes.c_void_p(Wq.data_ptr()))
    return wide


# ---------------------------------------------------------------- 4-bit variant (NVFP4)

def qurl_nvfp4_quant(X, pre_scale, q4, sblk, g, stream=None):
    """Rows of X (bf16 times pre_scale, or fp32) -> E2M1 codes q4 [R, K/2], E4M3
    block scales sblk [R, K/16], row scales g [R] (see include/qurl.h)."""
    _dense(q4, sblk, g)
    R, K = X.shape
    xt = FP32 if X.dtype == torch.float32 else BF16
    _ok(load().qurl_nvfp4_quant(_ptr(X), xt, R, K, _ld(X), float(pre_scale), _ptr(q4), _ptr(sblk), _ptr(g),
                                _stream(stream)), "qurl_nvfp4_quant")


def qurl_nvfp4_workspace_size(M, N, K) -> int:
    return int(load().qurl_nvfp4_workspace_size(M, N, K))


def qurl_nvfp4_linear(x, w, Y, workspace, stream=None):
    """Y = the 4-bit linear of x = (q4, sblk, g) tokens and w = (q4, sblk, g) channels."""
    (q4x, sbx, gx), (q4w, sbw, gw) = x, w
    _dense(q4x, sbx, gx, q4w, sbw, gw, workspace)
    M, N, K = q4x.shape[0], q4w.shape[0], q4x.shape[1] * 2
    _ok(load().qurl_nvfp4_linear(_ptr(q4x), _ptr(sbx), _ptr(gx), _ptr(q4w), _ptr(sbw), _ptr(gw), M, N, K, _ptr(Y),
                                 _ld(Y), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "qurl_nvfp4_linear")


def qurl_nvfp4_gemm_acc(x, w, acc, workspace, stream=None):
    (q4x, sbx, _), (q4w, sbw, _) = x, w
    _dense(q4x, sbx, q4w, sbw, acc, workspace)
    M, N, K = q4x.shape[0], q4w.shape[0], q4x.shape[1] * 2
    _ok(load().qurl_nvfp4_gemm_acc(_ptr(q4x), _ptr(sbx), _ptr(q4w), _ptr(sbw), M, N, K, _ptr(acc), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
        "qurl_nvfp4_gemm_acc")


def nvfp4_quant(X, pre_scale=1.0, stream=None):
    """Allocating wrapper: returns (q4 uint8 [R, K/2], sblk uint8 [R, K/16], g fp32 [R])."""
    R, K = X.shape
    q4 = torch.empty((R, K // 2), dtype=torch.uint8, device=X.device)
    sb = torch.empty((R, K // 16), dtype=torch.uint8, device=X.device)
    g = torch.empty(R, dtype=torch.float32, device=X.device)
    qurl_nvfp4_quant(X, pre_scale, q4, sb, g, stream)
    return q4, sb, g


def nvfp4_wide_weights(w, stream=None) -> torch.Tensor:
    """Allocate, fill and attach the fp16 copy of 4-bit weight rows w = (q4, sblk, g);
    detached when the returned tensor is freed (it holds a reference to q4)."""
    q4, sb, _ = w
    N, K = q4.shape[0], q4.shape[1] * 2
    wide = torch.empty(N * K * 2, dtype=torch.uint8, device=q4.device)
    _ok(load().qurl_nvfp4_widen_weights(_ptr(q4), _ptr(sb), N, K, _ptr(wide), _stream(stream)),
        "qurl_nvfp4_widen_weights")
    wide._qurl_wq = q4
    weakref.finalize(wide, load().qurl_detach_wide_weights, ctypes.c_void_p(q4.data_ptr()))
    return wide


def nvfp4_workspace(M, N, K, device="cuda") -> torch.Tensor:
    return torch.empty(max(qurl_nvfp4_workspace_size(M, N, K), 16), dtype=torch.uint8, device=device)


def nvfp4_linear(x, w, ws=None, stream=None):
    M, N = x[0].shape[0], w[0].shape[0]
    ws = nvfp4_workspace(M, N, x[0].shape[1] * 2, x[0].device) if ws is None else ws
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=x[0].device)
    qurl_nvfp4_linear(x, w, Y, ws, stream)
    return Y


def nvfp4_gemm_acc(x, w, ws=None, stream=None):
    M, N = x[0].shape[0], w[0].shape[0]
    ws = nvfp4_workspace(M, N, x[0].shape[1] * 2, x[0].device) if ws is None else ws
    acc = torch.empty((M, N), dtype=torch.float32, device=x[0].device)
    qurl_nvfp4_gemm_acc(x, w, acc, ws, stream)
    return acc


# ---------------------------------------------------------------- ACR objective

ACR_NSTATS = 6
ACR_STATS = ("objective", "n_valid", "clipped_frac", "mean_tis_weight", "capped_frac", "kl_behav_prox")


def acr_workspace(device="cuda") -> torch.Tensor:
    """Scratch for qurl_acr_objective: zero-filled once (its ticket counter),
    left ready for reuse by every call."""
    return torch.zeros(int(load().qurl_acr_workspace_size()), dtype=torch.uint8, device=device)


def acr_objective(logp, logp_prox, logp_behav, adv, mask, eps=0.2, C=2.0, adaptive=True, want_term=False,
                  want_dterm=True, workspace=None, stream=None):
    """The ACR token objective (qurl_acr_objective).  Returns (stats fp64 [6] in
    ACR_STATS order, dterm fp32 [T] or None, term fp32 [T] or None)."""
    dev = logp.device
    T = logp.numel()
    stats = torch.empty(ACR_NSTATS, dtype=torch.float64, device=dev)
    dterm = torch.empty(T, dtype=torch.float32, device=dev) if want_dterm else None
    term = torch.empty(T, dtype=torch.float32, device=dev) if want_term else None
    ws = acr_workspace(dev) if workspace is None else workspace
    qurl_acr_objective(logp, logp_prox, logp_behav, adv, mask, eps, C, adaptive, term, dterm, stats, ws, stream)
    return stats, dterm, term
