"""Benchmark of the W8A8 linear layer path on one GB300.

Headline workload: the 32B-class projections (hidden 5120, intermediate 27648,
fused qkv N = 7168) in INT8 and in FP8-E4M3, at M = 256 (decode), 1024 and 8192
(prefill) tokens.  One step is one pass of the whole hot path over one batch of
each M in each 8-bit type -- six passes of the projection chain

    RMSNorm(gamma*s) -> quant -> qkv (K=5120, N=7168)
    quant(q-slice of qkv, pre-scale s) -> o_proj (K=N=5120)
    RMSNorm(gamma*s) -> quant -> gate_up (K=5120, N=55296)
    SiLU(gate)*up -> quant (pre-scale s) -> down (K=27648, N=5120)

through the fused quantize -> linear entry points of the C ABI, with the
weights prepared once by the UAQ fold (s = 1.5) and per-output-channel
quantization.  Synthetic, seeded inputs: X ~ N(0,1) with 1% outlier channels
x20, W ~ N(0,0.02), gamma ~ 1 + N(0,0.1).  The step streams 976 MB of weights
(each projection's weights come back only after the other three's, >= 450 MB,
have passed through the 129 MB L2).

Reported beside it (not part of `value`): the 7B-class decode chain (M = 64 and
256), the 7B-class chain at M = 512 and 4096 with the code flips of a weight
update W' -> W' + dW' for s = 1 and s = 1.5, every GEMM and quantizer on its
own against its roofline, the per-RL-step weight re-quantization, the ACR
token objective, the tensor-rate probes, the FP8 KV-cache quantizer, the 4-bit
(NVFP4) variant of the linear, the end-to-end number through the C ABI with
host buffers and the CPU oracle as a baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from w8a8_precision_gemm_gb300 import synth  # noqa: E402  (seeded inputs only; no method arithmetic)

METRIC = "W8A8 linear TOPS/TFLOPS and HBM GB/s vs roofline at 1 GB300 (INT8 & FP8)"
S_UAQ = 1.5
EPS = 1e-6
PROJ = ("qkv", "o_proj", "gate_up", "down")
QTYPES = ("int8", "fp8")
MODELS = {"7b": {"hidden": 3584, "inter": 18944, "shapes": synth.SHAPES_7B},
          "32b": {"hidden": 5120, "inter": 27648, "shapes": synth.SHAPES_32B}}
HEADLINE = ("32b", (256, 1024, 8192))
DECODE_7B = ("7b", (64, 256))
CHAIN_7B = ("7b", (512, 4096))
WORKLOAD = ("32B-class projection chain, INT8 and FP8-E4M3: RMSNorm->quant->qkv (5120->7168), "
            "quant->o_proj (5120->5120), RMSNorm->quant->gate_up (5120->55296), SiLU*mul->quant->down "
            "(27648->5120); M in {256, 1024, 8192} tokens; UAQ s=1.5; per-channel W, per-token A; bf16 out")
CLOCK_LEAD = 0.5  # s of untimed step replays right before the timed region
L2_FALLBACK = 129 * 1024 * 1024
# the ACR token objective timed beside the step: one mini-batch of 512 responses x 8192 token slots
ACR_SEQ, ACR_LEN, ACR_EPS, ACR_C = 512, 8192, 0.2, 2.0
ACR_KEYS = ("logp", "logp_prox", "logp_behav", "adv", "mask")
_CSRC = "w8a8_precision_gemm_gb300/csrc/"
ACR_PROFILE = "profiles/acr_objective_kernel_512x8192.md"
ACR_SOURCES = [_CSRC + "objective.cu", _CSRC + "objective.h"]
# committed ncu summaries of the GEMM kernels, keyed by the kernel's name; a summary's DRAM traffic is
# used only while the kernel's sources hash to the ones it was captured from
GEMM_PROFILES = {
    "w8a8_gemm_i8w_kernel": ("profiles/w8a8_gemm_i8w_kernel_32b_gate_up_int8.md",
                             [_CSRC + f for f in ("gemm.cuh", "gemm_i8w.cu", "ptx.cuh", "internal.h")]),
    "w8a8_gemm_fp8_pair_kernel": ("profiles/w8a8_gemm_fp8_pair_kernel_32b_gate_up_fp8.md",
                                  [_CSRC + f for f in ("gemm.cuh", "gemm_fp8p.cu", "ptx.cuh", "internal.h")]),
}
KERNEL_NAMES = {0: "w8a8_gemm_kernel", 1: "w8a8_gemm_i8t_kernel", 2: "w8a8_gemm_i8p_kernel",
                3: "w8a8_gemm_fp8_pair_kernel", 4: "w8a8_gemm_i8w_kernel"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def tensor_peak(pk, qtype):
    """Dense tensor rate of a qtype (TFLOP/s): FP8 = 2 x the bf16 rate (the nominal ratio); INT8 runs on
    the fp16 tensor path, whose dense rate is the bf16 one."""
    return pk["bf16_tflops"] * (2.0 if qtype == "fp8" else 1.0)


def traffic_from_profile(path, sources):
    """DRAM bytes per launch from a committed ncu summary, while the sources
    still hash to the captured ones; else None."""
    if not path or not os.path.exists(os.path.join(ROOT, path)):
        return None
    h = hashlib.sha256()
    for f in sources:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    fields = dict(line.split(": ", 1) for line in open(os.path.join(ROOT, path)).read().splitlines() if ": " in line
                  and line.split(": ", 1)[0] in ("kernel_sources_sha256_16", "dram_bytes_per_launch"))
    if fields.get("kernel_sources_sha256_16", "").split()[0:1] != [h.hexdigest()[:16]]:
        return None
    return int(fields["dram_bytes_per_launch"])


def alg_bytes(M, K, N):
    """Algorithmic bytes of one W8A8 linear: weight and activation codes in, bf16 Y out, fp32 scales."""
    return N * K + M * K + 2 * M * N + 4 * (M + N)


def gemm_roof_s(M, K, N, qtype, pk):
    """Roofline time of one linear: max(tensor time, HBM time)."""
    return max(2 * M * N * K / (tensor_peak(pk, qtype) * 1e12), alg_bytes(M, K, N) / (pk["hbm_gbs"] * 1e9))


def quant_bytes(kind, M, K):
    """Algorithmic bytes of a quantizer: bf16 rows in (gate and up for SiLU*mul), codes and fp32 scales out."""
    return (4 * M * K if kind == "silu_mul_quant" else 2 * M * K) + M * K + 4 * M


def chain_shapes(model):
    sh = MODELS[model]["shapes"]
    return [(name, sh[name][0], sh[name][1]) for name in PROJ]


def chain_ops(model, Ms):
    return sum(2 * M * N * K for M in Ms for _, K, N in chain_shapes(model))


def chain_roofline(model, M, qtype, pk):
    """Roofline time of one chain pass: its four linears at max(tensor, HBM) and its four quantizers at HBM."""
    hid, inter = MODELS[model]["hidden"], MODELS[model]["inter"]
    t_gemm = sum(gemm_roof_s(M, K, N, qtype, pk) for _, K, N in chain_shapes(model))
    qb = (2 * quant_bytes("rmsnorm_quant", M, hid) + quant_bytes("quant_act", M, hid) +
          quant_bytes("silu_mul_quant", M, inter))
    return t_gemm, qb / (pk["hbm_gbs"] * 1e9)


def dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return rank, world


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world):
    """Max of a host scalar over the ranks (replicas time independently; the job
    takes as long as its slowest rank)."""
    if world <= 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, ms_per_step_rank, world):
    """Whole-job throughput of weak-scaled replicas: the units every rank
    processed, divided by the slowest rank's time."""
    ms = max_over_ranks(ms_per_step_rank, world)
    return units_per_rank * world / (ms * 1e-3), ms


# ------------------------------------------------------------------ clocks

REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x20: "sync_boost", 0x40: "sw_thermal_slowdown", 0x80: "hw_thermal_slowdown",
               0x100: "hw_power_brake_slowdown", 0x200: "display_clock_setting"}


class ClockSampler:
    """nvidia-smi every 100 ms while the timed region runs.  Each sample carries
    the host time it arrived, so the summary can keep those taken in and next to
    the timed region."""

    def __init__(self, index):
        self.index = index
        self.samples = []  # (host time, sm MHz, max sm MHz, event-reason mask)
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        deadline = time.perf_counter() + 3.0  # nvidia-smi's first sample, before any timing starts
        while self.proc and not self.samples and time.perf_counter() < deadline and self.proc.poll() is None:
            time.sleep(0.02)
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 3:
                try:
                    self.samples.append((time.perf_counter(), float(parts[0]), float(parts[1]), int(parts[2], 16)))
                except ValueError:
                    pass

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1, lead):
        """Clocks over [t0 - lead, t1 + 0.15 s]: the timed region [t0, t1] and
        the same step replayed for `lead` seconds right before it."""
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sel = [x for x in self.samples if t0 - lead <= x[0] <= t1 + 0.15] or self.samples
        sm = [x[1] for x in sel]
        mask = 0
        for x in sel:
            mask |= x[3]
        reasons = [name for bit, name in REASON_BITS.items() if mask & bit and name != "gpu_idle"]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(x[2] for x in sel), "reasons": reasons,
                "samples": len(sel), "samples_in_timed_region": sum(t0 <= x[0] <= t1 + 0.15 for x in sel),
                "window": f"the timed region ({(t1 - t0) * 1e3:.0f} ms) and {lead:.1f} s of the same step "
                          "replayed just before it"}


# ------------------------------------------------------------------ the layer

def qt_of(q, qtype):
    return q.INT8 if qtype == "int8" else q.FP8_E4M3


def make_weights(model):
    """fp32 master weights and RMSNorm gains of one decoder layer's projections (CPU)."""
    W = {name: synth.weights(f"bench/{model}/{name}/W", N, K) for name, K, N in chain_shapes(model)}
    gammas = {"qkv": synth.gamma(f"bench/{model}/ln1", MODELS[model]["hidden"]),
              "gate_up": synth.gamma(f"bench/{model}/ln2", MODELS[model]["hidden"])}
    return W, gammas


def rotated_rows(W, N, rotate):
    """Weight set `rotate` of a projection: its output channels rotated by N / 2 (a distinct set of
    weights with the same statistics, so alternating sets do not share L2 lines)."""
    return torch.roll(W, shifts=N // 2, dims=0).contiguous() if rotate else W


class Layer:
    """Weights of one decoder layer's projections, prepared on the GPU by the UAQ
    fold: qkv and gate_up fold s into their RMSNorm gain, o_proj and down carry
    it as their quantizer's pre-scale."""

    def __init__(self, q, qt, model, W, gammas, rotate=0):
        self.q, self.qt, self.model = q, qt, model
        self.w = {}
        self.wide = {}
        for name, K, N in chain_shapes(model):
            Wd = rotated_rows(W[name].cuda(), N, rotate)
            g = gammas.get(name)
            Wq, sw, gf, _ = q.prepare_weights(Wd, qt, s=S_UAQ, gamma=None if g is None else g.cuda(),
                                              keep_scaled=False)
            self.w[name] = (Wq, sw, gf)
            if qt == q.INT8:  # the fp16 copy the INT8 prefill GEMM reads, kept with the weights
                self.wide[name] = q.wide_weights(Wq)
            del Wd
        torch.cuda.synchronize()


class Buffers:
    """Activations of one chain pass of M tokens (one workspace shared by its four linears, which run one
    after the other on one stream)."""

    def __init__(self, q, qt, model, M):
        dev = "cuda"
        hid, inter = MODELS[model]["hidden"], MODELS[model]["inter"]
        self.M, self.model = M, model
        self.x = torch.empty((M, hid), dtype=torch.bfloat16, device=dev)
        self.xq = torch.empty((M, inter), dtype=q.code_dtype(qt), device=dev)
        self.sx = torch.empty(M, dtype=torch.float32, device=dev)
        self.y = {name: torch.empty((M, N), dtype=torch.bfloat16, device=dev) for name, _, N in chain_shapes(model)}
        nws = max(q.qurl_workspace_size(M, N, K, qt) for _, K, N in chain_shapes(model))
        self.ws = torch.zeros(max(nws, 16), dtype=torch.uint8, device=dev)  # its last bytes: handoff counters


def dense(buf, M, K):
    """A dense [M, K] view at the start of a code buffer."""
    return buf.view(-1)[: M * K].view(M, K)


def chain(q, qt, L, B):
    """One pass of the projection chain for one batch, through the fused
    quantize -> linear entry points of the C ABI."""
    M = B.M
    hid = MODELS[B.model]["hidden"]
    xq = dense(B.xq, M, hid)
    Wq, sw, gf = L.w["qkv"]
    q.qurl_rmsnorm_quant_linear(B.x, gf, EPS, Wq, sw, qt, B.y["qkv"], xq, B.sx, B.ws)
    Wq, sw, _ = L.w["o_proj"]
    # attention stand-in: the q slice of the qkv output feeds o_proj (s moves to the activation)
    q.qurl_quant_act_linear(B.y["qkv"][:, :hid], S_UAQ, Wq, sw, qt, B.y["o_proj"], xq, B.sx, B.ws)
    Wq, sw, gf = L.w["gate_up"]
    q.qurl_rmsnorm_quant_linear(B.y["o_proj"], gf, EPS, Wq, sw, qt, B.y["gate_up"], xq, B.sx, B.ws)
    Wq, sw, _ = L.w["down"]
    q.qurl_silu_mul_quant_linear(B.y["gate_up"], S_UAQ, Wq, sw, qt, B.y["down"], B.xq, B.sx, B.ws)


def input_name(model, M):
    return f"bench/{model}/X/{M}"


# ------------------------------------------------------------------ CUDA graphs and timing

def graph_of(fn, q):
    """Capture fn() (C-ABI calls on the current stream) into a CUDA graph;
    returns the graph and the number of the library's kernels it holds."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # one eager pass on the capture stream (first-use set-up happens outside capture)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    n0 = q.qurl_kernel_launches()
    with torch.cuda.graph(g):
        fn()
    n = q.qurl_kernel_launches() - n0
    torch.cuda.synchronize()
    return g, n


def time_graph(g, reps, stream):
    """Average ms per replay of g over reps back-to-back replays (CUDA events on the launching stream)."""
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def l2_bytes():
    p = torch.cuda.get_device_properties(torch.cuda.current_device())
    return int(getattr(p, "L2_cache_size", 0) or L2_FALLBACK)


def n_sets(nbytes, l2):
    """Distinct buffer sets to rotate over so that the sets touched between two uses of one exceed 2 x L2."""
    return max(2, int(-(-3 * l2 // max(nbytes, 1))))


def rotated_codes(Wq, sw, k):
    """k weight sets with the codes' rows (and their scales) rotated: same statistics, distinct bytes."""
    out = [(Wq, sw)]
    N = Wq.shape[0]
    for i in range(1, k):
        sh = (i * 1009) % N
        out.append((torch.roll(Wq.view(torch.uint8), sh, 0).contiguous().view(Wq.dtype), torch.roll(sw, sh, 0)))
    return out


# ------------------------------------------------------------------ blocks timed beside the step

def time_chain_block(q, qtype, layers, model, Ms, reps, stream, pk):
    """One graph of the chain over the batches Ms (batch i on weight set i % 2); µs per pass, and its
    roofline fractions (GEMMs alone; GEMMs plus quantizers)."""
    qt = qt_of(q, qtype)
    bufs = [Buffers(q, qt, model, M) for M in Ms]
    for B in bufs:
        B.x.copy_(synth.activations(input_name(model, B.M), B.M, MODELS[model]["hidden"]))

    def step():
        for i, B in enumerate(bufs):
            chain(q, qt, layers[i % len(layers)], B)

    g, nl = graph_of(step, q)
    for _ in range(3):
        g.replay()
    ms = time_graph(g, reps, stream)
    t_g = sum(chain_roofline(model, M, qtype, pk)[0] for M in Ms)
    t_q = sum(chain_roofline(model, M, qtype, pk)[1] for M in Ms)
    ops = chain_ops(model, Ms)
    out = {"M": list(Ms), "us_per_step": ms * 1e3, "TOPS": ops / (ms * 1e-3) / 1e12, "launches_per_step": nl,
           "gemm_roofline_frac": t_g / (ms * 1e-3), "step_roofline_frac": (t_g + t_q) / (ms * 1e-3)}
    del g, bufs
    return out


def time_per_gemm(q, qtype, layer, model, Ms, stream, pk, l2):
    """Each linear of the chain on its own (qurl_w8a8_linear): a graph of R calls rotating over enough
    weight sets that a set returns only after more than 2 x L2 of other weights."""
    qt = qt_of(q, qtype)
    res = {}
    for M in Ms:
        for name, K, N in chain_shapes(model):
            Wq, sw, _ = layer.w[name]
            k = n_sets(N * K, l2)
            sets = rotated_codes(Wq, sw, k)
            plan = q.plan(M, N, K, qt, torch.cuda.get_device_properties(0).multi_processor_count)
            # INT8 weights carry their fp16 copy as the benchmark's layers do; above 256 tokens the call
            # then runs on the CTA-pair kernel that reads it
            wides = [q.wide_weights(t[0]) for t in sets] if qtype == "int8" else []
            kernel = KERNEL_NAMES[4 if (qtype == "int8" and M > 256) else plan["kernel"]]
            Xq, sx = q.quant_act(synth.activations(f"bench/{model}/{name}/Xg/{M}", M, K).cuda(), qt)
            ws = q.workspace(M, N, K, qt)
            Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            R = max(k, 4)

            def calls(Xq=Xq, sx=sx, sets=sets, ws=ws, Y=Y, R=R):
                for r in range(R):
                    q.qurl_w8a8_linear(Xq, sx, sets[r % len(sets)][0], sets[r % len(sets)][1], qt, Y, ws)

            g, nl = graph_of(calls, q)
            g.replay()
            us = time_graph(g, 3, stream) / R * 1e3
            ops = 2 * M * N * K
            nb = alg_bytes(M, K, N)
            t_t = ops / (tensor_peak(pk, qtype) * 1e12)
            t_h = nb / (pk["hbm_gbs"] * 1e9)
            res[f"{name}/M{M}"] = {"M": M, "K": K, "N": N, "us": us, "TOPS": ops / (us * 1e-6) / 1e12,
                                   "GBps": nb / (us * 1e-6) / 1e9, "bound": "tensor" if t_t >= t_h else "hbm",
                                   "roofline_frac": max(t_t, t_h) / (us * 1e-6), "launches": nl // R,
                                   "kernel": kernel, "weight_sets": k}
            del g, wides, sets, Xq, sx, ws, Y
    torch.cuda.empty_cache()
    return res


def time_per_quant(q, qtype, model, Ms, stream, pk, l2, gamma):
    """Each quantizer of the chain on its own, rotating over enough input rows to stream from HBM."""
    qt = qt_of(q, qtype)
    hid, inter = MODELS[model]["hidden"], MODELS[model]["inter"]
    gf = (gamma * S_UAQ).cuda()
    res = {}
    for M in Ms:
        for kind, K in (("rmsnorm_quant", hid), ("quant_act", hid), ("silu_mul_quant", inter)):
            nb = quant_bytes(kind, M, K)
            k = min(n_sets(nb, l2), 64)
            cols = 2 * K if kind == "silu_mul_quant" else K
            base = synth.activations(f"bench/{model}/{kind}/{M}", M, cols).cuda()
            ins = [torch.roll(base, i * 7, 0).contiguous() for i in range(k)]
            Xq = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
            sx = torch.empty(M, dtype=torch.float32, device="cuda")
            R = max(k, 8)

            def calls(ins=ins, Xq=Xq, sx=sx, kind=kind, R=R):
                for r in range(R):
                    x = ins[r % len(ins)]
                    if kind == "rmsnorm_quant":
                        q.qurl_rmsnorm_quant(x, gf, EPS, qt, Xq, sx)
                    elif kind == "quant_act":
                        q.qurl_quant_act(x, S_UAQ, qt, Xq, sx)
                    else:
                        q.qurl_silu_mul_quant(x, S_UAQ, qt, Xq, sx)

            g, _ = graph_of(calls, q)
            g.replay()
            us = time_graph(g, 3, stream) / R * 1e3
            res[f"{kind}/K{K}/M{M}"] = {"us": us, "GBps": nb / (us * 1e-6) / 1e9,
                                        "roofline_frac": nb / (pk["hbm_gbs"] * 1e9) / (us * 1e-6)}
            del g, ins, base
    torch.cuda.empty_cache()
    return res


def flip_probe(q, model, stream, pk, l2):
    """Weight-update probe (the UAQ argument): for each projection, the codes of
    W' = W / s (s = 1, 1.5) against those of W' + dW', dW' = s dW (SGD reading:
    the update of the trained parameter W' is s times larger) and dW' = dW
    (size-preserving reading), dW ~ N(0, 1e-7).  The update itself is the RL
    optimiser's step (torch elementwise ops, one multiply and one add, both
    rounded); re-quantization and the count run in the library.  Also times the
    re-quantization of the fp32 master (the per-RL-step weight quantization)."""
    out = {}
    requant = {}
    for qtype in QTYPES:
        qt = qt_of(q, qtype)
        counts = {}
        for name, K, N in chain_shapes(model):
            W = synth.weights(f"bench/{model}/{name}/W", N, K).cuda()
            dW = synth.update(f"bench/{model}/{name}/dW", N, K).cuda()
            c = {}
            for s in (1.0, S_UAQ):
                Wq0, _, _, Wp = q.prepare_weights(W, qt, s=s, keep_scaled=True)
                for reading, upd in (("sgd", dW * s), ("same_size", dW)):
                    Wn = Wp + upd
                    Wq1, _, _, _ = q.prepare_weights(Wn, qt, s=1.0, keep_scaled=False)
                    c[f"{reading}/s{s:g}"] = int(q.count_diff(Wq0, Wq1).item())
                    del Wn, Wq1
                if s == S_UAQ and 4 * N * K > l2:
                    # per-RL-step re-quantization of the trained fp32 master W' (s = 1), timed alone on the
                    # projections whose master exceeds L2 (gate_up, down)
                    Wq = torch.empty((N, K), dtype=q.code_dtype(qt), device="cuda")
                    sw = torch.empty(N, dtype=torch.float32, device="cuda")

                    def calls(Wp=Wp, Wq=Wq, sw=sw):
                        for _ in range(4):
                            q.qurl_prepare_weights(Wp, None, 1.0, qt, Wq, sw)

                    g, _ = graph_of(calls, q)
                    g.replay()
                    us = time_graph(g, 3, stream) / 4 * 1e3
                    nb = N * K * 4 + N * K + 4 * N
                    requant[f"{qtype}/{name}"] = {"us": us, "GBps": nb / (us * 1e-6) / 1e9,
                                                  "roofline_frac": nb / (pk["hbm_gbs"] * 1e9) / (us * 1e-6)}
                    del g, Wq, sw
                del Wq0, Wp
            counts[name] = c
            del W, dW
        tot = {k: sum(c[k] for c in counts.values()) for k in next(iter(counts.values()))}
        out[qtype] = {"per_projection": counts, "total": tot,
                      "ratio_s1.5_over_s1": {r: tot[f"{r}/s1.5"] / max(tot[f"{r}/s1"], 1)
                                             for r in ("sgd", "same_size")}}
    torch.cuda.empty_cache()
    out["expected_ratio"] = {"sgd": "about s^2 = 2.25", "same_size": "about s = 1.5"}
    return out, requant


def acr_bytes(T):
    """Algorithmic bytes of one ACR objective call per token slot: the four fp32
    inputs and the mask byte in, the fp32 derivative out (the per-CTA partials
    and the statistics are a few KB)."""
    return T * (4 * 4 + 1 + 4)


def acr_inputs(q, j):
    T = ACR_SEQ * ACR_LEN
    r = synth.rollout(f"bench/acr/{j}", ACR_SEQ, ACR_LEN)
    d = {k: torch.from_numpy(r[k]).cuda() for k in ACR_KEYS}
    d["dterm"] = torch.empty(T, dtype=torch.float32, device="cuda")
    d["stats"] = torch.empty(q.ACR_NSTATS, dtype=torch.float64, device="cuda")
    return r, d


def acr_call(q, d, ws):
    q.qurl_acr_objective(d["logp"], d["logp_prox"], d["logp_behav"], d["adv"], d["mask"], ACR_EPS, ACR_C, True,
                         None, d["dterm"], d["stats"], ws)


def time_acr(q, stream, pk, cpu_baseline):
    """The ACR token objective on the mini-batch: a graph of R calls rotating
    over three input sets, 88 MB each (71 MB in, 17 MB of derivatives out), so
    the two sets touched since a set's last call (176 MB) exceed the 129 MB L2."""
    T = ACR_SEQ * ACR_LEN
    host, sets = zip(*(acr_inputs(q, j) for j in range(3)))
    ws = q.acr_workspace()
    R = 21

    def calls():
        for i in range(R):
            acr_call(q, sets[i % 3], ws)

    g, nl = graph_of(calls, q)
    g.replay()
    us = time_graph(g, 5, stream) / R * 1e3
    q.qurl_check_device_status()
    gbs = acr_bytes(T) / (us * 1e-6) / 1e9
    stats = sets[0]["stats"].cpu().tolist()
    out = {"workload": f"{ACR_SEQ} responses x {ACR_LEN} token slots (lengths uniform in [{ACR_LEN // 8}, {ACR_LEN}]), "
                       f"ACR, eps={ACR_EPS}, C={ACR_C}; dterm written, term not",
           "tokens": T, "valid_tokens": int(stats[1]), "us_per_call": us, "launches_per_call": nl // R,
           "tokens_per_s": T / (us * 1e-6),
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": gbs / pk["hbm_gbs"], "traffic": traffic_from_profile(ACR_PROFILE, ACR_SOURCES),
                        "peak_source": f"{pk['source']} HBM copy",
                        "timing": f"CUDA events around a graph of {R} calls (one kernel a call) rotating over "
                                  "three input sets (264 MB > L2); bytes = 21 per token slot"},
           "stats": dict(zip(q.ACR_STATS, stats))}
    if cpu_baseline:
        import oracle

        oracle.build()
        r = host[0]
        t0 = time.perf_counter()
        oracle.acr_objective(*(r[k] for k in ACR_KEYS), eps=ACR_EPS, C=ACR_C, adaptive=True)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": T / dt, "unit": "token slots/s", "cores": 1, "kind": "oracle",
                               "sample": f"the whole mini-batch ({T} slots) once, single-threaded C, {dt:.2f} s"}
    return out


def time_kv_cache(q, stream, pk, l2):
    """FP8 key/value cache quantization of the 32B-class qkv output at M = 8192
    tokens (8 KV heads of 128) into a paged cache through a shuffled slot
    mapping; a graph of calls rotating over enough qkv outputs that the key and
    value columns read exceed 2 x L2.  Bytes per token: the keys and values in
    (bf16), their codes and fp32 scales out, the slot index."""
    model, M = "32b", 8192
    hid = MODELS[model]["hidden"]
    kvh, hd = 8, 128
    N = MODELS[model]["shapes"]["qkv"][1]
    per_token = 2 * kvh * hd * 2 + 2 * kvh * hd + 2 * kvh * 4 + 8
    k = min(n_sets(M * 2 * kvh * hd * 2, l2), 16)
    base = synth.activations("bench/kv/qkv", M, N).cuda()
    ins = [torch.roll(base, i * 13, 0).contiguous() for i in range(k)]
    S = 2 * M
    slots = torch.from_numpy(np.random.Generator(np.random.PCG64(5)).permutation(S)[:M].astype(np.int64)).cuda()
    caches = q.kv_cache(S, kvh, hd)
    R = max(k, 8)

    def calls():
        for r in range(R):
            q.qurl_kv_cache_quant(ins[r % k], hid, kvh, hd, slots, *caches)

    g, nl = graph_of(calls, q)
    g.replay()
    us = time_graph(g, 5, stream) / R * 1e3
    q.qurl_check_device_status()
    nb = per_token * M
    return {"workload": f"32B-class qkv output, M = {M} tokens, {kvh} KV heads of {hd}, per-token-per-head FP8 "
                        "scales, paged cache through a shuffled slot mapping",
            "us_per_call": us, "tokens_per_s": M / (us * 1e-6), "launches_per_call": nl // R,
            "roofline": {"bound": "hbm", "achieved": nb / (us * 1e-6) / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": nb / (pk["hbm_gbs"] * 1e9) / (us * 1e-6),
                         "timing": f"CUDA events around a graph of {R} calls rotating over {k} inputs"}}


def nvfp4_bytes(M, K, N):
    """Algorithmic bytes of one 4-bit linear: codes (half a byte a value) and block scales (one byte per 16
    values) of both operands, fp32 row scales, bf16 Y."""
    return (M + N) * K // 2 + (M + N) * K // 16 + 4 * (M + N) + 2 * M * N


def time_nvfp4(q, stream, pk, l2):
    """The 4-bit (NVFP4, W4A4) variant on the 32B-class projections: each
    linear on its own (graph of calls rotating over enough weight sets, each
    with its fp16 copy attached), and the row quantizer on activations and on
    fp32 weights.  The GEMM runs on the fp16 tensor pipe (exact widening of the
    E2M1 x E4M3 values): its roofline is the measured bf16 = fp16 dense rate;
    the nominal FP4 rate (6x bf16) is reported beside it."""
    model = "32b"
    res = {"per_linear": {}}
    for name, K, N in chain_shapes(model):
        W = synth.weights(f"bench/nvfp4/{name}/W", N, K).cuda()
        w0 = q.nvfp4_quant(W)
        del W
        k = n_sets(N * K * 2, l2)  # the GEMM reads the weights' fp16 copy (attached, as for INT8)
        sets = [w0] + [tuple(torch.roll(t, (i * 1009) % N, 0).contiguous() for t in w0) for i in range(1, k)]
        wides = [q.nvfp4_wide_weights(t) for t in sets]
        for M in (256, 8192):
            x = q.nvfp4_quant(synth.activations(f"bench/nvfp4/{name}/X/{M}", M, K).cuda(), S_UAQ)
            ws = q.nvfp4_workspace(M, N, K)
            Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            R = max(k, 4)

            def calls(x=x, ws=ws, Y=Y, R=R):
                for r in range(R):
                    q.qurl_nvfp4_linear(x, sets[r % len(sets)], Y, ws)

            g, nl = graph_of(calls, q)
            g.replay()
            us = time_graph(g, 3, stream) / R * 1e3
            ops = 2 * M * N * K
            t_fp16 = ops / (pk["bf16_tflops"] * 1e12)
            nb = nvfp4_bytes(M, K, N)
            t_h = nb / (pk["hbm_gbs"] * 1e9)
            res["per_linear"][f"{name}/M{M}"] = {
                "M": M, "K": K, "N": N, "us": us, "TOPS": ops / (us * 1e-6) / 1e12, "launches": nl // R,
                "frac_fp16_path": max(t_fp16, t_h) / (us * 1e-6),
                "frac_nvfp4_nominal": max(t_fp16 / 6, t_h) / (us * 1e-6), "weight_sets": k}
            del g, x, ws, Y
        del wides, sets, w0
        torch.cuda.empty_cache()
    # the row quantizer: activations (bf16, M = 8192, K = 5120) and the gate_up weights (fp32 W')
    for what, R_, K_, f32 in (("act/M8192/K5120", 8192, 5120, False), ("weights/gate_up", 55296, 5120, True)):
        src = (synth.weights("bench/nvfp4/qw", R_, K_) if f32 else synth.activations("bench/nvfp4/qa", R_, K_)).cuda()
        out = q.nvfp4_quant(src)

        def qcalls(src=src, out=out):
            for _ in range(4):
                q.qurl_nvfp4_quant(src, 1.0, *out)

        g, _ = graph_of(qcalls, q)
        g.replay()
        us = time_graph(g, 3, stream) / 4 * 1e3
        nb = R_ * K_ * (4 if f32 else 2) + R_ * K_ // 2 + R_ * K_ // 16 + 4 * R_
        res[f"quant/{what}"] = {"us": us, "GBps": nb / (us * 1e-6) / 1e9,
                                "roofline_frac": nb / (pk["hbm_gbs"] * 1e9) / (us * 1e-6)}
        del g, src, out
        torch.cuda.empty_cache()
    q.qurl_check_device_status()
    return res


def time_tensor_routes(q, stream, pk):
    """The rate of each tensor route an 8-bit product can take on this GPU, from
    the library's probe kernels (fixed instruction counts on zero operands),
    timed with CUDA events: which route INT8 should take, and what its roofline
    divides by."""
    nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    routes = {0: ("mma.sync.m16n8k32 s8*s8->s32 (warp MMA)", 4 * nsm, 20000),
              1: ("tcgen05.mma kind::f16 fp16*fp16->fp32, M128 N256 K16, operands in shared memory", nsm, 20000),
              2: ("tcgen05.mma kind::f16, A in tensor memory", nsm, 20000),
              3: ("tcgen05.mma kind::f8f6f4 e4m3*e4m3->fp32, M128 N256 K32", nsm, 20000)}
    out = {}
    for r, (name, ctas, iters) in routes.items():
        q.qurl_debug_mma_probe(r, ctas, 100, stream)  # warm (module load, TMEM)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ops = q.qurl_debug_mma_probe(r, ctas, iters, stream)
        b.record(stream)
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        out[f"route{r}"] = {"instruction": name, "ctas": ctas, "TOPS": ops / (ms * 1e-3) / 1e12,
                            "frac_of_bf16_peak": ops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"]}
    q.qurl_check_device_status()
    best = max(("route0", "route1", "route2"), key=lambda k: out[k]["TOPS"])
    out["int8_best"] = best
    out["note"] = ("INT8 codes are exact in fp16, so route 1/2 multiply them exactly; the INT8 roofline divides by "
                   "the measured bf16 (= fp16) dense rate")
    return out


# ------------------------------------------------------------------ CPU oracle leg

def oracle_chain(oracle, oq, prepared, hid, X_bits, nthreads):
    """The chain for a subset of the tokens, on the CPU oracle."""
    xq, sx, _, _ = oracle.rmsnorm_quant(X_bits, prepared["qkv"][2], oq, eps=EPS)
    y, _ = oracle.w8a8_linear(xq, sx, prepared["qkv"][0], prepared["qkv"][1], oq, nthreads)
    xq, sx = oracle.quant_act(np.ascontiguousarray(y[:, :hid]), oq, pre_scale=S_UAQ)
    y, _ = oracle.w8a8_linear(xq, sx, prepared["o_proj"][0], prepared["o_proj"][1], oq, nthreads)
    xq, sx, _, _ = oracle.rmsnorm_quant(y, prepared["gate_up"][2], oq, eps=EPS)
    y, _ = oracle.w8a8_linear(xq, sx, prepared["gate_up"][0], prepared["gate_up"][1], oq, nthreads)
    xq, sx, _ = oracle.silu_mul_quant(y, oq, pre_scale=S_UAQ)
    y, _ = oracle.w8a8_linear(xq, sx, prepared["down"][0], prepared["down"][1], oq, nthreads)
    return y


def oracle_prepare(oracle, oq, model, W, gammas):
    out = {}
    for name, _, _ in chain_shapes(model):
        g = gammas.get(name)
        Wq, sw, gf, _ = oracle.prepare_weights(W[name].numpy(), oq, s=S_UAQ, gamma=None if g is None else g.numpy())
        out[name] = (Wq, sw, gf)
    return out


class OracleStep:
    """The oracle on a bounded sample of the headline step: `tokens` tokens of the
    32B-class chain in each 8-bit type (weights prepared once, not timed)."""

    def __init__(self, oracle, tokens):
        self.oracle = oracle
        self.tokens = tokens
        self.nthreads = os.cpu_count() or 1
        model = HEADLINE[0]
        W, gammas = make_weights(model)
        self.prepared = {qtype: oracle_prepare(oracle, oracle.INT8 if qtype == "int8" else oracle.FP8_E4M3, model,
                                               W, gammas) for qtype in QTYPES}
        del W
        self.X = synth.bf16_bits(synth.activations(input_name(model, "oracle"), tokens, MODELS[model]["hidden"]))
        self.ops = len(QTYPES) * chain_ops(model, [tokens])

    def run(self, n=None):
        X = self.X if n is None else self.X[:n]
        for qtype in QTYPES:
            oq = self.oracle.INT8 if qtype == "int8" else self.oracle.FP8_E4M3
            oracle_chain(self.oracle, oq, self.prepared[qtype], MODELS[HEADLINE[0]]["hidden"], X, self.nthreads)

    def describe(self, dt):
        return (f"oracle chain (all four 32B-class projections at full N and K) on {self.tokens} of the step's "
                f"{sum(HEADLINE[1])} tokens per 8-bit type, INT8 and FP8: {self.ops / 1e9:.1f} GOP in {dt:.2f} s; "
                "per-token work is independent, so ops/s scale to the whole step")


# ------------------------------------------------------------------ arms

def run_reference(args):
    rank, world = dist()
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    ref = OracleStep(oracle, args.ref_tokens)
    for _ in range(max(args.warmup, 0)):
        ref.run(2)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ref.run()
    dt = (time.perf_counter() - t0) / args.steps
    value = ref.ops / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8+fp8_e4m3", "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_step_per_qtype": args.ref_tokens},
            "cpu_baseline": {"value": value, "unit": "TOPS", "cores": min(ref.nthreads, args.ref_tokens),
                             "kind": "oracle", "sample": ref.describe(dt)},
            "e2e": {"value": value, "unit": "TOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    rank, world = dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    import w8a8_precision_gemm_gb300 as q

    q.load()
    pk = peaks()
    l2 = l2_bytes()
    stream = torch.cuda.current_stream()
    model, Ms = HEADLINE
    hid = MODELS[model]["hidden"]
    W, gammas = make_weights(model)
    layers = {qtype: Layer(q, qt_of(q, qtype), model, W, gammas) for qtype in QTYPES}
    del W
    passes = [(qtype, M) for qtype in QTYPES for M in Ms]
    bufs = {(qtype, M): Buffers(q, qt_of(q, qtype), model, M) for qtype, M in passes}
    X_host = {M: synth.activations(input_name(model, M), M, hid).pin_memory() for M in Ms}
    Y_host = {p: torch.empty((p[1], hid), dtype=torch.bfloat16).pin_memory() for p in passes}
    for (qtype, M), B in bufs.items():
        B.x.copy_(X_host[M])
    torch.cuda.synchronize()

    def step():
        for qtype, M in passes:
            chain(q, qt_of(q, qtype), layers[qtype], bufs[(qtype, M)])

    copy_stream = torch.cuda.Stream()

    def step_e2e():
        """Every pass's input goes host -> device on a copy stream (all of them
        while the first pass computes); each pass's output goes device -> host
        on the copy stream as soon as its chain ends, overlapping the next one."""
        main = torch.cuda.current_stream()
        copy_stream.wait_stream(main)
        landed = []
        with torch.cuda.stream(copy_stream):
            for p in passes:
                bufs[p].x.copy_(X_host[p[1]], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copy_stream)
                landed.append(ev)
        for p, ev in zip(passes, landed):
            main.wait_event(ev)
            chain(q, qt_of(q, p[0]), layers[p[0]], bufs[p])
            done = torch.cuda.Event()
            done.record(main)
            copy_stream.wait_event(done)
            with torch.cuda.stream(copy_stream):
                Y_host[p].copy_(bufs[p].y["down"], non_blocking=True)
        main.wait_stream(copy_stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    g_step, launches_step = graph_of(step, q)
    g_e2e, _ = graph_of(step_e2e, q)
    for _ in range(3):
        g_step.replay()
    torch.cuda.synchronize()

    # ---- the timed region: K steps back to back
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        # untimed lead-in: the same step replayed for CLOCK_LEAD s, so that clock samples next to a
        # short timed region see the GPU under this load
        t_lead = time.perf_counter()
        while time.perf_counter() - t_lead < CLOCK_LEAD:
            for _ in range(4):
                g_step.replay()
            torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t0_wall = time.perf_counter()
        torch.cuda.nvtx.range_push("timed_step")  # lets a profiler select the timed region's launches
        start.record(stream)
        for _ in range(args.steps):
            g_step.replay()
        end.record(stream)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        t1_wall = time.perf_counter()
        t_wall = t1_wall - t0_wall
        barrier(world)
    q.qurl_check_device_status()
    ops = len(QTYPES) * chain_ops(model, Ms)
    _, ms_step = job_throughput(ops, start.elapsed_time(end) / args.steps, world)

    # ---- end to end: H2D of X, the chain, D2H of the output, every step
    for _ in range(2):
        g_e2e.replay()
    e2e_ms = max_over_ranks(time_graph(g_e2e, args.steps, stream), world)
    h2d = sum(p[1] * hid * 2 for p in passes)
    d2h = h2d
    del g_e2e

    # ---- each qtype's chain on its own (the step's parts), with its roofline fractions
    by_qtype = {}
    for qtype in QTYPES:
        def part(qtype=qtype):
            for M in Ms:
                chain(q, qt_of(q, qtype), layers[qtype], bufs[(qtype, M)])

        g, nl = graph_of(part, q)
        g.replay()
        ms = time_graph(g, max(3, args.steps // 4), stream)
        t_g = sum(chain_roofline(model, M, qtype, pk)[0] for M in Ms)
        t_q = sum(chain_roofline(model, M, qtype, pk)[1] for M in Ms)
        by_qtype[qtype] = {"ms_per_step": ms, "TOPS": chain_ops(model, Ms) / (ms * 1e-3) / 1e12,
                           "launches_per_step": nl, "gemm_roofline_frac": t_g / (ms * 1e-3),
                           "step_roofline_frac": (t_g + t_q) / (ms * 1e-3),
                           "roofline_ms": {"gemms": t_g * 1e3, "quantizers": t_q * 1e3}}
        del g
    t_all = sum(sum(chain_roofline(model, M, qtype, pk)) for qtype, M in passes)
    t_all_g = sum(chain_roofline(model, M, qtype, pk)[0] for qtype, M in passes)
    step_roof = {"roofline_ms": t_all * 1e3, "frac": t_all / (ms_step * 1e-3),
                 "gemm_roofline_ms": t_all_g * 1e3, "gemm_frac": t_all_g / (ms_step * 1e-3),
                 "definition": "sum over the step's linears of max(2MNK / tensor peak, bytes / HBM) plus its "
                               "quantizers' bytes / HBM, divided by the measured step time"}
    del bufs
    torch.cuda.empty_cache()

    # ---- each GEMM and quantizer of the headline on its own
    per_gemm = {qtype: time_per_gemm(q, qtype, layers[qtype], model, Ms, stream, pk, l2) for qtype in QTYPES}
    per_quant = {qtype: time_per_quant(q, qtype, model, Ms, stream, pk, l2, gammas["qkv"]) for qtype in QTYPES}

    # ---- the dominant kernel of the step: the linear with the largest time share
    dom_q, dom_k = max(((qtype, key) for qtype in QTYPES for key in per_gemm[qtype]),
                       key=lambda t: per_gemm[t[0]][t[1]]["us"])
    d = per_gemm[dom_q][dom_k]
    if d["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": 2 * d["M"] * d["N"] * d["K"] / (d["us"] * 1e-6) / 1e12,
                "peak": tensor_peak(pk, dom_q), "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": d["GBps"], "peak": pk["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    prof = GEMM_PROFILES.get(d["kernel"])
    roof["traffic"] = traffic_from_profile(*prof) if prof else None
    if roof["traffic"] is not None:
        roof["traffic"] = int(roof["traffic"])
    roof["traffic_source"] = prof[0] if prof and roof["traffic"] is not None else None
    roof["kernel"] = f"{d['kernel']} {model} {dom_k} K={d['K']} N={d['N']} ({dom_q})"
    roof["peak_source"] = (f"{pk['source']} " + ("bf16 burst (INT8 runs on the fp16 tensor pipe, same dense rate)"
                                                if dom_q == "int8" else "bf16 burst x 2 (nominal fp8:bf16 ratio)")
                           if roof["bound"] == "tensor" else f"{pk['source']} HBM copy")
    roof["timing"] = (f"CUDA events around a graph of qurl_w8a8_linear calls rotating over {d['weight_sets']} "
                      f"weight sets; a call is {d['launches']} kernel(s)")
    del layers
    torch.cuda.empty_cache()

    # ---- the 7B-class chains: decode (M = 64, 256) and config-5 sizes (M = 512, 4096), plus the flip probe
    W7, g7 = make_weights("7b")
    decode_7b, chain_7b = {}, {}
    for qtype in QTYPES:
        qt = qt_of(q, qtype)
        layers7 = [Layer(q, qt, "7b", W7, g7, rotate=0), Layer(q, qt, "7b", W7, g7, rotate=1)]
        decode_7b[qtype] = time_chain_block(q, qtype, layers7, "7b", DECODE_7B[1], 20, stream, pk)
        decode_7b[qtype]["per_gemm"] = time_per_gemm(q, qtype, layers7[0], "7b", DECODE_7B[1], stream, pk, l2)
        chain_7b[qtype] = time_chain_block(q, qtype, layers7, "7b", CHAIN_7B[1], 10, stream, pk)
        del layers7
        torch.cuda.empty_cache()
    del W7
    flips, requant = flip_probe(q, "7b", stream, pk, l2)
    chain_7b["flips"] = flips
    q.qurl_check_device_status()

    # ---- the ACR token objective of the same RL step (beside the rollout's linear layers)
    acr = time_acr(q, stream, pk, rank == 0 and world == 1 and not args.no_cpu_baseline)
    routes = time_tensor_routes(q, stream, pk)
    kv = time_kv_cache(q, stream, pk, l2)
    nvfp4 = time_nvfp4(q, stream, pk, l2)

    value = ops * world / (ms_step * 1e-3) / 1e12
    step_bytes = sum(alg_bytes(M, K, N) for qtype, M in passes for _, K, N in chain_shapes(model))
    line = {"metric": METRIC, "value": value, "unit": "TOPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8+fp8_e4m3", "data": "synthetic",
            "config": {"workload": WORKLOAD, "qtypes": list(QTYPES), "M": list(Ms), "uaq_s": S_UAQ,
                       "parallelism": "replicas" if world > 1 else "single",
                       "launch": "one CUDA graph per step (six chain passes, 24 fused calls)",
                       "l2": "inputs larger than L2: 976 MB of weights per step; a projection's weights return "
                             "only after >= 450 MB of other weights (129 MB L2)"},
            "hbm_gbs": step_bytes * world / (ms_step * 1e-3) / 1e9, "wall_s": t_wall,
            "by_qtype": by_qtype, "step_roofline": step_roof,
            "roofline": roof,
            "e2e": {"value": ops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TOPS", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": launches_step * args.steps,
            "launches_per_step": launches_step,
            "clocks": clocks.summary(t0_wall, t1_wall, CLOCK_LEAD),
            "per_gemm": per_gemm, "per_quant": per_quant,
            "decode_7b": decode_7b, "chain_7b": chain_7b, "weight_requant": requant,
            "acr_objective": acr, "tensor_routes": routes, "kv_cache_fp8": kv, "nvfp4_w4a4": nvfp4}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        ref = OracleStep(oracle, args.ref_tokens)
        ref.run(2)
        t0 = time.perf_counter()
        ref.run()
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": ref.ops / dt / 1e12, "unit": "TOPS",
                                "cores": min(ref.nthreads, args.ref_tokens), "kind": "oracle",
                                "sample": ref.describe(dt)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_single(args):
    """One projection's W8A8 linear call, repeated -- a small, fixed launch
    sequence for profilers (e.g. ncu -k regex:w8a8_gemm -s 1 -c 1)."""
    import w8a8_precision_gemm_gb300 as q

    if args.single == "acr":
        _, d = acr_inputs(q, 0)
        ws = q.acr_workspace()
        for _ in range(args.single_reps):
            acr_call(q, d, ws)
        torch.cuda.synchronize()
        q.qurl_check_device_status()
        print(json.dumps({"single": "acr", "tokens": ACR_SEQ * ACR_LEN, "reps": args.single_reps}))
        return 0
    model, proj = args.single.split(":")
    M = args.single_m
    qt = qt_of(q, args.qtype)
    if proj in ("rmsnorm_quant", "quant_act", "silu_mul_quant"):
        K = MODELS[model]["inter"] if proj == "silu_mul_quant" else MODELS[model]["hidden"]
        cols = 2 * K if proj == "silu_mul_quant" else K
        X = synth.activations(f"single/{model}/{proj}/X", M, cols).cuda()
        Xq = torch.empty((M, K), dtype=q.code_dtype(qt), device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        gf = (synth.gamma(f"single/{model}/g", K) * S_UAQ).cuda()
        for _ in range(args.single_reps):
            if proj == "rmsnorm_quant":
                q.qurl_rmsnorm_quant(X, gf, EPS, qt, Xq, sx)
            elif proj == "quant_act":
                q.qurl_quant_act(X, S_UAQ, qt, Xq, sx)
            else:
                q.qurl_silu_mul_quant(X, S_UAQ, qt, Xq, sx)
        torch.cuda.synchronize()
        q.qurl_check_device_status()
        print(json.dumps({"single": args.single, "M": M, "K": K, "qtype": args.qtype, "reps": args.single_reps}))
        return 0
    K, N = MODELS[model]["shapes"][proj]
    W = synth.weights(f"single/{model}/{proj}/W", N, K).cuda()
    Wq, sw, _, _ = q.prepare_weights(W, qt, s=S_UAQ, keep_scaled=False)
    del W
    wide = q.wide_weights(Wq) if qt == q.INT8 else None  # as the benchmark's layers keep it
    Xq, sx = q.quant_act(synth.activations(f"single/{model}/{proj}/X", M, K).cuda(), qt)
    ws = q.workspace(M, N, K, qt)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for _ in range(args.single_reps):
        q.qurl_w8a8_linear(Xq, sx, Wq, sw, qt, Y, ws)
    torch.cuda.synchronize()
    q.qurl_check_device_status()
    print(json.dumps({"single": args.single, "M": M, "K": K, "N": N, "qtype": args.qtype, "reps": args.single_reps}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-tokens", type=int, default=32,
                    help="tokens per 8-bit type in one oracle step (reference arm and cpu_baseline)")
    ap.add_argument("--single", default=None,
                    help="model:proj, e.g. 32b:gate_up -- run one linear for profiling (or one quantizer: "
                         "32b:rmsnorm_quant, 32b:quant_act, 32b:silu_mul_quant); 'acr': the ACR objective")
    ap.add_argument("--qtype", choices=list(QTYPES), default="int8", help="qtype of --single")
    ap.add_argument("--single-m", type=int, default=256)
    ap.add_argument("--single-reps", type=int, default=3)
    args = ap.parse_args()
    if args.single:
        return run_single(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
