"""The C-ABI library builds, loads without a GPU, exports every entry point the
public header declares, and rejects bad arguments on the host before any launch
(no compute call is made here)."""
import ctypes
import os
import re
import subprocess

import pytest

import w8a8_precision_gemm_gb300 as q
from w8a8_precision_gemm_gb300 import _build


@pytest.fixture(scope="module")
def L():
    _build.build()
    return q.load()


def test_header_declares_the_boundary():
    names = q.exported_names()
    for required in ("qurl_prepare_weights", "qurl_quant_act", "qurl_w8a8_linear", "qurl_rmsnorm_quant_linear",
                     "qurl_rmsnorm_quant", "qurl_silu_mul_quant", "qurl_w8a8_gemm_acc", "qurl_count_diff",
                     "qurl_workspace_size", "qurl_check_device_status", "qurl_status_string", "qurl_version",
                     "qurl_acr_objective", "qurl_acr_workspace_size"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in q.exported_names():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_plain_c_client_compiles_links_and_calls(L, tmp_path):
    """The header is strict C99 and a C program links libqurl and calls the
    entry points that need no device (version, sizes, status strings, and an
    argument error returned before any launch)."""
    src = tmp_path / "client.c"
    src.write_text(
        '#include <stdio.h>\n#include "qurl.h"\n'
        "int main(void) {\n"
        "  const int v = qurl_version();\n"
        "  const size_t ws = qurl_acr_workspace_size();\n"
        "  const qurl_status e = qurl_quant_act(0, 4, 256, 256, 1.0f, QURL_INT8, 0, 0, 0);\n"
        '  printf("%d %zu %s %d\\n", v, ws, qurl_status_string(e), (int)e);\n'
        "  return (v > 0 && ws > 0 && e == QURL_ERR_INVALID_ARG) ? 0 : 1;\n"
        "}\n")
    exe = tmp_path / "client"
    libdir = os.path.dirname(_build.LIB)
    subprocess.run(["cc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.dirname(q.HEADER),
                    str(src), "-L", libdir, "-lqurl", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert out == [str(L.qurl_version()), str(L.qurl_acr_workspace_size()), "QURL_ERR_INVALID_ARG", "1"]


def test_header_entry_points_are_extern_c():
    text = open(q.HEADER).read()
    assert 'extern "C"' in text
    # no torch / C++ types in the declarations (comments stripped)
    code = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    assert not re.search(r"\b(torch|at::|std::|Tensor)\b", code)


def test_status_strings_and_version(L):
    assert L.qurl_status_string(0) == b"QURL_OK"
    assert L.qurl_status_string(6) == b"QURL_ERR_TIMEOUT"
    assert L.qurl_status_string(99) == b"QURL_ERR_UNKNOWN"
    assert L.qurl_version() == 102


FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced: calls fail validation first
FAKE_ODD = ctypes.c_void_p(0x10008)  # 8-byte aligned only


def test_quant_act_validation(L):
    assert L.qurl_quant_act(None, 4, 256, 256, 1.0, 0, FAKE, FAKE, None) == 1       # null X
    assert L.qurl_quant_act(FAKE, 0, 256, 256, 1.0, 0, FAKE, FAKE, None) == 1       # M = 0
    assert L.qurl_quant_act(FAKE, 4, 256, 128, 1.0, 0, FAKE, FAKE, None) == 1       # ldx < K
    assert L.qurl_quant_act(FAKE, 4, 250, 256, 1.0, 0, FAKE, FAKE, None) == 2       # K % 16
    assert L.qurl_quant_act(FAKE_ODD, 4, 256, 256, 1.0, 0, FAKE, FAKE, None) == 3   # alignment
    assert L.qurl_quant_act(FAKE, 4, 256, 260, 1.0, 0, FAKE, FAKE, None) == 3       # row stride not 16 B
    assert L.qurl_quant_act(FAKE, 4, 256, 256, 1.0, 7, FAKE, FAKE, None) == 1       # bad qtype
    assert L.qurl_quant_act(FAKE, 4, 256, 256, float("nan"), 0, FAKE, FAKE, None) == 1


def test_linear_validation(L):
    f = L.qurl_w8a8_linear
    assert f(None, FAKE, FAKE, FAKE, 4, 8, 256, 0, FAKE, 8, None, 0, None) == 1
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 8, 250, 0, FAKE, 8, None, 0, None) == 2
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 8, 256, 0, FAKE, 4, None, 0, None) == 1     # ldy < N
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 8, 256, 0, FAKE_ODD, 8, None, 0, None) == 3
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 8, 256, 0, FAKE, 12, None, 0, None) == 3    # ldy * 2 % 16
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 8, 256, 0, FAKE, 8, None, 64, None) == 1    # ws bytes without ws
    assert f(FAKE, FAKE, FAKE, FAKE, 4, 8, 256, 2, FAKE, 8, None, 0, None) == 1     # bad qtype
    assert L.qurl_w8a8_gemm_acc(FAKE, FAKE, 4, 8, 256, 0, None, None, 0, None) == 1


def test_prepare_weights_validation(L):
    f = L.qurl_prepare_weights
    assert f(FAKE, 0, 8, 256, 256, None, 0.0, 0, FAKE, FAKE, None, None, None) == 1     # s = 0
    assert f(FAKE, 0, 8, 256, 256, None, float("inf"), 0, FAKE, FAKE, None, None, None) == 1
    assert f(FAKE, 0, 8, 256, 256, FAKE, 1.5, 0, FAKE, FAKE, None, None, None) == 1     # gamma without out
    assert f(FAKE, 3, 8, 256, 256, None, 1.5, 0, FAKE, FAKE, None, None, None) == 1     # bad w_type
    assert f(FAKE, 0, 8, 248, 248, None, 1.5, 0, FAKE, FAKE, None, None, None) == 2     # K % 16
    assert f(FAKE, 0, 8, 256, 260, None, 1.5, 0, FAKE, FAKE, None, None, None) == 3     # bf16 ldw
    # W' may alias W only for a dense fp32 W
    assert f(FAKE, 0, 8, 256, 256, None, 1.5, 0, FAKE, FAKE, None, FAKE, None) == 1


def test_other_validation(L):
    assert L.qurl_silu_mul_quant(FAKE, 4, 100, 200, 1.0, 0, FAKE, FAKE, None, None) == 2   # I % 16
    assert L.qurl_silu_mul_quant(FAKE, 4, 128, 200, 1.0, 0, FAKE, FAKE, None, None) == 1   # ld < 2I
    assert L.qurl_rmsnorm_quant(FAKE, 4, 256, 256, None, 1e-6, 0, FAKE, FAKE, None, None) == 1
    assert L.qurl_rmsnorm_quant(FAKE, 4, 256, 256, FAKE, -1.0, 0, FAKE, FAKE, None, None) == 1
    assert L.qurl_count_diff(FAKE, None, 16, FAKE, None) == 1
    assert L.qurl_count_diff(FAKE_ODD, FAKE, 16, FAKE, None) == 3
    assert L.qurl_rmsnorm_quant_linear(FAKE, 256, FAKE, 1e-6, FAKE, FAKE, 4, 8, 256, 0, FAKE, 8, FAKE, None,
                                       None, 0, None) == 1


def test_acr_objective_validation(L):
    ws = L.qurl_acr_workspace_size()
    assert ws >= 1024 * 64
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE)
    acr = L.qurl_acr_objective
    assert acr(*ok, 100, 0.2, 2.0, 1, None, FAKE, None, FAKE, ws, None) == 1      # stats NULL
    assert acr(*ok, 100, 0.2, 2.0, 1, None, FAKE, FAKE, None, ws, None) == 1      # workspace NULL
    assert acr(None, *ok[1:], 100, 0.2, 2.0, 1, None, FAKE, FAKE, FAKE, ws, None) == 1  # logp NULL, T > 0
    assert acr(*ok, -1, 0.2, 2.0, 1, None, FAKE, FAKE, FAKE, ws, None) == 1       # T < 0
    assert acr(*ok, 100, 0.0, 2.0, 1, None, FAKE, FAKE, FAKE, ws, None) == 1      # eps out of (0, 1)
    assert acr(*ok, 100, 1.0, 2.0, 1, None, FAKE, FAKE, FAKE, ws, None) == 1
    assert acr(*ok, 100, 0.2, 0.0, 1, None, FAKE, FAKE, FAKE, ws, None) == 1      # C <= 0
    assert acr(*ok, 100, 0.2, float("nan"), 1, None, FAKE, FAKE, FAKE, ws, None) == 1
    assert acr(*ok, 100, 0.2, 2.0, 2, None, FAKE, FAKE, FAKE, ws, None) == 1      # adaptive not 0 / 1
    assert acr(*ok, 100, 0.2, 2.0, 1, None, FAKE, FAKE, FAKE, ws - 1, None) == 4  # workspace too small
    assert acr(FAKE_ODD, *ok[1:], 100, 0.2, 2.0, 1, None, FAKE, FAKE, FAKE, ws, None) == 3
    assert acr(*ok, 100, 0.2, 2.0, 1, FAKE_ODD, FAKE, FAKE, FAKE, ws, None) == 3  # term misaligned
    assert acr(*ok, 100, 0.2, 2.0, 1, None, FAKE, ctypes.c_void_p(0x10004), FAKE, ws, None) == 3  # stats % 8


def test_workspace_size_without_gpu(L):
    # sized for the SM count of the device (or the largest target when none is visible)
    assert L.qurl_workspace_size(0, 8, 256, 0) == 0
    ws = L.qurl_workspace_size(64, 4608, 3584, 1)  # FP8 decode: split-K partials and the handoff counters
    assert ws > 256 and (ws - 256) % (64 * 4608 * 4) == 0
    assert L.qurl_workspace_size(8192, 55296, 5120, 1) == 256  # prefill fills the GPU without splitting K


def _tile_widths(p):
    """(token tile width, channel tile width) of a plan."""
    pair = p["kernel"] in (2, 3, 4)
    if p["swap"]:
        return p["bn"], (256 if pair else 128)
    return (256 if pair else 128), p["bn"]


@pytest.mark.parametrize("M,N,K,qt,kernel", [
    # INT8 with its workspace: the TMEM-operand kernel; from 2048 tokens on, and
    # where 256 x 256 pair units would fill their waves, CTA pairs with both
    # operands widened in the workspace
    (64, 37888, 3584, 0, 1), (256, 37888, 3584, 0, 1), (256, 4608, 3584, 0, 1),
    (1536, 8192, 4096, 0, 4), (2000, 4000, 4000, 0, 4),
    (4096, 37888, 3584, 0, 4), (4096, 3584, 18944, 0, 4), (8192, 7168, 5120, 0, 4), (2048, 256, 16384, 0, 4),
    (1024, 7168, 5120, 0, 1), (1024, 5120, 27648, 0, 1),
    # FP8: pairs for prefill and for the larger decode shapes
    (64, 37888, 3584, 1, 0), (256, 4608, 3584, 1, 0), (256, 37888, 3584, 1, 3),
    (256, 3584, 18944, 1, 3), (4096, 37888, 3584, 1, 3), (300, 520, 2048, 1, 3),
])
def test_plan_routing_and_coverage(M, N, K, qt, kernel):
    """The kernel each shape is routed to (the choices the measurements made) and
    that every plan's tiles and K splits cover the problem exactly once."""
    import w8a8_precision_gemm_gb300 as q

    p = q.plan(M, N, K, qt, 152)
    assert p["kernel"] == kernel, p
    tw, cw = _tile_widths(p)
    assert (p["tiles_tok"] - 1) * tw < M <= p["tiles_tok"] * tw
    assert (p["tiles_ch"] - 1) * cw < N <= p["tiles_ch"] * cw
    bk = 256 if p["kernel"] in (1, 2) else (64 if qt == 0 else 128)
    if p["kernel"] == 4:
        assert p["kb_per_split"] % 4 == 0 or p["splits"] == 1  # split ranges hold whole 256-code sum ranges
    num_kb = -(-K // bk)
    assert (p["splits"] - 1) * p["kb_per_split"] < num_kb <= p["splits"] * p["kb_per_split"]


def _check_schedule(p, K, qt, slots):
    """A plan's units cover every tile's K range once: all tiles split, or the
    first whole_units whole (full rounds of SM pairs) and the rest split."""
    tiles = p["tiles_tok"] * p["tiles_ch"]
    bk = 64 if (qt == 0 and p["kernel"] == 4) else (256 if p["kernel"] in (1, 2) else (64 if qt == 0 else 128))
    num_kb = -(-K // bk)
    assert (p["splits"] - 1) * p["kb_per_split"] < num_kb <= p["splits"] * p["kb_per_split"]
    w = p["whole_units"]
    if w:
        assert p["kernel"] in (3, 4) and not p["swap"] and p["splits"] >= 2
        assert 0 < w < tiles and w % slots == 0
        assert tiles - w < slots  # the split tail is the last round's tiles alone
        units = w + (tiles - w) * p["splits"]
        assert units > tiles


@pytest.mark.parametrize("qt", [0, 1])
@pytest.mark.parametrize("attached", [False, True])
def test_plan_split_tails_cover_every_tile(L, qt, attached):
    """Over a sweep of prefill shapes and SM counts, every plan with a split
    tail keeps whole rounds of whole-K units and covers K once per tile; and the
    32B-class projections take the schedules measured fastest on 152 SMs."""
    import w8a8_precision_gemm_gb300 as q

    for sms in (132, 148, 152, 160):
        for M in (300, 777, 1024, 2048, 4096, 8192):
            for N, K in ((7168, 5120), (5120, 5120), (55296, 5120), (5120, 27648), (3584, 18944), (5000, 12288)):
                _check_schedule(q.plan(M, N, K, qt, sms, attached=attached), K, qt, sms // 2)
    if attached and qt == 0:  # INT8 with persistent fp16 weight copies, as the benchmark's layers keep them
        expect = {(1024, 5120, 5120): 76, (1024, 7168, 5120): 0, (1024, 5120, 27648): 76, (8192, 5120, 27648): 608,
                  (8192, 55296, 5120): 0}
    elif qt == 1:
        expect = {(1024, 5120, 5120): 0, (1024, 5120, 27648): 76, (8192, 5120, 27648): 608, (8192, 55296, 5120): 0}
    else:
        expect = {}
    for (M, N, K), w in expect.items():
        p = q.plan(M, N, K, qt, 152, attached=attached)
        assert p["whole_units"] == w, ((M, N, K), p)


def test_plan_workspace_and_fallbacks(L):
    import ctypes
    import w8a8_precision_gemm_gb300 as q

    # the plan's workspace is what qurl_workspace_size reports (160 SMs without a device) -- for INT8
    # above 256 tokens (and from 129 tokens for weights of 2^26 codes or more) at least that, and enough
    # for the CTA-pair plan of weights with an attached fp16 copy: the activations' fp16 copy, one
    # 256 x 128 int32 region per SM, the counters
    for M, N, K, qt in ((64, 4608, 3584, 0), (256, 4608, 3584, 0), (64, 3584, 18944, 1), (4096, 3584, 3584, 0),
                        (256, 4608, 3584, 1)):
        assert q.plan(M, N, K, qt, 160)["ws_bytes"] == L.qurl_workspace_size(M, N, K, qt)
    for M, N, K in ((512, 37888, 3584), (1024, 7168, 5120), (256, 37888, 3584)):
        ws = L.qurl_workspace_size(M, N, K, 0)
        assert ws == max(q.plan(M, N, K, 0, 160)["ws_bytes"], q.plan(M, N, K, 0, 160, attached=True)["ws_bytes"])
        assert ws >= M * K * 2 + 160 * 256 * 128 * 4 + 256
    # no workspace: INT8 widens both operands in shared memory and K is not split
    p = q.plan(64, 4608, 3584, 0, 152, ws_bytes=0)
    assert p["kernel"] == 0 and p["splits"] == 1 and p["ws_bytes"] == 256  # (a fused call wants the counters)
    # a workspace too small for split partials keeps the TMEM kernel unsplit (fp16 codes, their
    # sums, and one 128 x 128 int32 running-sum region per SM)
    act = 64 * 3584 * 2 + 256 + 152 * 128 * 128 * 4 + 256  # ... and the handoff counters
    p = q.plan(64, 4608, 3584, 0, 152, ws_bytes=act)
    assert p["kernel"] == 1 and p["splits"] == 1 and p["ws_bytes"] <= act
    # without room for the running sums: both operands widened in shared memory
    assert q.plan(64, 4608, 3584, 0, 152, ws_bytes=act - 1024)["kernel"] == 0
    # a workspace too small to widen the weights keeps the CTA-pair kernel with the weights in TMEM
    wide = q.plan(1536, 8192, 4096, 0, 152)
    assert wide["kernel"] == 4
    assert q.plan(1536, 8192, 4096, 0, 152, ws_bytes=wide["ws_bytes"] - 1)["kernel"] == 2
    out = (ctypes.c_longlong * 8)()
    assert L.qurl_debug_plan(64, 4608, 3584, 0, 0, 0, out) == 1
    assert L.qurl_debug_plan(64, 4608, 3584, 7, 152, 0, out) == 1
    assert L.qurl_debug_plan(64, 4608, 3584, 0, 152, 0, None) == 1
    assert L.qurl_debug_plan_ex(64, 4608, 3584, 0, 0, 0, 1, out) == 1
    assert L.qurl_debug_plan_ex(64, 4608, 3584, 0, 152, 0, 0, None) == 1
