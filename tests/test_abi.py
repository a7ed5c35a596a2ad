"""Host-side checks of the C library (no GPU needed, no kernel launched).

* the library loads and exports every function that include/mxfp8.h declares;
* size helpers match the pages' formulas (8x4 scale buffer: prhub summary of
  vLLM PR #52204, key source snippets; N padded to 128: vLLM PR #52204);
* argument checks return their status before touching the device
  (K % 256 != 0 is the load-time error of process_weights_after_loading).
"""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def mx():
    import __graft_entry__
    __graft_entry__.build()
    import mxfp8_block_scaled_x4_gb300 as m
    return m


def declared_functions():
    names = []
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*[\w\s\*]+?\b(mxfp8_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mxfp8_prepare_weight", "mxfp8_quantize_act", "mxfp8_linear",
                     "mxfp8_gemm", "mxfp8_grouped_linear", "mxfp8_act_scale_bytes",
                     "mxfp8_moe_route", "mxfp8_prepare_gate_up_weight", "mxfp8_moe_gate_up_swiglu",
                     "mxfp8_moe_finalize", "mxfp8_moe_expert_mlp", "mxfp8_autotune_linear",
                     "mxfp8_tactic_set", "mxfp8_tactic_get"):
        assert required in names


def test_library_exports_every_declared_symbol(mx):
    lib = ctypes.CDLL(mx.library_path())
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_size_helpers(mx):
    for m in (0, 1, 7, 8, 9, 16, 129):
        for k in (256, 512, 2048, 8192):
            kb = k // 32
            assert mx.act_scale_bytes(m, k) == math.ceil(m / 8) * 8 * math.ceil(kb / 4) * 4
            ws = mx.linear_workspace_bytes(m, k)
            assert ws == (m * k + 255) // 256 * 256 + mx.act_scale_bytes(m, k)
    assert mx.weight_bytes(130, 256) == 256 * 256
    assert mx.weight_scale_bytes(130, 256) == 256 * 8
    assert mx.weight_bytes(5120, 2048) == 5120 * 2048
    assert mx.act_scale_bytes(-1, 256) == 0
    assert mx.weight_bytes(0, 256) == 0
    # beyond the library's limits (rows < 2^31 - 256, K <= 2^20): invalid, no overflow
    lib = mx.library()
    big = 1 << 62
    assert mx.act_scale_bytes(big, 256) == 0 and mx.linear_workspace_bytes(big, 256) == 0
    assert mx.linear_workspace_bytes(16, 1 << 40) == 0
    assert mx.weight_bytes(big, 256) == 0 and mx.weight_scale_bytes(130, 1 << 40) == 0
    assert lib.mxfp8_linear_host_workspace_bytes(16, big, 2048) == 0
    assert lib.mxfp8_act_scale_bytes_128x4(big, 256) == 0
    assert lib.mxfp8_linear_128x4_workspace_bytes(16, 1 << 40) == 0
    assert lib.mxfp8_moe_route_workspace_bytes(big, 128, 8) == 0
    assert lib.mxfp8_moe_workspace_bytes(256, 128, 8, 1 << 40, 768) == 0
    # the largest valid shapes still give exact sizes
    m_max = (1 << 31) - 256
    assert mx.act_scale_bytes(m_max, 256) == m_max * 8
    assert mx.linear_workspace_bytes(m_max, 1 << 20) == m_max * (1 << 20) + m_max * (1 << 15)


def test_status_strings(mx):
    lib = mx.library()
    for s in range(8):
        assert lib.mxfp8_status_string(s)
    assert b"256" in lib.mxfp8_status_string(2)
    assert mx.status_string(5) == "workspace too small"
    assert isinstance(mx.last_cuda_error(), int) and mx.last_cuda_error() >= 0
    assert mx.act_scale_bytes_128x4(130, 256) == 256 * 8
    assert mx.linear_128x4_workspace_bytes(130, 256) == 130 * 256 + 256 * 8


def _view(mx, e, n, k, q, sf):
    w = mx.mxfp8_weight()
    st = mx.library().mxfp8_weight_view(ctypes.byref(w), e, n, k, q, sf)
    return st, w


def test_weight_view_checks(mx):
    A = 1 << 20  # fake, aligned addresses: never dereferenced by the view
    st, w = _view(mx, 1, 130, 256, A, A)
    assert st == 0 and w.n_pad == 256
    assert _view(mx, 1, 130, 320, A, A)[0] == 2          # K % 256
    assert _view(mx, 1, 130, 256, A + 8, A)[0] == 3      # misaligned data
    assert _view(mx, 1, 130, 256, A, A + 4)[0] == 3      # misaligned scales
    assert _view(mx, 0, 130, 256, A, A)[0] == 1          # no experts
    assert _view(mx, 1, 0, 256, A, A)[0] == 1            # no rows
    assert _view(mx, 1, 130, 256, None, A)[0] == 1       # null
    assert _view(mx, 1025, 128, 256, A, A)[0] == 1       # too many experts


def test_argument_errors_before_launch(mx):
    lib = mx.library()
    A = 1 << 20
    st, w = _view(mx, 1, 130, 256, A, A)
    assert st == 0
    wp = ctypes.byref(w)
    # quantize: K % 256, negative M, M = 0 is a no-op
    assert lib.mxfp8_quantize_act(A, 4, 320, A, A, None) == 2
    assert lib.mxfp8_quantize_act(A, -1, 256, A, A, None) == 1
    assert lib.mxfp8_quantize_act(A, 0, 256, A, A, None) == 0
    assert lib.mxfp8_quantize_act(A + 2, 4, 256, A, A, None) == 3
    # linear: M = 0 no-op, null / misaligned / small workspace
    assert lib.mxfp8_linear(A, 0, wp, None, A, A, 0, None) == 0
    assert lib.mxfp8_linear(None, 4, wp, None, A, A, 1 << 20, None) == 1
    assert lib.mxfp8_linear(A + 8, 4, wp, None, A, A, 1 << 20, None) == 3
    assert lib.mxfp8_linear(A, 4, wp, None, A + 1, A, 1 << 20, None) == 3
    assert lib.mxfp8_linear(A, 4, wp, None, A, A, 16, None) == 5
    assert lib.mxfp8_linear(A, 4, None, None, A, A, 1 << 20, None) == 1
    # host-buffer linear: sizes, M = 0 no-op, null / misaligned / small workspace
    assert lib.mxfp8_linear_host_workspace_bytes(4, 130, 256) == 2048 + 1280 + 1024 + 64
    assert lib.mxfp8_linear_host_workspace_bytes(4, 0, 256) == 0
    assert lib.mxfp8_linear_host(A, 0, wp, None, A, A, 0, None) == 0
    assert lib.mxfp8_linear_host(None, 4, wp, None, A, A, 1 << 20, None) == 1
    assert lib.mxfp8_linear_host(A, 4, wp, None, None, A, 1 << 20, None) == 1
    assert lib.mxfp8_linear_host(A, 4, wp, None, A, A + 8, 1 << 20, None) == 3
    assert lib.mxfp8_linear_host(A, 4, wp, None, A, A, 4415, None) == 5
    # gemm: dense only
    st2, w2 = _view(mx, 2, 128, 256, A, A)
    assert st2 == 0
    assert lib.mxfp8_gemm(A, A, 4, ctypes.byref(w2), None, A, None) == 1
    assert lib.mxfp8_linear(A, 4, ctypes.byref(w2), None, A, A, 1 << 20, None) == 1
    assert lib.mxfp8_linear_host(A, 4, ctypes.byref(w2), None, A, A, 1 << 20, None) == 1
    # grouped: offsets required
    assert lib.mxfp8_grouped_linear(A, 4, None, ctypes.byref(w2), None, A, A, 1 << 20, None) == 1
    assert lib.mxfp8_grouped_linear(A, 0, A, ctypes.byref(w2), None, A, A, 1 << 20, None) == 0
    # prepare: bad dtype, misaligned source
    assert lib.mxfp8_prepare_weight(A, 7, wp, None) == 1
    assert lib.mxfp8_prepare_weight(A + 4, 0, wp, None) == 3


def test_moe_size_helpers_and_argument_checks(mx):
    lib = mx.library()
    assert lib.mxfp8_moe_route_workspace_bytes(256, 128, 8) == ((256 + 7) // 8 * 128 + 256 * 8) * 4  # 8-token groups
    assert lib.mxfp8_moe_route_workspace_bytes(-1, 128, 8) == 0
    assert lib.mxfp8_moe_workspace_bytes(256, 128, 17, 2048, 768) == 0   # topk > 16
    assert lib.mxfp8_moe_workspace_bytes(256, 4, 8, 2048, 768) == 0      # topk > experts
    assert lib.mxfp8_moe_workspace_bytes(256, 128, 8, 2048, 768) > 0
    assert lib.mxfp8_moe_gate_up_workspace_bytes(2048, 2048) == mx.linear_workspace_bytes(2048, 2048)
    # checked before the device is touched (1 = MXFP8_ERR_INVALID_ARG)
    assert lib.mxfp8_moe_route(None, 4, 8, 0, 0, None, None, None, None, None, None, 0, None) == 1
    assert lib.mxfp8_moe_route(None, 4, 8, 2, 5, None, None, None, None, None, None, 0, None) == 1
    assert lib.mxfp8_moe_route(None, 0, 8, 2, 0, None, None, None, None, None, None, 0, None) == mx.OK
    assert lib.mxfp8_moe_finalize(None, None, None, 4, 2, 12, None, None) == 1  # hidden % 8: invalid argument
    assert lib.mxfp8_moe_finalize(None, None, None, 0, 2, 16, None, None) == mx.OK


def test_tactic_table_host_operations(mx):
    mx.tactic_clear()
    assert mx.tactic_count() == 0
    assert mx.tactic_get(mx.KIND_LINEAR, 16, 5120, 2048) is None
    mx.tactic_set(mx.KIND_LINEAR, 16, 5120, 2048, 1, (16, 4, 1, 2))
    assert mx.tactic_get(mx.KIND_LINEAR, 16, 5120, 2048) == (16, 4, 1, 2)
    # M buckets are powers of two: 9..16 share one entry, 17 does not
    assert mx.tactic_get(mx.KIND_LINEAR, 9, 5120, 2048) == (16, 4, 1, 2)
    assert mx.tactic_get(mx.KIND_LINEAR, 17, 5120, 2048) is None
    # kinds are separate
    assert mx.tactic_get(mx.KIND_GEMM, 16, 5120, 2048) is None
    mx.tactic_set(mx.KIND_GEMM, 8192, 8192, 8192, 1, (192, -1, 0, 2))
    mx.tactic_set(mx.KIND_GROUPED, 2048, 1536, 2048, 128, (32, -1, 0, 2))
    assert mx.tactic_count() == 3
    bad = [
        (mx.KIND_LINEAR, (48, -1, 0, 1)),    # no such tile
        (mx.KIND_LINEAR, (16, 9, 0, 1)),     # cluster of 9
        (mx.KIND_LINEAR, (128, -1, 0, 2)),   # two pipes need tiles <= 64
        (mx.KIND_LINEAR, (64, 1, 0, 4)),     # four pipes only with 16- or 32-token tiles
        (mx.KIND_GATED, (16, -1, 0, 4)),     # no four-pipe gated kernel of 16-token tiles
        (mx.KIND_GEMM, (16, 4, 1, 2)),       # fused quantization needs x
        (mx.KIND_GROUPED, (32, 2, 0, 2)),    # grouped tiles are persistent
        (mx.KIND_GROUPED, (192, -1, 0, 2)),  # two weight tiles: dense only
        (mx.KIND_GATED, (256, -1, 0, 1)),    # the gated exchange holds <= 128 tokens
        (mx.KIND_LINEAR, (256, 2, 0, 1)),    # one-tile schedules take <= 128 tokens
    ]
    for kind, t in bad:
        with pytest.raises(mx.Mxfp8Error):
            mx.tactic_set(kind, 16, 512, 2048, 1, t)
    with pytest.raises(mx.Mxfp8Error):
        mx.tactic_set(mx.KIND_LINEAR, 16, 512, 2048, 1, (16, 16, 0, 1))  # split beyond K/128 = 16? (cluster <= 8)
    assert mx.tactic_count() == 3
    mx.tactic_clear()
    assert mx.tactic_count() == 0


def test_heuristic_schedules_on_the_workloads(mx):
    """The built-in schedule rules on a 152-SM GB300, queried without a GPU:
    (tokens per tile, split-K cluster or -1 = persistent, fused quantization,
    MMA pipelines)."""
    mx.tactic_clear()
    L, G, GR, GA = mx.KIND_LINEAR, mx.KIND_GEMM, mx.KIND_GROUPED, mx.KIND_GATED
    cases = [
        # decode: 40 weight tiles x split 4 = 160 CTAs, quantization fused
        ((L, 16, 5120, 2048, 1), (16, 4, 1, 2)),
        ((L, 1, 5120, 2048, 1), (16, 4, 1, 2)),
        # pre-quantized input: nothing to fuse
        ((G, 16, 5120, 2048, 1), (16, 4, 0, 2)),
        # mid batch: 64-token tiles, split 4, two pipes (128 CTAs <= 152)
        ((L, 128, 2048, 4096, 1), (64, 4, 0, 2)),
        ((L, 128, 130, 4096, 1), (64, 4, 0, 2)),
        # tiny: K = 256 is two K blocks, so no split
        ((L, 7, 130, 256, 1), (16, 1, 1, 2)),
        # prefill: two weight tiles x 176 tokens, persistent (1504 tiles =
        # 9.9 waves of 152; the tile-cost model prefers it to 192 tokens)
        ((L, 8192, 8192, 8192, 1), (176, -1, 0, 2)),
        # M = 4096: 192-token tiles (704 tiles = 4.6 waves; 176 would need 6)
        ((L, 4096, 8192, 8192, 1), (192, -1, 0, 2)),
        # large M but too few tiles for the dual kernel: persistent 256
        ((L, 1024, 256, 1024, 1), (256, -1, 0, 1)),
        # grouped: mean segment 16 rows -> 32-token tiles, four pipes
        ((GR, 2048, 1536, 2048, 128), (32, -1, 0, 4)),
        ((GA, 2048, 1536, 2048, 128), (32, -1, 0, 4)),
        # gated with long segments: capped at 128 tokens
        ((GA, 12800, 1536, 2048, 128), (128, -1, 0, 1)),
    ]
    for args, want in cases:
        assert mx.plan_tactic(*args, sms=152) == want, (args, mx.plan_tactic(*args, sms=152))
    # a table entry takes precedence for its class only
    mx.tactic_set(L, 16, 5120, 2048, 1, (64, 2, 0, 2))
    assert mx.plan_tactic(L, 12, 5120, 2048, 1, sms=152) == (64, 2, 0, 2)
    assert mx.plan_tactic(G, 16, 5120, 2048, 1, sms=152) == (16, 4, 0, 2)
    mx.tactic_clear()
    assert mx.plan_tactic(L, 12, 5120, 2048, 1, sms=152) == (16, 4, 1, 2)
    # every heuristic choice is a valid tactic for its kind
    for args, want in cases:
        mx.tactic_set(args[0], args[1], args[2], args[3], args[4], want)
    mx.tactic_clear()
    # argument checks
    lib = mx.library()
    out = (ctypes.c_int32 * 4)()
    assert lib.mxfp8_plan_tactic(9, 16, 5120, 2048, 1, 152, out) == 1        # unknown kind
    assert lib.mxfp8_plan_tactic(L, 16, 5120, 2000, 1, 152, out) == 2        # K % 256
    assert lib.mxfp8_plan_tactic(L, 16, 5120, 2048, 2, 152, out) == 1        # dense with experts
    assert lib.mxfp8_plan_tactic(GA, 16, 1000, 2048, 4, 152, out) == 1       # gated n % 128
    assert lib.mxfp8_plan_tactic(L, 0, 5120, 2048, 1, 152, out) == 1         # m < 1
    assert lib.mxfp8_plan_tactic(L, 16, 5120, 2048, 1, 152, None) == 1
