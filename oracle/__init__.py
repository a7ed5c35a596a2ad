"""CPU oracle for the MXFP8 block-scaled linear layer (numpy front end).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  It shares no
code with the CUDA library and never imports it.

Every function here is a thin numpy wrapper over the plain C oracle in
``mxfp8_oracle.c`` (single-threaded, double precision).  The C file's header
lists what the pages fix and which readings were taken where they are silent.
Sources, by page:
  * vLLM PR #52204 "[Kernel] Add FlashInfer TRTLLM MXFP8 linear backend"
    (Purpose; review thread on apply_weights): quantize BF16 activations with
    the 8x4 scale layout, block-scaled GEMM, slice padded N, add bias.
  * prhub summary of vLLM PR #52204 (key source snippets): 8x4 scale-buffer
    size ceil(m/8)*8 * ceil(k/32/4)*4; weight scales viewed as [N, K/32].
  * OCP Microscaling Formats v1.0 (public spec, named by the pages as
    "MXFP8"): E4M3 elements, one E8M0 scale per 32 elements.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_value.restype = ctypes.c_double
        lib.oracle_e4m3_round.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_round.restype = ctypes.c_uint8
        lib.oracle_e4m3_round_n.argtypes = [p, i64, p]
        lib.oracle_e4m3_round_n.restype = None
        lib.oracle_quantize_block.argtypes = [p, ctypes.c_int, p]
        lib.oracle_quantize_block.restype = ctypes.c_uint8
        lib.oracle_quantize_rows.argtypes = [p, i64, i64, ctypes.c_int, p, p]
        lib.oracle_quantize_rows.restype = None
        lib.oracle_dequant_rows.argtypes = [p, p, i64, i64, p]
        lib.oracle_dequant_rows.restype = None
        lib.oracle_offset_8x4.argtypes = [i64, i64, i64]
        lib.oracle_offset_8x4.restype = i64
        lib.oracle_act_scale_bytes.argtypes = [i64, i64]
        lib.oracle_act_scale_bytes.restype = i64
        lib.oracle_act_scale_8x4.argtypes = [p, i64, i64, p]
        lib.oracle_act_scale_8x4.restype = None
        lib.oracle_offset_w128x4.argtypes = [i64, i64, i64]
        lib.oracle_offset_w128x4.restype = i64
        lib.oracle_weight_layout.argtypes = [p, p, i64, i64, p, p]
        lib.oracle_weight_layout.restype = None
        lib.oracle_linear.argtypes = [p, i64, i64, p, p, i64, p, p, i64, p]
        lib.oracle_linear.restype = None
        lib.oracle_grouped_linear.argtypes = [p, i64, i64, p, i64, p, p, i64,
                                              p, p, i64, p]
        lib.oracle_grouped_linear.restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


RULE_OCP = 0       # reading S1 (A): floor(log2(amax)) - 8, the layer's rule
RULE_NO_SAT = 1    # reading S1 (B): smallest power of two that never saturates


# ------------------------------------------------------------------ formats
def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(int(code))


def e8m0_value(code: int) -> float:
    return _load().oracle_e8m0_value(int(code))


def e4m3_round(t) -> np.ndarray:
    """Round each double to an E4M3 byte (RNE, saturating at 448)."""
    t = np.ascontiguousarray(t, dtype=np.float64).ravel()
    out = np.zeros(t.size, dtype=np.uint8)
    _load().oracle_e4m3_round_n(_ptr(t), t.size, _ptr(out))
    return out


# ------------------------------------------------------------- quantization
def quantize_block(v, rule: int = RULE_OCP):
    """One block of 32 values -> (scale byte, 32 element bytes)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    assert v.shape == (32,)
    out = np.zeros(32, dtype=np.uint8)
    s = _load().oracle_quantize_block(_ptr(v), rule, _ptr(out))
    return int(s), out


def quantize_rows(x, rule: int = RULE_OCP):
    """[rows, k] float32 -> (q uint8 [rows, k], sf uint8 [rows, k/32] linear)."""
    x = _f32(x)
    rows, k = x.shape
    assert k % 32 == 0
    q = np.zeros((rows, k), dtype=np.uint8)
    sf = np.zeros((rows, k // 32), dtype=np.uint8)
    _load().oracle_quantize_rows(_ptr(x), rows, k, rule, _ptr(q), _ptr(sf))
    return q, sf


def dequant_rows(q, sf):
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    rows, k = q.shape
    out = np.zeros((rows, k), dtype=np.float64)
    _load().oracle_dequant_rows(_ptr(q), _ptr(sf), rows, k, _ptr(out))
    return out


# ------------------------------------------------------------------ layouts
def offset_8x4(m: int, b: int, kb: int) -> int:
    return _load().oracle_offset_8x4(m, b, kb)


def act_scale_bytes(m: int, k: int) -> int:
    return _load().oracle_act_scale_bytes(m, k)


def act_scale_8x4(sf_lin, m: int, k: int):
    sf_lin = np.ascontiguousarray(sf_lin, dtype=np.uint8)
    out = np.zeros(act_scale_bytes(m, k), dtype=np.uint8)
    _load().oracle_act_scale_8x4(_ptr(sf_lin), m, k, _ptr(out))
    return out


def quantize_act(x):
    """The per-call activation quantizer: [m, k] -> (q [m, k], sf 8x4 bytes)."""
    q, sf = quantize_rows(x, RULE_OCP)
    return q, act_scale_8x4(sf, x.shape[0], x.shape[1])


def quantize_act_128x4(x):
    """BF16 activations [m, k] -> (E4M3 bytes [m, k], scales in the 128x4
    tiling of the prepared weights, rows padded with 0x00 to ceil128(m))."""
    q, sf_lin = quantize_rows(x, RULE_OCP)
    _, sf_t = weight_layout(q, sf_lin)
    return q, sf_t


def offset_w128x4(n: int, b: int, kb: int) -> int:
    return _load().oracle_offset_w128x4(n, b, kb)


def weight_layout(q, sf_lin):
    """Quantized weight [n, k] + linear scales -> (q_pad [n_pad, k],
    sf_tiled [n_pad * k/32])."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sf_lin = np.ascontiguousarray(sf_lin, dtype=np.uint8)
    n, k = q.shape
    n_pad = (n + 127) // 128 * 128
    q_pad = np.zeros((n_pad, k), dtype=np.uint8)
    sf_t = np.zeros(n_pad * (k // 32), dtype=np.uint8)
    _load().oracle_weight_layout(_ptr(q), _ptr(sf_lin), n, k, _ptr(q_pad), _ptr(sf_t))
    return q_pad, sf_t


def prepare_weight(w):
    """The load-time weight preparation: float [n, k] -> (q_pad, sf_tiled)."""
    q, sf = quantize_rows(w, RULE_OCP)
    return weight_layout(q, sf)


# ------------------------------------------------------------------- linear
def linear(x, wq, wsf, bias=None, rows=None):
    """y_ref (double) = quantize(x) . dequant(W)^T + bias.

    x: float32 [m, k] (BF16 values widened exactly); wq uint8 [n, k];
    wsf uint8 [n, k/32] (linear); bias float32 [n] or None;
    rows: optional int64 row indices to compute (y has len(rows) rows)."""
    x = _f32(x)
    m, k = x.shape
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    wsf = np.ascontiguousarray(wsf, dtype=np.uint8)
    n = wq.shape[0]
    b = None if bias is None else _f32(bias)
    sel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    cnt = m if sel is None else len(sel)
    y = np.zeros((cnt, n), dtype=np.float64)
    _load().oracle_linear(_ptr(x), m, k, _ptr(wq), _ptr(wsf), n, _ptr(b),
                          _ptr(sel), 0 if sel is None else len(sel), _ptr(y))
    return y


def grouped_linear(x, offsets, wq, wsf, bias=None, rows=None):
    """Per-expert linear over expert-sorted rows.

    x float32 [rows, k]; offsets int32 [E+1]; wq uint8 [E, n, k];
    wsf uint8 [E, n, k/32]; bias float32 [E, n] or None."""
    x = _f32(x)
    r, k = x.shape
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    wsf = np.ascontiguousarray(wsf, dtype=np.uint8)
    e, n, _ = wq.shape
    b = None if bias is None else _f32(bias)
    sel = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    cnt = r if sel is None else len(sel)
    y = np.zeros((cnt, n), dtype=np.float64)
    _load().oracle_grouped_linear(_ptr(x), r, k, _ptr(off), e, _ptr(wq), _ptr(wsf),
                                  n, _ptr(b), _ptr(sel),
                                  0 if sel is None else len(sel), _ptr(y))
    return y


def within_tolerance(y, y_ref, rms_ref=None):
    """The layer's tolerance: |y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref),
    elementwise.  Returns (ok, worst ratio of error to bound)."""
    y = np.asarray(y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    if rms_ref is None:
        rms_ref = float(np.sqrt(np.mean(y_ref * y_ref))) if y_ref.size else 0.0
    bound = 8e-3 * np.abs(y_ref) + 1e-3 * rms_ref
    err = np.abs(y - y_ref)
    ratio = float(np.max(err / np.maximum(bound, 1e-300))) if y.size else 0.0
    return bool(np.all(err <= bound)), ratio
