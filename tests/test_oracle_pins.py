"""Pins for the CPU oracle: checks against things other than the oracle itself.

* hand-worked blocks (tests/golden/quant_blocks.txt, derived from the E4M3 /
  E8M0 definitions; the pages print no quantized value);
* library special cases: torch's and ml_dtypes' float8_e4m3fn casts (RNE, no
  saturation, so inputs are pre-clamped to |t| <= 448) and decoders;
* invariants of the format (round trip, idempotence, sign symmetry,
  power-of-two covariance);
* the 8x4 scale-buffer size printed in the prhub summary of vLLM PR #52204
  (key source snippets): ceil(m/8)*8 * ceil(k/32/4)*4 bytes;
* closed forms and exact brute force for the block-scaled product, with the
  operands decoded by torch, not by the oracle;
* the pages' own acceptance criterion (vLLM PR #52204 GPU test): cosine
  similarity > 0.98 against the unquantized product.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_blocks.txt")


def _golden_cases():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, rule, vals, scale, elems = [f.strip() for f in line.split("|")]
        v = np.zeros(32, dtype=np.float64)
        lead = [float(t) for t in vals.split(",")]
        v[:len(lead)] = lead
        cases.append((name, 0 if rule == "A" else 1, v, int(scale, 16),
                      [int(t, 16) for t in elems.split(",")]))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_golden_blocks(case):
    name, rule, v, scale, elems = case
    s, q = oracle.quantize_block(v, rule)
    assert s == scale, name
    assert list(q[:len(elems)]) == elems, name
    assert not q[len(elems):].any(), name


def test_nonfinite_block():
    for bad in (float("nan"), float("inf"), float("-inf")):
        v = np.ones(32)
        v[3] = bad
        s, q = oracle.quantize_block(v)
        assert s == 0xFF and (q == 0x7F).all()


def _lib_decode(codes):
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = _lib_decode(codes)
    mine = np.array([oracle.e4m3_value(c) for c in codes])
    nan = np.isnan(ref)
    assert (np.isnan(mine) == nan).all()
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert (mine[~nan] == ref[~nan]).all()
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x01) == 2.0 ** -9


def test_e8m0_decode():
    assert oracle.e8m0_value(127) == 1.0
    assert oracle.e8m0_value(0) == 2.0 ** -127
    assert oracle.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_value(255))


def _all_bf16_finite():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    f = bits.view(np.float32)
    return f[np.isfinite(f)].astype(np.float64)


def _torch_cast(t):
    return torch.from_numpy(np.asarray(t, dtype=np.float64)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_round_matches_torch_on_all_bf16():
    v = _all_bf16_finite()
    v = np.clip(v, -448.0, 448.0)  # library casts do not saturate
    assert (oracle.e4m3_round(v) == _torch_cast(v)).all()


def test_e4m3_round_matches_torch_on_random_fp32():
    rng = np.random.default_rng(123)
    # spread over the whole E4M3 range including subnormals and ties
    v = (rng.standard_normal(200000) * np.exp2(rng.integers(-12, 9, 200000))).astype(np.float32)
    v = np.clip(v.astype(np.float64), -448.0, 448.0)
    assert (oracle.e4m3_round(v) == _torch_cast(v)).all()
    # exact ties between neighbouring E4M3 values
    codes = np.arange(0, 0x7E, dtype=np.uint8)
    lo = _lib_decode(codes)
    hi = _lib_decode(codes + 1)
    mids = (lo + hi) / 2
    expect = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    assert (oracle.e4m3_round(mids) == expect).all()
    assert (oracle.e4m3_round(-mids) == (expect | 0x80)).all()


def test_e4m3_round_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    v = np.clip(_all_bf16_finite(), -448.0, 448.0)
    ref = v.astype(ml.float8_e4m3fn).view(np.uint8)
    assert (oracle.e4m3_round(v) == ref).all()


def test_e4m3_round_is_monotone():
    """Rounding to a grid is monotone: a larger input never decodes smaller
    (decoded by torch; -0 and +0 compare equal)."""
    rng = np.random.default_rng(321)
    _, grid = _e4m3_grid()
    g = grid[np.isfinite(grid)]
    t = np.concatenate([rng.uniform(-470.0, 470.0, 100000),
                        rng.standard_normal(50000) * 2.0 ** -7, g, (g[:-1] + g[1:]) / 2])
    t = np.sort(t)
    vals = _lib_decode(oracle.e4m3_round(t))
    assert (np.diff(vals) >= 0).all()


def test_quantization_error_within_half_an_e4m3_step():
    """The format's error bound, per element of random blocks spanning 60
    binades: with s = 2^(scale byte - 127) and t = |v|/s, an element that does
    not saturate (t <= 448) decodes within half the E4M3 spacing at t, times
    s (spacing 2^(floor(log2 t) - 3) for t >= 2^-6, 2^-9 below); one that
    does decodes to 448*s with v's sign."""
    rng = np.random.default_rng(77)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-30, 30, (64, 1)))).astype(np.float32)
    x[3, 32:64] *= 1.9  # more saturating blocks
    q, sf = oracle.quantize_rows(x)
    deq = _lib_dequant(q, sf)
    v = x.astype(np.float64)
    s = np.repeat(np.exp2(sf.astype(np.float64) - 127.0), 32, axis=1)
    t = np.abs(v) / s
    spacing = np.where(t >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(t, 2.0 ** -6))) - 3), 2.0 ** -9)
    sat = t > 448.0
    assert sat.any() and (~sat).any()
    assert (np.abs(deq - v)[~sat] <= (spacing * s / 2)[~sat]).all()
    assert (deq[sat] == np.sign(v[sat]) * 448.0 * s[sat]).all()


def test_e4m3_round_saturates():
    assert list(oracle.e4m3_round([448.0, 463.9, 464.0, 464.1, 500.0, 1e30, -1e30])) == \
        [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def _e4m3_grid():
    c = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    return c, _lib_decode(c)


def test_scale_rule_a_closed_form():
    """Rule A: 2^(s-127+8) <= amax < 2^(s-127+9) whenever no clamp applies."""
    rng = np.random.default_rng(7)
    for _ in range(2000):
        v = rng.standard_normal(32) * 2.0 ** rng.integers(-60, 60)
        v = v.astype(np.float32).astype(np.float64)
        s, _q = oracle.quantize_block(v)
        amax = np.max(np.abs(v))
        assert 2.0 ** (s - 119) <= amax < 2.0 ** (s - 118)


def test_scale_rule_b_closed_form():
    rng = np.random.default_rng(8)
    for _ in range(2000):
        v = rng.standard_normal(32) * 2.0 ** rng.integers(-60, 60)
        v = v.astype(np.float32).astype(np.float64)
        s, _q = oracle.quantize_block(v, oracle.RULE_NO_SAT)
        amax = np.max(np.abs(v))
        assert 448.0 * 2.0 ** (s - 127) >= amax > 448.0 * 2.0 ** (s - 128)


def test_round_trip_representable_blocks():
    """dequant(quant(x)) == x for blocks v_i * 2^j with v_i on the E4M3 grid
    and max |v_i| = 448, under both rules."""
    codes, vals = _e4m3_grid()
    rng = np.random.default_rng(9)
    for rule in (oracle.RULE_OCP, oracle.RULE_NO_SAT):
        for _ in range(300):
            v = vals[rng.integers(0, len(vals), 32)]
            v[rng.integers(0, 32)] = 448.0 * (1 if rng.random() < 0.5 else -1)
            j = int(rng.integers(-100, 100))
            x = v * 2.0 ** j
            s, q = oracle.quantize_block(x, rule)
            back = _lib_decode(q) * 2.0 ** (s - 127)
            assert (back == x).all()


def test_idempotence_and_symmetry_and_covariance():
    rng = np.random.default_rng(10)
    for _ in range(500):
        x = (rng.standard_normal(32) * 2.0 ** rng.integers(-20, 20)).astype(np.float32).astype(np.float64)
        s, q = oracle.quantize_block(x)
        deq = _lib_decode(q) * 2.0 ** (s - 127)
        s2, q2 = oracle.quantize_block(deq)
        assert s2 == s and (q2 == q).all()               # idempotence
        s3, q3 = oracle.quantize_block(-x)
        assert s3 == s and (q3 == (q ^ 0x80)).all()      # sign symmetry
        j = int(rng.integers(-30, 30))
        s4, q4 = oracle.quantize_block(x * 2.0 ** j)
        assert s4 == s + j and (q4 == q).all()           # 2^j covariance


def test_quantize_rows_is_blockwise():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((3, 96)).astype(np.float32)
    q, sf = oracle.quantize_rows(x)
    for r in range(3):
        for b in range(3):
            s, qb = oracle.quantize_block(x[r, b * 32:(b + 1) * 32].astype(np.float64))
            assert sf[r, b] == s and (q[r, b * 32:(b + 1) * 32] == qb).all()


# ------------------------------------------------------------------ layouts
@pytest.mark.parametrize("m,k", [(1, 256), (7, 256), (8, 512), (13, 768), (130, 256)])
def test_8x4_layout_size_and_bijection(m, k):
    kb = k // 32
    size = oracle.act_scale_bytes(m, k)
    # the fake (meta) implementation's size formula from the pages
    assert size == math.ceil(m / 8) * 8 * math.ceil(kb / 4) * 4
    m8 = math.ceil(m / 8) * 8
    offs = sorted(oracle.offset_8x4(r, b, kb) for r in range(m8) for b in range(kb))
    assert offs == list(range(size))
    # the 4 scales of one row and one group of 4 blocks form an aligned word
    for r in range(m8):
        for b4 in range(kb // 4):
            o0 = oracle.offset_8x4(r, 4 * b4, kb)
            assert o0 % 4 == 0
            assert [oracle.offset_8x4(r, 4 * b4 + c, kb) - o0 for c in range(4)] == [0, 1, 2, 3]
    # 8 rows x 4 blocks share one 32-byte tile
    assert {oracle.offset_8x4(r, b, kb) // 32 for r in range(8) for b in range(4)} == {0}


def test_8x4_layout_explicit_and_padding():
    m, k = 9, 256
    kb = 8
    sf = np.arange(m * kb, dtype=np.uint8).reshape(m, kb) + 1
    out = oracle.act_scale_8x4(sf, m, k)
    assert out.size == 16 * 8
    # row 0 blocks 0..3 -> bytes 0..3; row 1 -> 4..7; row 0 blocks 4..7 -> tile 1
    assert list(out[0:4]) == list(sf[0, 0:4])
    assert list(out[4:8]) == list(sf[1, 0:4])
    assert list(out[32:36]) == list(sf[0, 4:8])
    # row 8 (second row group) -> tile 2 (group 1, block quad 0)
    assert list(out[64:68]) == list(sf[8, 0:4])
    # rows 9..15 are padding: zero
    for r in range(9, 16):
        for b in range(kb):
            assert out[oracle.offset_8x4(r, b, kb)] == 0


def test_weight_layout():
    rng = np.random.default_rng(12)
    n, k = 130, 512
    kb = k // 32
    q = rng.integers(0, 255, (n, k), dtype=np.uint8)
    sf = rng.integers(1, 255, (n, kb), dtype=np.uint8)
    q_pad, sf_t = oracle.weight_layout(q, sf)
    assert q_pad.shape == (256, k) and (q_pad[:n] == q).all() and not q_pad[n:].any()
    assert sf_t.size == 256 * kb
    offs = sorted(oracle.offset_w128x4(r, b, kb) for r in range(256) for b in range(kb))
    assert offs == list(range(256 * kb))
    # explicit: rows 0, 32, 64, 96 share one 16-byte line of the first tile
    assert [oracle.offset_w128x4(r, 0, kb) for r in (0, 32, 64, 96, 1)] == [0, 4, 8, 12, 16]
    assert oracle.offset_w128x4(0, 4, kb) == 512           # next block quad
    assert oracle.offset_w128x4(128, 0, kb) == (kb // 4) * 512  # next row tile
    for r in range(n):
        for b in range(kb):
            assert sf_t[oracle.offset_w128x4(r, b, kb)] == sf[r, b]
    pad = [sf_t[oracle.offset_w128x4(r, b, kb)] for r in range(n, 256) for b in range(kb)]
    assert not any(pad)


# ------------------------------------------------------------------- linear
def _lib_dequant(q, sf):
    """Dequantize with torch's E4M3 decoder and exact powers of two."""
    vals = _lib_decode(q.reshape(-1)).reshape(q.shape)
    scale = np.exp2(sf.astype(np.float64) - 127.0)
    return vals * np.repeat(scale, 32, axis=1)


def test_linear_closed_form_all_ones():
    for k in (256, 2048):
        m, n = 3, 5
        x = np.ones((m, k), dtype=np.float32)
        wq, wsf = oracle.quantize_rows(np.ones((n, k), dtype=np.float32))
        y = oracle.linear(x, wq, wsf)
        assert (y == k).all()
        bias = np.arange(n, dtype=np.float32) * 0.5
        y = oracle.linear(x, wq, wsf, bias)
        assert (y == k + bias[None, :]).all()


def test_linear_exact_brute_force_tiny():
    """Exact rational sum over torch-decoded operands equals the oracle to
    within the double rounding of the final sum."""
    rng = np.random.default_rng(13)
    m, n, k = 3, 4, 64
    x = workloads.bf16_round(rng.standard_normal((m, k)).astype(np.float32))
    w = rng.standard_normal((n, k)).astype(np.float32) * np.float32(0.02)
    bias = workloads.bf16_round(rng.standard_normal(n).astype(np.float32) * 0.1)
    wq, wsf = oracle.quantize_rows(w)
    xq, xsf = oracle.quantize_rows(x)
    a = _lib_dequant(xq, xsf)
    b = _lib_dequant(wq, wsf)
    y = oracle.linear(x, wq, wsf, bias)
    for i in range(m):
        for j in range(n):
            exact = sum((Fraction(a[i, t]) * Fraction(b[j, t]) for t in range(k)), Fraction(0))
            exact += Fraction(float(bias[j]))
            assert abs(Fraction(y[i, j]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)


def test_linear_vs_library_matmul():
    """Non-square shapes (a transposed operand would not even conform) against
    a float64 matmul of torch-decoded operands."""
    rng = np.random.default_rng(14)
    m, n, k = 9, 130, 512
    x = workloads.bf16_round(rng.standard_normal((m, k)).astype(np.float32))
    w = rng.standard_normal((n, k)).astype(np.float32) * np.float32(0.02)
    bias = workloads.bf16_round(rng.standard_normal(n).astype(np.float32) * 0.1)
    wq, wsf = oracle.quantize_rows(w)
    xq, xsf = oracle.quantize_rows(x)
    ref = _lib_dequant(xq, xsf) @ _lib_dequant(wq, wsf).T + bias[None, :].astype(np.float64)
    y = oracle.linear(x, wq, wsf, bias)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # sampled rows are the same rows
    rows = np.array([8, 0, 5])
    assert (oracle.linear(x, wq, wsf, bias, rows=rows) == y[rows]).all()
    # 2^j covariance of the whole layer (no bias)
    y0 = oracle.linear(x, wq, wsf)
    assert (oracle.linear(x * np.float32(4.0), wq, wsf) == 4.0 * y0).all()


def test_linear_cosine_vs_unquantized():
    """The pages' GPU acceptance criterion: cosine similarity > 0.98 against
    the plain product of the unquantized operands (vLLM PR #52204 test)."""
    for (m, n, k) in [(1, 130, 256), (7, 256, 512), (128, 130, 768)]:
        torch.manual_seed(0)
        x = torch.randn(m, k, dtype=torch.bfloat16).float().numpy()
        w = torch.randn(n, k, dtype=torch.bfloat16).float().numpy()
        wq, wsf = oracle.quantize_rows(w)
        y = oracle.linear(x, wq, wsf)
        ref = x.astype(np.float64) @ w.astype(np.float64).T
        cos = (y * ref).sum() / np.sqrt((y * y).sum() * (ref * ref).sum())
        assert cos > 0.98


def test_grouped_linear_matches_per_expert_dense():
    g = workloads.grouped_from_counts([5, 0, 17, 1, 0, 9], n=130, k=256, seed=15, bias=True)
    wq = np.zeros((g.experts, g.n, g.k), dtype=np.uint8)
    wsf = np.zeros((g.experts, g.n, g.k // 32), dtype=np.uint8)
    for e in range(g.experts):
        wq[e], wsf[e] = oracle.quantize_rows(g.w[e])
    y = oracle.grouped_linear(g.x_sorted, g.offsets, wq, wsf, g.bias)
    assert y.shape == (g.rows, g.n)
    for e in range(g.experts):
        lo, hi = g.offsets[e], g.offsets[e + 1]
        if hi > lo:
            ref = oracle.linear(g.x_sorted[lo:hi], wq[e], wsf[e], g.bias[e])
            assert (y[lo:hi] == ref).all()
    # against torch-decoded float64 matmul, segment by segment
    xq, xsf = oracle.quantize_rows(g.x_sorted)
    a = _lib_dequant(xq, xsf)
    for e in range(g.experts):
        lo, hi = g.offsets[e], g.offsets[e + 1]
        ref = a[lo:hi] @ _lib_dequant(wq[e], wsf[e]).T + g.bias[e][None, :]
        assert np.allclose(y[lo:hi], ref, rtol=1e-12, atol=1e-12)
    rows = np.array([g.rows - 1, 0, 7])
    assert (oracle.grouped_linear(g.x_sorted, g.offsets, wq, wsf, g.bias, rows=rows) == y[rows]).all()


def test_prepare_weight_composes_quantize_and_layout():
    rng = np.random.default_rng(16)
    w = rng.standard_normal((200, 256)).astype(np.float32)
    q, sf = oracle.quantize_rows(w)
    q_pad, sf_t = oracle.prepare_weight(w)
    q2, sf2 = oracle.weight_layout(q, sf)
    assert (q_pad == q2).all() and (sf_t == sf2).all()


def test_act_128x4_places_each_rows_scales_in_the_weight_tiling():
    """The 128x4 activation scales: byte offset_w128x4(r, b) holds row r's
    block-b scale, the quantized bytes equal the 8x4 path's, and rows
    m .. ceil128(m)-1 hold 0x00."""
    rng = np.random.default_rng(17)
    m, k = 130, 512
    kb = k // 32
    x = rng.standard_normal((m, k)).astype(np.float32)
    x[5, 32:64] = 0.0
    q, sf_t = oracle.quantize_act_128x4(x)
    q8, _ = oracle.quantize_act(x)
    _, sf_lin = oracle.quantize_rows(x)
    assert (q == q8).all() and sf_t.size == 256 * kb
    for r in range(m):
        for b in range(kb):
            assert sf_t[oracle.offset_w128x4(r, b, kb)] == sf_lin[r, b]
    assert sf_t[oracle.offset_w128x4(5, 1, kb)] == 0
    assert not any(sf_t[oracle.offset_w128x4(r, b, kb)] for r in range(m, 256) for b in range(kb))


def test_tolerance_helper():
    y_ref = np.array([1.0, -2.0, 0.0, 100.0])
    ok, _ = oracle.within_tolerance(y_ref * (1 + 7e-3), y_ref)
    assert ok
    ok, _ = oracle.within_tolerance(y_ref * (1 + 2e-2), y_ref)
    assert not ok
