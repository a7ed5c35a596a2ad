"""Pins of the expert-MLP oracle (oracle/moe.py) against closed forms, hand
examples, library special cases and an independent dense composition.

Sources: FlashInfer PR #1214 "TRT-LLM Gen MoE" (Highlights: Renormalize =
TopK -> Softmax, RenormalizeNaive = Softmax -> TopK -> Renormalize; row
reordering for gated activations) and the unified-MoE per-tensor FP8 PR
(GEMM1 gate/linear, GEMM2).  The readings taken where they are silent are
listed in oracle/moe.py's header.
"""
import numpy as np
import pytest

import oracle
import oracle.moe as M


# ------------------------------------------------------------------ bf16_rne
def test_bf16_rne_hand_values():
    x = np.array([0.0, -0.0, 1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 3 * 2.0 ** -8),
                  2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134, 3.39e38, 3.40e38, np.inf, 255.5])
    # 3.39e38 is below the midpoint (2 - 2^-8) * 2^127 between the largest BF16
    # (2 - 2^-7) * 2^127 and 2^128, so it rounds to the largest BF16; 3.40e38 overflows.
    want = np.array([0.0, -0.0, 1.0, 1.0, 1.015625, -1.015625,
                     2.0 ** -133, 0.0, 2.0 ** -132, (2 - 2.0 ** -7) * 2.0 ** 127, np.inf, np.inf, 256.0])
    got = M.bf16_rne(x)
    assert np.array_equal(got, want)
    assert np.signbit(got[1])


def test_bf16_rne_matches_torch_on_float32_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000)).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(M.bf16_rne(x.astype(np.float64)), want)


# --------------------------------------------------------------------- silu
def test_silu_closed_forms():
    assert M.silu(0.0) == 0.0
    x = np.linspace(-20, 20, 401)
    # silu(x) - silu(-x) = x (sigma(x) + sigma(-x) = 1)
    assert np.allclose(M.silu(x) - M.silu(-x), x, rtol=0, atol=1e-12)
    assert abs(M.silu(1.0) - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15
    assert M.silu(-800.0) == -0.0 or abs(M.silu(-800.0)) < 1e-300


# -------------------------------------------------------------------- route
def test_route_hand_example_ties_and_order():
    logits = np.array([[1.0, 3.0, 3.0, 2.0],
                       [0.5, -1.0, 4.0, 4.0]])
    ids, w = M.route(logits, 2, M.RENORMALIZE)
    assert ids.tolist() == [[1, 2], [2, 3]]
    assert np.allclose(w, 0.5, rtol=0, atol=1e-15)
    ids, w = M.route(logits, 3, M.RENORMALIZE)
    assert ids.tolist() == [[1, 2, 3], [2, 3, 0]]
    e = np.exp([0.0, 0.0, -1.0])
    assert np.allclose(w[0], e / e.sum(), rtol=1e-15)


def test_route_methods_agree_and_match_argsort():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((40, 16)).astype(np.float32)
    logits[5, 3] = logits[5, 7]  # a tie
    a_ids, a_w = M.route(logits, 4, M.RENORMALIZE)
    b_ids, b_w = M.route(logits, 4, M.RENORMALIZE_NAIVE)
    assert np.array_equal(a_ids, b_ids)
    assert np.allclose(a_w, b_w, rtol=1e-12, atol=0)
    # top-k of the logits, descending, ties to the lower id (a stable argsort)
    ref = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :4]
    assert np.array_equal(a_ids, ref)
    assert np.allclose(a_w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(np.diff(a_w, axis=1) <= 0)
    # Naive from its own definition: softmax over all, renormalized on the top-k
    lg = logits.astype(np.float64)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p = p / p.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(p, b_ids, axis=1)
    assert np.allclose(b_w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)


def test_route_rejects_unknown_method():
    with pytest.raises(ValueError):
        M.route(np.zeros((1, 4)), 1, 7)


# ---------------------------------------------------------- sort_by_expert
def test_sort_by_expert_invariants():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((50, 12))
    ids, _ = M.route(logits, 3)
    off, tok, row_of = M.sort_by_expert(ids, 12)
    assert off[0] == 0 and off[-1] == 150
    assert np.array_equal(np.diff(off), np.bincount(ids.reshape(-1), minlength=12))
    # bijection and inverse
    assert sorted(row_of.tolist()) == list(range(150))
    for t in range(50):
        for s in range(3):
            r = row_of[t * 3 + s]
            assert tok[r] == t
            assert off[ids[t, s]] <= r < off[ids[t, s] + 1]
    # within an expert, tokens ascend
    for e in range(12):
        seg = tok[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)


def test_gated_row_source_is_the_tile_interleave():
    src = M.gated_row_source(256, 128)
    assert sorted(src.tolist()) == list(range(256))
    assert src[:64].tolist() == list(range(64))
    assert src[64:128].tolist() == list(range(128, 192))
    assert src[128:192].tolist() == list(range(64, 128))
    assert src[192:].tolist() == list(range(192, 256))


# ------------------------------------------------------------- expert_mlp
def _dense_reference(x, ids, w, w13q, w13sf, w2q, w2sf):
    """The same layer from dequantized dense matrices and numpy matmuls."""
    t, h = x.shape
    e, n2, _ = w13q.shape
    inter = n2 // 2
    xq, xsf = oracle.quantize_rows(x)
    xd = oracle.dequant_rows(xq, xsf)
    out = np.zeros((t, h))
    for i in range(t):
        for s in range(ids.shape[1]):
            ex = ids[i, s]
            gu = oracle.dequant_rows(w13q[ex], w13sf[ex]) @ xd[i]
            hh = M.bf16_rne(M.silu(gu[:inter]) * gu[inter:])
            hq, hsf = oracle.quantize_rows(hh.astype(np.float32)[None, :])
            hd = oracle.dequant_rows(hq, hsf)[0]
            out[i] += w[i, s] * M.bf16_rne(oracle.dequant_rows(w2q[ex], w2sf[ex]) @ hd)
    return out


@pytest.mark.parametrize("method", [M.RENORMALIZE, M.RENORMALIZE_NAIVE])
def test_expert_mlp_equals_dense_composition(method):
    rng = np.random.default_rng(7)
    t, h, inter, e, k = 6, 64, 64, 4, 2
    x = (rng.standard_normal((t, h))).astype(np.float32)
    logits = rng.standard_normal((t, e))
    w13 = rng.standard_normal((e, 2 * inter, h)) * 0.1
    w2 = rng.standard_normal((e, h, inter)) * 0.1
    w13q, w13sf = M.prepare_experts(w13)
    w2q, w2sf = M.prepare_experts(w2)
    ids, w = M.route(logits, k, method)
    out, hv, off = M.expert_mlp(x, ids, w, w13q, w13sf, w2q, w2sf)
    ref = _dense_reference(x, ids, w, w13q, w13sf, w2q, w2sf)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # a subset of tokens gives the same rows
    sub, _, _ = M.expert_mlp(x, ids, w, w13q, w13sf, w2q, w2sf, rows=[4, 1])
    assert np.array_equal(sub, out[[4, 1]])


def test_expert_mlp_gate_and_up_are_not_interchangeable():
    # silu(gate) * up != silu(up) * gate: swapping GEMM1's halves must change h.
    rng = np.random.default_rng(9)
    t, h, inter, e = 3, 64, 64, 1
    x = rng.standard_normal((t, h)).astype(np.float32)
    w13 = rng.standard_normal((e, 2 * inter, h)) * 0.2
    w2 = rng.standard_normal((e, h, inter)) * 0.2
    ids = np.zeros((t, 1), dtype=np.int32)
    w = np.ones((t, 1))
    a, _, _ = M.expert_mlp(x, ids, w, *M.prepare_experts(w13), *M.prepare_experts(w2))
    sw = np.concatenate([w13[:, inter:], w13[:, :inter]], axis=1)
    b, _, _ = M.expert_mlp(x, ids, w, *M.prepare_experts(sw), *M.prepare_experts(w2))
    assert not np.allclose(a, b)


def test_down_finalize_agrees_with_expert_mlp():
    rng = np.random.default_rng(12)
    t, h, inter, e, k = 5, 64, 64, 3, 2
    x = rng.standard_normal((t, h)).astype(np.float32)
    logits = rng.standard_normal((t, e))
    w13 = rng.standard_normal((e, 2 * inter, h)) * 0.1
    w2 = rng.standard_normal((e, h, inter)) * 0.1
    w13q, w13sf = M.prepare_experts(w13)
    w2q, w2sf = M.prepare_experts(w2)
    ids, w = M.route(logits, k)
    out, hv, off = M.expert_mlp(x, ids, w, w13q, w13sf, w2q, w2sf)
    _, _, row_of = M.sort_by_expert(ids, e)
    out2 = M.down_finalize(hv, off, row_of, w, w2q, w2sf, list(range(t)))
    assert np.array_equal(out, out2)
