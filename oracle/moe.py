"""CPU oracle for the MXFP8 mixture-of-experts expert MLP (numpy, float64).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this module.  It shares no
code with the CUDA library and never imports it.

What it follows, by page:
  * FlashInfer PR #1214 "TRT-LLM Gen MoE" (summary, Highlights): two routing
    methods, Renormalize (top-k of the logits, then a softmax over those k)
    and RenormalizeNaive (a softmax over all experts, the top-k, then the k
    picks rescaled to sum to 1); the GEMM1 weight rows are reordered for the
    gated activation during weight preparation.
  * FlashInfer unified-MoE PR for per-tensor FP8 (What changed): the layer is
    GEMM1 (gate/linear) then GEMM2, the GEMM1 weights carry the gated-row
    reorder, and the MXFP8 scales of the row-permuted GEMM1/GEMM2 weights are
    in the 128x4 interleaved layout.
Readings where the pages are silent (each listed in the design notes):
  * The gated activation is SwiGLU: h = silu(gate) * up with
    silu(g) = g / (1 + exp(-g)); GEMM1's output rows are [gate; up] (gate
    rows 0..I-1, up rows I..2I-1).
  * Expert selection is made on the raw logits for both methods (softmax is
    strictly monotone, so this is the top-k of the probabilities in exact
    arithmetic); ties go to the lower expert id; the k experts of a token
    are listed in descending order of logit.
  * The per-expert rows are the (token, slot) pairs sorted by expert, then
    token (stable); offsets are the exclusive prefix of per-expert counts.
  * The intermediate activation h is a BF16 tensor (round to nearest even),
    quantized to MXFP8 like any layer input before GEMM2; GEMM2's output is
    BF16 too (every GEMM of the layer emits BF16, as the linear layer does).
  * The output of token t is sum_s w[t,s] * y2[row(t,s)] over its k slots
    (y2 the BF16 GEMM2 rows), no bias; returned unrounded (float64).
"""
import numpy as np

from . import grouped_linear

RENORMALIZE = 0
RENORMALIZE_NAIVE = 1


def bf16_rne(a):
    """Round float64 values to the nearest BF16 value (ties to even), returned
    as float64.  BF16 keeps 8 significant bits down to 2^-126 and a fixed
    spacing of 2^-133 below: with |a| = m * 2^e (m in [0.5, 1)) the spacing is
    2^q, q = max(e - 8, -133), and the result is rint(|a| / 2^q) * 2^q
    (np.rint rounds half to even; the scaling by 2^-q is exact)."""
    a = np.asarray(a, dtype=np.float64)
    out = np.array(a, dtype=np.float64, copy=True)
    fin = np.isfinite(a) & (a != 0)
    m, e = np.frexp(np.abs(a[fin]))
    q = np.maximum(e - 8, -133)
    r = np.ldexp(np.rint(np.ldexp(np.abs(a[fin]), -q)), q)
    r[r > 3.3895313892515355e38] = np.inf  # above the largest BF16 after rounding
    out[fin] = np.copysign(r, a[fin])
    return out


def route(logits, topk, method=RENORMALIZE):
    """Top-k expert selection and weights per token.

    logits: float [T, E]; returns (ids int32 [T, topk], weights float64
    [T, topk]), experts in descending order of logit (ties: lower id first).
      RENORMALIZE: w = softmax over the k selected logits.
      RENORMALIZE_NAIVE: p = softmax over all E logits; w = p_sel / sum(p_sel).
    """
    lg = np.asarray(logits, dtype=np.float64)
    t, e = lg.shape
    ids = np.zeros((t, topk), dtype=np.int32)
    w = np.zeros((t, topk), dtype=np.float64)
    for i in range(t):
        order = sorted(range(e), key=lambda j: (-lg[i, j], j))[:topk]
        ids[i] = order
        sel = lg[i, order]
        if method == RENORMALIZE:
            z = np.exp(sel - sel.max())
            w[i] = z / z.sum()
        elif method == RENORMALIZE_NAIVE:
            z = np.exp(lg[i] - lg[i].max())
            p = z / z.sum()
            ps = p[order]
            w[i] = ps / ps.sum()
        else:
            raise ValueError("unknown routing method %r" % (method,))
    return ids, w


def sort_by_expert(ids, experts):
    """Expert-sorted row order of the (token, slot) pairs.

    Returns (offsets int32 [E+1], sorted_token int32 [T*k] = token of sorted
    row r, row_of int32 [T*k] = sorted row of pair (t, s) at index t*k + s)."""
    ids = np.asarray(ids)
    t, k = ids.shape
    pairs = [(int(ids[i, s]), i, s) for i in range(t) for s in range(k)]
    pairs.sort(key=lambda p: (p[0], p[1]))  # by expert, then token
    counts = np.zeros(experts, dtype=np.int64)
    sorted_token = np.zeros(t * k, dtype=np.int32)
    row_of = np.zeros(t * k, dtype=np.int32)
    for r, (ex, i, s) in enumerate(pairs):
        counts[ex] += 1
        sorted_token[r] = i
        row_of[i * k + s] = r
    off = np.zeros(experts + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    return off, sorted_token, row_of


def gated_row_source(n_pad, inter):
    """Source row of each prepared GEMM1 weight row (gated-row reorder): the
    128-row tile j holds gate rows [64j, 64j + 64) then up rows
    [inter + 64j, inter + 64j + 64), so one tile produces 64 features of h."""
    src = np.zeros(n_pad, dtype=np.int64)
    for r in range(n_pad):
        j, o = divmod(r, 128)
        src[r] = 64 * j + o if o < 64 else inter + 64 * j + (o - 64)
    return src


def silu(g):
    g = np.asarray(g, dtype=np.float64)
    return g / (1.0 + np.exp(-g))


def prepare_experts(w):
    """Per-expert load-time preparation of float weights [E, n, k]: quantized
    bytes [E, n, k] and linear scales [E, n, k/32] (the oracle's own layout)."""
    from . import quantize_rows, RULE_OCP
    e, n, k = w.shape
    q = np.zeros((e, n, k), dtype=np.uint8)
    sf = np.zeros((e, n, k // 32), dtype=np.uint8)
    for i in range(e):
        q[i], sf[i] = quantize_rows(w[i], RULE_OCP)
    return q, sf


def down_finalize(h_sorted, off, row_of, weights, w2q, w2sf, rows):
    """GEMM2 of given expert-sorted h rows (BF16 values) and the weighted sum
    per token: out[a] = sum_s weights[t,s] * bf16(GEMM2(h)[row(t,s)]) for the
    tokens t = rows[a]."""
    k = weights.shape[1]
    need = np.array(sorted(int(row_of[i * k + s]) for i in rows for s in range(k)), dtype=np.int64)
    y2 = bf16_rne(grouped_linear(np.asarray(h_sorted, dtype=np.float32), off, w2q, w2sf, rows=need))
    pos = {int(r): j for j, r in enumerate(need)}
    out = np.zeros((len(rows), w2q.shape[1]), dtype=np.float64)
    for a, i in enumerate(rows):
        for s in range(k):
            out[a] += weights[i, s] * y2[pos[int(row_of[i * k + s])]]
    return out


def expert_mlp(x, ids, weights, w13q, w13sf, w2q, w2sf, rows=None):
    """The expert MLP of one MoE layer for given routing.

    x float32 [T, H] (BF16 values); ids/weights [T, k] from route();
    w13q/w13sf: GEMM1 weights [E, 2I, H] (rows [gate; up], original order)
    and linear scales [E, 2I, H/32]; w2q/w2sf: GEMM2 [E, H, I], [E, H, I/32].
    rows: optional token indices to evaluate (others are not computed).
    Returns (out float64 [len(rows) or T, H], h_bf16 float64 [T*k, I] in
    expert-sorted row order for the evaluated rows' pairs, offsets)."""
    x = np.asarray(x, dtype=np.float32)
    t, hdim = x.shape
    e, n2, _ = w13q.shape
    inter = n2 // 2
    k = ids.shape[1]
    off, sorted_token, row_of = sort_by_expert(ids, e)
    toks = np.arange(t) if rows is None else np.asarray(rows, dtype=np.int64)
    need = np.array(sorted(int(row_of[i * k + s]) for i in toks for s in range(k)), dtype=np.int64)
    x_sorted = x[sorted_token]
    gu = grouped_linear(x_sorted, off, w13q, w13sf, rows=need)       # [len(need), 2I]
    h = bf16_rne(silu(gu[:, :inter]) * gu[:, inter:])
    h_full = np.zeros((t * k, inter), dtype=np.float32)
    h_full[need] = h.astype(np.float32)                                # exact (BF16 values)
    y2 = bf16_rne(grouped_linear(h_full, off, w2q, w2sf, rows=need))    # [len(need), H], BF16 values
    pos = {int(r): j for j, r in enumerate(need)}
    out = np.zeros((len(toks), hdim), dtype=np.float64)
    for a, i in enumerate(toks):
        for s in range(k):
            out[a] += weights[i, s] * y2[pos[int(row_of[i * k + s])]]
    return out, h, off
