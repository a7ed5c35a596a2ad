"""Seeded synthetic inputs for the MXFP8 linear layer.

This module only draws random numbers and arranges them into the shapes of the
five workloads; it holds none of the method's arithmetic (no quantization, no
layouts, no products).  It is the one module that both the CPU oracle's tests
and the CUDA path's tests/benchmark use, so that both sides see the same bytes.

Recipe (numpy PCG64 ``default_rng(seed)``, ``standard_normal(dtype=float32)``):
  * activations x ~ N(0, 1), rounded to BF16 (torch RNE cast); returned as
    float32 arrays holding exact BF16 values;
  * weights W ~ N(0, 0.02) as float32 (the load-time input is FP32);
  * bias ~ N(0, 0.1), rounded to BF16.
Workload-specific structure:
  * tiny (M=7, N=130, K=256, seed 0): x[2, 64:96] = 0 and W[129, 0:32] = 0
    (all-zero 32-blocks), x[5, :] and W[7, :] scaled by 1e3 before rounding;
  * decode (M in {1, 16}, N=5120, K=2048): 20 outlier K-channels (1% of K,
    drawn without replacement) scaled by 20 on every row;
  * mid (M=128, K=4096, N=2048 without bias or N=130 with bias);
  * prefill (M=N=K=8192, no bias);
  * grouped MoE gate_up: 256 tokens, 128 experts, router logits ~ N(0, 1),
    each token routed to its 8 largest logits (ties -> lower expert id), the
    2048 (token, expert) pairs stable-sorted by (expert, token); expert e owns
    rows [off[e], off[e+1]) of x_sorted, x_sorted[r] = x[token(r)]; K=2048,
    per-expert N=1536, no bias.
  * MoE expert MLP (the whole layer around the grouped gate_up): tokens x
    ~ N(0, 1) rounded to BF16, router logits ~ N(0, 1) float32, GEMM1 weights
    [E, 2I, H] and GEMM2 weights [E, H, I] ~ N(0, 0.02) float32; 256 tokens,
    128 experts, top-8, H=2048, I=768 (the shapes of the gate_up workload
    plus its down projection).  The routing itself is part of the method and
    is not done here.
These stand in for the layers of the 30B-A3B MoE model the pages benchmark
end to end; no dataset or checkpoint is involved.
"""
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest BF16 (torch's RNE cast), returned
    as float32 holding the exact BF16 values."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def normal(rng, shape, std=1.0) -> np.ndarray:
    a = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


@dataclass
class Dense:
    name: str
    m: int
    n: int
    k: int
    x: np.ndarray                 # float32 [m, k], exact BF16 values
    w: np.ndarray                 # float32 [n, k]
    bias: Optional[np.ndarray]    # float32 [n], exact BF16 values, or None
    seed: int = 0


@dataclass
class Grouped:
    name: str
    tokens: int
    experts: int
    topk: int
    n: int
    k: int
    x_sorted: np.ndarray          # float32 [rows, k]
    offsets: np.ndarray           # int32 [experts + 1]
    token_of_row: np.ndarray      # int64 [rows]
    w: np.ndarray                 # float32 [experts, n, k]
    bias: Optional[np.ndarray]    # float32 [experts, n] or None
    seed: int = 0

    @property
    def rows(self) -> int:
        return int(self.x_sorted.shape[0])


def dense(m, n, k, seed, bias=True, w_std=0.02, name="dense") -> Dense:
    rng = np.random.default_rng(seed)
    x = bf16_round(normal(rng, (m, k)))
    w = normal(rng, (n, k), w_std)
    b = bf16_round(normal(rng, (n,), 0.1)) if bias else None
    return Dense(name, m, n, k, x, w, b, seed)


def tiny(seed=0) -> Dense:
    """M=7, N=130 (padded to 256), K=256 with zero blocks and x1e3 rows."""
    m, n, k = 7, 130, 256
    rng = np.random.default_rng(seed)
    x = normal(rng, (m, k))
    w = normal(rng, (n, k), 0.02)
    b = bf16_round(normal(rng, (n,), 0.1))
    x[2, 64:96] = 0.0
    w[129, 0:32] = 0.0
    x[5, :] *= np.float32(1e3)
    w[7, :] *= np.float32(1e3)
    return Dense("tiny_m7_n130_k256", m, n, k, bf16_round(x), w, b, seed)


def decode(m=16, seed=1, n=5120, k=2048, outlier_frac=0.01, outlier_gain=20.0) -> Dense:
    """Decode-shaped fused QKV: BF16 x with outlier channels."""
    rng = np.random.default_rng(seed)
    x = normal(rng, (m, k))
    n_out = int(round(outlier_frac * k))
    ch = rng.choice(k, size=n_out, replace=False)
    x[:, ch] *= np.float32(outlier_gain)
    w = normal(rng, (n, k), 0.02)
    b = bf16_round(normal(rng, (n,), 0.1))
    return Dense("decode_m%d_n%d_k%d" % (m, n, k), m, n, k, bf16_round(x), w, b, seed)


def mid(n=2048, bias=False, seed=3, m=128, k=4096) -> Dense:
    d = dense(m, n, k, seed, bias=bias)
    d.name = "mid_m%d_n%d_k%d%s" % (m, n, k, "_bias" if bias else "")
    return d


def prefill(seed=4, m=8192, n=8192, k=8192) -> Dense:
    d = dense(m, n, k, seed, bias=False)
    d.name = "prefill_m%d_n%d_k%d" % (m, n, k)
    return d


def route_topk(logits: np.ndarray, topk: int):
    """Expert ids of each token's top-k logits (descending; ties -> lower id).
    Softmax is monotone, so the top-k of softmax(logits) is the top-k of the
    logits themselves."""
    order = np.argsort(-logits, axis=1, kind="stable")
    return order[:, :topk]


def grouped(seed=5, tokens=256, experts=128, topk=8, n=1536, k=2048,
            bias=False, weights=True) -> Grouped:
    rng = np.random.default_rng(seed)
    logits = normal(rng, (tokens, experts))
    sel = route_topk(logits, topk)                     # [tokens, topk]
    tok = np.repeat(np.arange(tokens), topk)
    exp = sel.reshape(-1)
    order = np.lexsort((tok, exp))                     # by expert, then token
    tok_sorted = tok[order].astype(np.int64)
    exp_sorted = exp[order]
    counts = np.bincount(exp_sorted, minlength=experts)
    off = np.zeros(experts + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    x = bf16_round(normal(rng, (tokens, k)))
    w = normal(rng, (experts, n, k), 0.02) if weights else None
    b = bf16_round(normal(rng, (experts, n), 0.1)) if bias else None
    return Grouped("grouped_t%d_e%d_top%d_n%d_k%d" % (tokens, experts, topk, n, k),
                   tokens, experts, topk, n, k, np.ascontiguousarray(x[tok_sorted]),
                   off, tok_sorted, w, b, seed)


def grouped_from_counts(counts, n, k, seed, bias=False) -> Grouped:
    """Grouped input with explicit per-expert row counts (for edge cases such
    as empty experts and long segments)."""
    rng = np.random.default_rng(seed)
    counts = np.asarray(counts, dtype=np.int64)
    e = len(counts)
    off = np.zeros(e + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    rows = int(off[-1])
    x = bf16_round(normal(rng, (rows, k)))
    w = normal(rng, (e, n, k), 0.02)
    b = bf16_round(normal(rng, (e, n), 0.1)) if bias else None
    return Grouped("grouped_counts_e%d_n%d_k%d" % (e, n, k), rows, e, 1, n, k, x,
                   off, np.arange(rows, dtype=np.int64), w, b, seed)


@dataclass
class Moe:
    name: str
    tokens: int
    experts: int
    topk: int
    hidden: int
    inter: int
    x: np.ndarray                 # float32 [tokens, hidden], exact BF16 values
    logits: np.ndarray            # float32 [tokens, experts]
    w13: np.ndarray               # float32 [experts, 2*inter, hidden], rows [gate; up]
    w2: np.ndarray                # float32 [experts, hidden, inter]
    seed: int = 0


def router_logits(seed, tokens, experts, logit_ties=False) -> np.ndarray:
    """Router logits alone (float32 [tokens, experts]): N(0, 1), or with
    logit_ties integer values in [-3, 3]."""
    rng = np.random.default_rng(seed)
    if logit_ties:
        return rng.integers(-3, 4, size=(tokens, experts)).astype(np.float32)
    return normal(rng, (tokens, experts))


def moe(seed=6, tokens=256, experts=128, topk=8, hidden=2048, inter=768, logit_ties=False) -> Moe:
    """Inputs of one MoE expert-MLP layer.  logit_ties: integer-valued logits
    in [-3, 3] (many equal logits, to exercise the tie rule)."""
    rng = np.random.default_rng(seed)
    x = bf16_round(normal(rng, (tokens, hidden)))
    if logit_ties:
        logits = rng.integers(-3, 4, size=(tokens, experts)).astype(np.float32)
    else:
        logits = normal(rng, (tokens, experts))
    w13 = normal(rng, (experts, 2 * inter, hidden), 0.02)
    w2 = normal(rng, (experts, hidden, inter), 0.02)
    return Moe("moe_t%d_e%d_top%d_h%d_i%d" % (tokens, experts, topk, hidden, inter),
               tokens, experts, topk, hidden, inter, x, logits, w13, w2, seed)
