"""GPU parity: the MXFP8 MoE expert MLP (routing, gated GEMM1 with SwiGLU,
down projection, finalize) against the CPU oracle in oracle/moe.py.

Integer results (expert ids, offsets, the sorted order) and the prepared
weight bytes are compared exactly; floating-point results with the layer
tolerance |y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref), routing weights to
1e-6 relative (FP32 exp and division against float64).  Each GEMM stage is
checked at that tolerance on the same inputs as the oracle: GEMM1 + SwiGLU
from x, GEMM2 + finalize from the oracle's own h.  The whole layer end to end
has a wider, derived bound (test_expert_mlp_matches_oracle's docstring): h is
re-quantized to MXFP8 between the GEMMs, and a one-ulp BF16 difference in h
(FP32 tensor-core accumulation against the oracle's exact sum) moves an
E4M3 code by one step now and then.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.moe as M
import workloads
from gpu_common import assert_close_to_oracle, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu


def _route_both(mx, logits, topk, method):
    r = mx.moe_route(to_dev_f32(logits), topk, method)
    torch.cuda.synchronize()
    ids, w = M.route(logits, topk, method)
    return r, ids, w


@pytest.mark.parametrize("method", [M.RENORMALIZE, M.RENORMALIZE_NAIVE])
@pytest.mark.parametrize("shape", [(256, 128, 8, False), (37, 8, 2, False), (64, 16, 16, False),
                                   (33, 8, 8, False), (200, 32, 4, True), (1, 4, 1, False),
                                   # up to 512 tokens one cluster routes (two passes above 256);
                                   # above, two kernels (per-group selection, then one scan)
                                   (300, 128, 8, False), (512, 64, 4, True), (513, 32, 2, False),
                                   (3000, 64, 8, False), (2100, 32, 8, True)])
def test_route_matches_oracle(lib, method, shape):
    t, e, k, ties = shape
    mw = workloads.moe(seed=20 + t, tokens=t, experts=e, topk=k, hidden=256, inter=256, logit_ties=ties)
    r, ids, w = _route_both(lib, mw.logits, k, method)
    assert np.array_equal(r.ids.cpu().numpy(), ids)
    assert np.allclose(r.weights.cpu().numpy(), w, rtol=1e-6, atol=1e-7)
    off, stok, row_of = M.sort_by_expert(ids, e)
    assert np.array_equal(r.offsets.cpu().numpy(), off)
    assert np.array_equal(r.sorted_token.cpu().numpy(), stok)
    assert np.array_equal(r.row_of.cpu().numpy(), row_of)


@pytest.mark.parametrize("method", [M.RENORMALIZE, M.RENORMALIZE_NAIVE])
@pytest.mark.parametrize("shape", [(40, 512, 8, False), (70, 300, 4, True), (17, 1024, 16, False)])
def test_route_wide_expert_counts(lib, method, shape):
    """More experts than a warp keeps in registers (256): every selection
    round reads the logits again; 1024 experts and top-16 are the limits."""
    t, e, k, ties = shape
    logits = workloads.router_logits(90 + e, t, e, logit_ties=ties)
    r, ids, w = _route_both(lib, logits, k, method)
    assert np.array_equal(r.ids.cpu().numpy(), ids)
    assert np.allclose(r.weights.cpu().numpy(), w, rtol=1e-6, atol=1e-7)
    off, stok, row_of = M.sort_by_expert(ids, e)
    assert np.array_equal(r.offsets.cpu().numpy(), off)
    assert np.array_equal(r.sorted_token.cpu().numpy(), stok)
    assert np.array_equal(r.row_of.cpu().numpy(), row_of)


def test_route_is_deterministic(lib):
    mw = workloads.moe(seed=3, tokens=300, experts=64, topk=6, hidden=256, inter=256, logit_ties=True)
    a = lib.moe_route(to_dev_f32(mw.logits), 6)
    b = lib.moe_route(to_dev_f32(mw.logits), 6)
    torch.cuda.synchronize()
    for x, y in ((a.ids, b.ids), (a.weights, b.weights), (a.sorted_token, b.sorted_token), (a.row_of, b.row_of)):
        assert torch.equal(x, y)


def test_prepare_gate_up_weight_bytes(lib):
    e, inter, h = 3, 192, 256
    rng = np.random.default_rng(4)
    w13 = rng.standard_normal((e, 2 * inter, h)).astype(np.float32) * 0.05
    pw = lib.prepare_gate_up_weight(to_dev_f32(w13))
    torch.cuda.synchronize()
    src = M.gated_row_source(2 * inter, inter)
    for i in range(e):
        q_ref, sf_ref = oracle.prepare_weight(w13[i][src])
        assert np.array_equal(pw.q[i].cpu().numpy(), q_ref)
        assert np.array_equal(pw.sf[i].cpu().numpy(), sf_ref)


def _oracle_gate_up(mw, ids, rows):
    """h (BF16 values, float64) of the given expert-sorted rows."""
    w13q, w13sf = M.prepare_experts(mw.w13)
    off, stok, _ = M.sort_by_expert(ids, mw.experts)
    gu = oracle.grouped_linear(mw.x[stok], off, w13q, w13sf, rows=rows)
    return M.bf16_rne(M.silu(gu[:, :mw.inter]) * gu[:, mw.inter:])


@pytest.mark.parametrize("shape", [(37, 8, 2, 256, 256), (64, 4, 3, 512, 320), (256, 128, 8, 2048, 768)])
def test_gate_up_swiglu_matches_oracle(lib, shape):
    t, e, k, h, inter = shape
    mw = workloads.moe(seed=7 + t, tokens=t, experts=e, topk=k, hidden=h, inter=inter)
    r = lib.moe_route(to_dev_f32(mw.logits), k)
    w13 = lib.prepare_gate_up_weight(to_dev_f32(mw.w13))
    hv = lib.moe_gate_up_swiglu(to_dev_bf16(mw.x), r, w13)
    torch.cuda.synchronize()
    ids, _ = M.route(mw.logits, k)
    rows = np.arange(t * k) if t * k <= 512 else np.random.default_rng(1).choice(t * k, 256, replace=False)
    rows = np.sort(rows)
    ref = _oracle_gate_up(mw, ids, rows)
    assert_close_to_oracle(hv[torch.as_tensor(rows, device=hv.device)], ref, mw.name + " h")


def test_finalize_matches_weighted_sum(lib):
    rng = np.random.default_rng(8)
    t, e, k, hidden = 50, 16, 4, 264
    mw = workloads.moe(seed=8, tokens=t, experts=e, topk=k, hidden=256, inter=256)
    r = lib.moe_route(to_dev_f32(mw.logits), k)
    y2 = workloads.bf16_round(rng.standard_normal((t * k, hidden)).astype(np.float32))
    out = lib.moe_finalize(to_dev_bf16(y2), r)
    torch.cuda.synchronize()
    ids, w = M.route(mw.logits, k)
    _, _, row_of = M.sort_by_expert(ids, e)
    ref = np.zeros((t, hidden))
    for i in range(t):
        for s in range(k):
            ref[i] += w[i, s] * y2[row_of[i * k + s]].astype(np.float64)
    assert_close_to_oracle(out, ref, "finalize")


@pytest.mark.parametrize("shape", [(37, 8, 2, 256, 256), (100, 16, 4, 512, 512), (256, 128, 8, 2048, 768)])
def test_down_and_finalize_from_oracle_h(lib, shape):
    t, e, k, h, inter = shape
    mw = workloads.moe(seed=40 + t, tokens=t, experts=e, topk=k, hidden=h, inter=inter)
    ids, w = M.route(mw.logits, k)
    off, stok, row_of = M.sort_by_expert(ids, e)
    w13q, w13sf = M.prepare_experts(mw.w13)
    gu = oracle.grouped_linear(mw.x[stok], off, w13q, w13sf)
    h_ref = M.bf16_rne(M.silu(gu[:, :inter]) * gu[:, inter:])
    r = lib.moe_route(to_dev_f32(mw.logits), k)
    w2 = lib.prepare_weight(to_dev_f32(mw.w2))
    y2 = lib.grouped_linear(to_dev_bf16(h_ref), r.offsets, w2)
    out = lib.moe_finalize(y2, r)
    torch.cuda.synchronize()
    toks = list(range(t)) if t <= 100 else [0, 5, 99, 128, 255]
    ref = M.down_finalize(h_ref, off, row_of, w, *M.prepare_experts(mw.w2), toks)
    assert_close_to_oracle(out[torch.as_tensor(toks, device=out.device)], ref, mw.name + " down+finalize")


def assert_mlp_close(out, ref, what):
    """End-to-end bound of the expert MLP.  Between GEMM1 and GEMM2, h is
    rounded to BF16 and re-quantized to MXFP8 on both sides; where the GPU's
    FP32 GEMM1 sum and the oracle's exact sum round h to neighbouring BF16
    values, the E4M3 code of that element can differ by one step (up to 2^-3
    of the element).  Such a step perturbs every output of the row it feeds
    by |W2[c][i]| times that step, i.e. by a few per mille to a few percent of
    the row's outputs; it is rare (a fraction of order 1e-4 of h's elements).
    So: every element within 8e-3 |ref| + 2e-2 rms(ref), at least 98% of the
    elements within the single-layer bound 8e-3 |ref| + 1e-3 rms(ref), and the
    relative L2 error at most 5e-3."""
    y = out.float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(y - ref)
    assert np.isfinite(y).all(), what
    loose = err <= 8e-3 * np.abs(ref) + 2e-2 * rms
    tight = err <= 8e-3 * np.abs(ref) + 1e-3 * rms
    rel_l2 = float(np.linalg.norm(y - ref) / np.linalg.norm(ref))
    assert loose.all(), "%s: %d elements beyond the loose bound; worst err/rms %.3g" % (
        what, int((~loose).sum()), float((err / rms).max()))
    assert tight.mean() >= 0.98, "%s: only %.4f within the single-layer bound" % (what, tight.mean())
    assert rel_l2 <= 5e-3, "%s: relative L2 error %.3g" % (what, rel_l2)


@pytest.mark.parametrize("method", [M.RENORMALIZE, M.RENORMALIZE_NAIVE])
@pytest.mark.parametrize("shape", [(37, 8, 2, 256, 256), (100, 16, 4, 512, 512)])
def test_expert_mlp_matches_oracle(lib, method, shape):
    t, e, k, h, inter = shape
    mw = workloads.moe(seed=30 + t, tokens=t, experts=e, topk=k, hidden=h, inter=inter)
    w13 = lib.prepare_gate_up_weight(to_dev_f32(mw.w13))
    w2 = lib.prepare_weight(to_dev_f32(mw.w2))
    out = lib.moe_expert_mlp(to_dev_bf16(mw.x), to_dev_f32(mw.logits), k, w13, w2, method)
    torch.cuda.synchronize()
    ids, w = M.route(mw.logits, k, method)
    ref, _, _ = M.expert_mlp(mw.x, ids, w, *M.prepare_experts(mw.w13), *M.prepare_experts(mw.w2))
    assert_mlp_close(out, ref, mw.name)


def test_expert_mlp_workload_sampled_tokens(lib):
    mw = workloads.moe()  # 256 tokens, 128 experts, top-8, H=2048, I=768
    w13 = lib.prepare_gate_up_weight(to_dev_f32(mw.w13))
    w2 = lib.prepare_weight(to_dev_f32(mw.w2))
    out = lib.moe_expert_mlp(to_dev_bf16(mw.x), to_dev_f32(mw.logits), mw.topk, w13, w2)
    torch.cuda.synchronize()
    toks = [0, 1, 77, 128, 200, 255]
    ids, w = M.route(mw.logits, mw.topk)
    ref, _, _ = M.expert_mlp(mw.x, ids, w, *M.prepare_experts(mw.w13), *M.prepare_experts(mw.w2), rows=toks)
    assert_mlp_close(out[torch.as_tensor(toks, device=out.device)], ref, mw.name)
    # deterministic and graph-capturable
    ws = torch.empty(lib.moe_workspace_bytes(mw.tokens, mw.experts, mw.topk, mw.hidden, mw.inter),
                     dtype=torch.uint8, device="cuda")
    x, lg = to_dev_bf16(mw.x), to_dev_f32(mw.logits)
    again = lib.moe_expert_mlp(x, lg, mw.topk, w13, w2, workspace=ws)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lib.moe_expert_mlp(x, lg, mw.topk, w13, w2, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    holder = {}
    with torch.cuda.graph(g):
        holder["y"] = lib.moe_expert_mlp(x, lg, mw.topk, w13, w2, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(again, out)
    assert torch.equal(holder["y"], out)


def test_moe_arguments_rejected(lib):
    mw = workloads.moe(seed=1, tokens=8, experts=8, topk=2, hidden=256, inter=256)
    w13 = lib.prepare_gate_up_weight(to_dev_f32(mw.w13))
    w2 = lib.prepare_weight(to_dev_f32(mw.w2))
    x, lg = to_dev_bf16(mw.x), to_dev_f32(mw.logits)
    with pytest.raises(lib.Mxfp8Error):
        lib.moe_expert_mlp(x, lg, 9, w13, w2)     # topk > experts
    with pytest.raises(lib.Mxfp8Error):
        lib.moe_expert_mlp(x, lg, 2, w2, w13)     # weights swapped: shapes do not chain
    with pytest.raises(lib.Mxfp8Error):
        lib.moe_route(lg, 17)                     # topk > 16


def test_gate_up_every_row_many_experts(lib):
    """GEMM1 + SwiGLU over 128 experts with several tiles per persistent CTA
    (128 experts x 4 n-tiles, two K blocks per tile, so each of the two MMA
    pipelines takes one): every row of h against the oracle, and the layer
    against its stages bit for bit."""
    t, e, k, h, inter = 256, 128, 8, 256, 256
    mw = workloads.moe(seed=71, tokens=t, experts=e, topk=k, hidden=h, inter=inter)
    r = lib.moe_route(to_dev_f32(mw.logits), k)
    w13 = lib.prepare_gate_up_weight(to_dev_f32(mw.w13))
    hv = lib.moe_gate_up_swiglu(to_dev_bf16(mw.x), r, w13)
    torch.cuda.synchronize()
    ids, _ = M.route(mw.logits, k)
    rows = np.arange(t * k)
    assert_close_to_oracle(hv, _oracle_gate_up(mw, ids, rows), mw.name + " h")
    w2 = lib.prepare_weight(to_dev_f32(mw.w2))
    x, lg = to_dev_bf16(mw.x), to_dev_f32(mw.logits)
    out = lib.moe_expert_mlp(x, lg, k, w13, w2)
    y2 = lib.grouped_linear(hv, r.offsets, w2)
    chain = lib.moe_finalize(y2, r)
    torch.cuda.synchronize()
    assert torch.equal(out, chain)


def _layer_and_chain(lib, mw, k, w13, w2, ws=None):
    x, lg = to_dev_bf16(mw.x), to_dev_f32(mw.logits)
    out = lib.moe_expert_mlp(x, lg, k, w13, w2, workspace=ws)
    r = lib.moe_route(lg, k)
    hv = lib.moe_gate_up_swiglu(x, r, w13)
    chain = lib.moe_finalize(lib.grouped_linear(hv, r.offsets, w2), r)
    torch.cuda.synchronize()
    return out, chain


@pytest.mark.parametrize("shape", [(600, 16, 2, 256, 256),    # > 512 tokens: two routing kernels + gather
                                   (40, 520, 4, 256, 256),    # > 512 experts: the 8-CTA cluster
                                   (512, 64, 8, 256, 256),    # the one-launch limit: two passes per CTA
                                   (3, 4, 1, 256, 256),       # 3 rows: 5 pad rows in the scale group
                                   (40, 16, 16, 256, 256),    # top-16 (the limit): 16 copies of each row
                                   (1, 64, 8, 2048, 256)])    # one token, K = 2048: 8 rows, one scale group
def test_expert_mlp_routing_paths_are_the_stage_chain(lib, shape):
    """Each routing path of the layer (the one-launch cluster router, 16- or
    8-CTA, up to 512 tokens; the two-kernel router above) gives the bytes of
    the stages run one by one."""
    t, e, k, h, inter = shape
    mw = workloads.moe(seed=80 + t, tokens=t, experts=e, topk=k, hidden=h, inter=inter)
    w13 = lib.prepare_gate_up_weight(to_dev_f32(mw.w13))
    w2 = lib.prepare_weight(to_dev_f32(mw.w2))
    out, chain = _layer_and_chain(lib, mw, k, w13, w2)
    assert torch.equal(out.view(torch.int16), chain.view(torch.int16))


def test_expert_mlp_back_to_back_on_one_workspace(lib):
    """Consecutive layer calls on one workspace with different routings,
    queued back to back (the kernels of neighbouring calls overlap through
    programmatic dependent launch): each call's GEMMs take that call's
    offsets and rows, never the previous call's (same total, different
    segments)."""
    t, e, k, h, inter = 128, 32, 4, 256, 256
    base = workloads.moe(seed=90, tokens=t, experts=e, topk=k, hidden=h, inter=inter)
    w13 = lib.prepare_gate_up_weight(to_dev_f32(base.w13))
    w2 = lib.prepare_weight(to_dev_f32(base.w2))
    ws = torch.empty(lib.moe_workspace_bytes(t, e, k, h, inter), dtype=torch.uint8, device="cuda")
    x = to_dev_bf16(base.x)
    rng = np.random.default_rng(91)
    logits = [to_dev_f32(rng.standard_normal((t, e)).astype(np.float32) * (1 + i)) for i in range(4)]
    outs = [lib.moe_expert_mlp(x, lg, k, w13, w2, workspace=ws) for lg in logits]  # queued back to back
    torch.cuda.synchronize()
    for lg, out in zip(logits, outs):
        r = lib.moe_route(lg, k)
        hv = lib.moe_gate_up_swiglu(x, r, w13)
        chain = lib.moe_finalize(lib.grouped_linear(hv, r.offsets, w2), r)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), chain.view(torch.int16))


@pytest.mark.parametrize("shape", [(37, 8, 2, 256, 256), (100, 16, 4, 512, 512), (256, 128, 8, 2048, 768)])
def test_expert_mlp_is_the_stage_chain_and_each_stage_is_strict(lib, shape):
    """The whole layer equals, bit for bit, its stages run one by one (inside
    the layer GEMM1's epilogue quantizes h to MXFP8; the chain rounds h to
    BF16 and GEMM2's call quantizes it: the same bytes).  Each stage of that
    chain is then held to the single-layer tolerance on the GPU's own input:
    GEMM1 + SwiGLU from x (test_gate_up_swiglu_matches_oracle), GEMM2 from the
    GPU's h against the oracle's GEMM2, and finalize from the GPU's y2 against
    the exact weighted sum.  (GEMM2 and finalize composed carry two roundings,
    y2 to BF16 and the sum, so they are checked one at a time.)"""
    t, e, k, h, inter = shape
    mw = workloads.moe(seed=60 + t, tokens=t, experts=e, topk=k, hidden=h, inter=inter)
    w13 = lib.prepare_gate_up_weight(to_dev_f32(mw.w13))
    w2 = lib.prepare_weight(to_dev_f32(mw.w2))
    x, lg = to_dev_bf16(mw.x), to_dev_f32(mw.logits)
    out = lib.moe_expert_mlp(x, lg, k, w13, w2)
    r = lib.moe_route(lg, k)
    hv = lib.moe_gate_up_swiglu(x, r, w13)
    y2 = lib.grouped_linear(hv, r.offsets, w2)
    chain = lib.moe_finalize(y2, r)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), chain.view(torch.int16))
    ids, w = M.route(mw.logits, k)
    off, _, row_of = M.sort_by_expert(ids, e)
    rows = np.arange(t * k) if t * k <= 512 else np.sort(np.random.default_rng(2).choice(t * k, 256, replace=False))
    h_gpu = hv.float().cpu().numpy()
    y2_ref = oracle.grouped_linear(h_gpu, off, *M.prepare_experts(mw.w2), rows=rows)
    assert_close_to_oracle(y2[torch.as_tensor(rows, device=y2.device)], y2_ref, mw.name + " GEMM2 from its own h")
    y2_gpu = y2.float().cpu().numpy().astype(np.float64)
    ref = np.zeros((t, h))
    for i in range(t):
        for s in range(k):
            ref[i] += w[i, s] * y2_gpu[row_of[i * k + s]]
    assert_close_to_oracle(out, ref, mw.name + " finalize from its own y2")
