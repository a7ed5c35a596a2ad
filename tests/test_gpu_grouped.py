"""GPU parity: the grouped (MoE expert gate_up) MXFP8 layer against the CPU
oracle, and CUDA-graph capture/replay of the dense layer (vLLM PR #52204
tests CUDA Graph capture and replay equality)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_close_to_oracle, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu


def _oracle_expert_weights(w):
    e, n, k = w.shape
    wq = np.zeros((e, n, k), dtype=np.uint8)
    wsf = np.zeros((e, n, k // 32), dtype=np.uint8)
    for i in range(e):
        wq[i], wsf[i] = oracle.quantize_rows(w[i])
    return wq, wsf


def _run_grouped(mx, g, rows=None, schedule=(0, 0, -1), pipes=0):
    pw = mx.prepare_weight(to_dev_f32(g.w))
    x = to_dev_bf16(g.x_sorted)
    off = torch.from_numpy(g.offsets).cuda()
    b = None if g.bias is None else to_dev_bf16(g.bias)
    mx.set_schedule(*schedule)
    mx.set_pipes(pipes)
    try:
        y = mx.grouped_linear(x, off, pw, b)
    finally:
        mx.set_schedule(0, 0, -1)
        mx.set_pipes(0)
    torch.cuda.synchronize()
    wq, wsf = _oracle_expert_weights(g.w)
    y_ref = oracle.grouped_linear(g.x_sorted, g.offsets, wq, wsf, g.bias, rows=rows)
    yy = y if rows is None else y[torch.as_tensor(rows, device=y.device)]
    assert_close_to_oracle(yy, y_ref, g.name)
    return y


def test_moe_gate_up_config_sampled(lib):
    """256 tokens, 128 experts, top-8, N=1536, K=2048: the first and last row
    of every expert segment plus seeded random rows, all columns."""
    g = workloads.grouped()
    off = g.offsets
    edges = [int(off[e]) for e in range(g.experts) if off[e + 1] > off[e]] + \
            [int(off[e + 1]) - 1 for e in range(g.experts) if off[e + 1] > off[e]]
    rng = np.random.default_rng(50)
    rows = np.unique(np.concatenate([edges, rng.integers(0, g.rows, 64)]))
    _run_grouped(lib, g, rows=rows)


@pytest.mark.parametrize("tt", [16, 32, 64, 128, 256])
def test_grouped_edge_segments(lib, tt):
    """Empty experts, one-row experts, a segment longer than the token tile,
    ragged N, bias."""
    g = workloads.grouped_from_counts([5, 0, 300, 1, 0, 17, 40, 0], n=260, k=512, seed=51, bias=True)
    _run_grouped(lib, g, schedule=(tt, 0, -1))


@pytest.mark.parametrize("tt,pipes", [(16, 2), (16, 4), (32, 2), (32, 4), (64, 2)])
def test_grouped_multi_pipe(lib, tt, pipes):
    g = workloads.grouped_from_counts([5, 0, 300, 1, 0, 17, 40, 0], n=260, k=512, seed=53, bias=True)
    _run_grouped(lib, g, schedule=(tt, 0, -1), pipes=pipes)


def test_grouped_max_experts(lib):
    """The limit of 1024 experts (the per-expert tile-count table is full):
    mostly empty experts, rows in the first, last and two middle ones,
    ragged N, bias."""
    counts = [0] * 1024
    counts[0], counts[511], counts[700], counts[1023] = 3, 40, 1, 17
    g = workloads.grouped_from_counts(counts, n=130, k=256, seed=54, bias=True)
    _run_grouped(lib, g)


def test_grouped_all_rows_one_expert(lib):
    g = workloads.grouped_from_counts([0, 0, 70, 0], n=128, k=256, seed=52)
    _run_grouped(lib, g)


def test_cuda_graph_replay_equals_eager(lib):
    d = workloads.decode(m=16)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    x = to_dev_bf16(d.x)
    b = to_dev_bf16(d.bias)
    ws = torch.empty(lib.linear_workspace_bytes(16, d.k), dtype=torch.uint8, device="cuda")
    eager = lib.linear(x, pw, b, workspace=ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lib.linear(x, pw, b, workspace=ws)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        y_graph = lib.linear(x, pw, b, workspace=ws)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager, y_graph)
    # new input values through the same captured pointers
    x.copy_(to_dev_bf16(workloads.decode(m=16, seed=9).x))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(lib.linear(x, pw, b), y_graph)
