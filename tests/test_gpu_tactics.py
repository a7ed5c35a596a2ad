"""GPU checks of the tactic table: autotuning picks a valid schedule that the
following calls use, manual tactics are honoured, results stay within the
layer tolerance of the oracle, and tuning refuses a capturing stream."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_close_to_oracle, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu


@pytest.fixture
def mx(lib):
    lib.tactic_clear()
    yield lib
    lib.tactic_clear()


def _dense(mx, d):
    pw = mx.prepare_weight(to_dev_f32(d.w))
    x = to_dev_bf16(d.x)
    b = None if d.bias is None else to_dev_bf16(d.bias)
    wq, wsf = oracle.quantize_rows(d.w)
    return pw, x, b, wq, wsf


def _schedule_matches(sched, tactic):
    tt, split, fuse, pipes = tactic
    if tt in (144, 160, 176, 192):
        return sched["split"] == -2
    return (sched["tokens_per_tile"] == tt and sched["pipes"] == pipes and sched["split"] == split
            and int(sched["fused"]) == fuse)


def _time(mx, fn, calls=200):
    for _ in range(10):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(calls):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / calls


def test_autotune_decode_linear(mx):
    d = workloads.decode(m=16)
    pw, x, b, wq, wsf = _dense(mx, d)
    ws = torch.empty(mx.linear_workspace_bytes(d.m, d.k), dtype=torch.uint8, device="cuda")
    t_heur = _time(mx, lambda: mx.linear(x, pw, b, workspace=ws))
    chosen = mx.autotune_linear(x, pw, b, iters=30)
    assert mx.tactic_get(mx.KIND_LINEAR, d.m, d.n, d.k) == chosen
    assert mx.tactic_count() == 1
    y = mx.linear(x, pw, b, workspace=ws)
    torch.cuda.synchronize()
    assert _schedule_matches(mx.last_schedule(), chosen), (mx.last_schedule(), chosen)
    assert_close_to_oracle(y, oracle.linear(d.x, wq, wsf, d.bias), "decode16 tuned")
    t_tuned = _time(mx, lambda: mx.linear(x, pw, b, workspace=ws))
    # the tuned tactic is not slower than the heuristic's (timing noise allowed)
    assert t_tuned <= t_heur * 1.15, (t_tuned, t_heur, chosen)


@pytest.mark.parametrize("tactic", [(32, 2, 0, 1), (64, -1, 0, 1), (16, 1, 1, 4), (16, 3, 0, 2), (128, -1, 0, 1)])
def test_manual_tactic_is_used_and_correct(mx, tactic):
    d = workloads.mid(n=1024, bias=True, seed=9, m=100)
    pw, x, b, wq, wsf = _dense(mx, d)
    mx.tactic_set(mx.KIND_LINEAR, d.m, d.n, d.k, 1, tactic)
    y = mx.linear(x, pw, b)
    torch.cuda.synchronize()
    assert _schedule_matches(mx.last_schedule(), tactic), (mx.last_schedule(), tactic)
    rows = np.arange(0, d.m, 7)
    assert_close_to_oracle(y[torch.as_tensor(rows, device=y.device)],
                           oracle.linear(d.x, wq, wsf, d.bias, rows=rows), "manual %s" % (tactic,))


def test_autotune_grouped(mx):
    g = workloads.grouped_from_counts([40, 0, 17, 64, 3, 90, 33, 8], 384, 512, seed=12)
    pw = mx.prepare_weight(to_dev_f32(g.w))
    x = to_dev_bf16(g.x_sorted)
    off = torch.from_numpy(g.offsets).cuda()
    chosen = mx.autotune_grouped_linear(x, off, pw, iters=10)
    assert mx.tactic_get(mx.KIND_GROUPED, g.rows, g.n, g.k, g.experts) == chosen
    y = mx.grouped_linear(x, off, pw)
    torch.cuda.synchronize()
    assert _schedule_matches(mx.last_schedule(), chosen)
    wq = np.zeros((g.experts, g.n, g.k), dtype=np.uint8)
    wsf = np.zeros((g.experts, g.n, g.k // 32), dtype=np.uint8)
    for i in range(g.experts):
        wq[i], wsf[i] = oracle.quantize_rows(g.w[i])
    assert_close_to_oracle(y, oracle.grouped_linear(g.x_sorted, g.offsets, wq, wsf), "grouped tuned")


def test_autotune_refuses_capturing_stream(mx):
    d = workloads.tiny()
    pw, x, b, _, _ = _dense(mx, d)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        mx.linear(x, pw, b)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    raised = False
    with torch.cuda.graph(g):
        try:
            mx.autotune_linear(x, pw, b, iters=2)
        except mx.Mxfp8Error:
            raised = True
    assert raised
    assert mx.tactic_count() == 0


@pytest.mark.parametrize("m,n,k", [(16, 5120, 2048), (1, 5120, 2048), (128, 2048, 4096), (7, 130, 256),
                                   (300, 390, 1024), (2000, 4096, 512)])
def test_plan_tactic_is_what_the_call_runs(mx, m, n, k):
    """mxfp8_plan_tactic (this device's SM count) names the schedule that the
    next call of that shape launches, with and without a table entry."""
    d = workloads.dense(m=m, n=n, k=k, seed=m + k, bias=False)
    pw, x, _, _, _ = _dense(mx, d)
    plan = mx.plan_tactic(mx.KIND_LINEAR, m, n, k)
    mx.linear(x, pw)
    torch.cuda.synchronize()
    assert _schedule_matches(mx.last_schedule(), plan), (plan, mx.last_schedule())
    if m <= 128:
        mx.tactic_set(mx.KIND_LINEAR, m, n, k, 1, (32, 2, 0, 2))
        assert mx.plan_tactic(mx.KIND_LINEAR, m, n, k) == (32, 2, 0, 2)
        mx.linear(x, pw)
        torch.cuda.synchronize()
        assert _schedule_matches(mx.last_schedule(), (32, 2, 0, 2)), mx.last_schedule()
