"""Failure detection and weight refit on the GPU.

Failure detection (the kernels' waits are bounded): a testing hook shortens
the limit of every pipeline wait to 1 ns, so the first wait that is not
already satisfied runs out.  The kernel must record the timeout, unwind and
return; mxfp8_device_error() must report MXFP8_ERR_DEVICE_TIMEOUT, and with the
default limit restored the same context must compute correct results again.
No fault, trap or hang is involved.

Refit (weights updated in place after load, as the pages' serving runs do
with "update_weights_from_disk"): re-preparing a new weight into the same
buffers must be seen by a CUDA graph captured before the refit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_close_to_oracle, oracle_weight, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu

TIMEOUT = 6  # MXFP8_ERR_DEVICE_TIMEOUT


def _dense_inputs(mx, d):
    pw = mx.prepare_weight(to_dev_f32(d.w))
    b = None if d.bias is None else to_dev_bf16(d.bias)
    return pw, to_dev_bf16(d.x), b


@pytest.mark.parametrize("m", [16, 300])
def test_wait_timeout_is_reported_and_recovers(lib, m):
    d = workloads.dense(m=m, n=640, k=1024, seed=70 + m, bias=True)
    pw, x, b = _dense_inputs(lib, d)
    assert lib.device_error() == 0
    lib.set_wait_limit_ns(1)
    try:
        lib.linear(x, pw, b)
        torch.cuda.synchronize()
    finally:
        lib.set_wait_limit_ns(0)
    assert lib.device_error() == TIMEOUT
    assert lib.device_error() == 0          # read-and-clear
    y = lib.linear(x, pw, b)               # the context is still usable
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    wq, wsf = oracle_weight(d.w)
    assert_close_to_oracle(y, oracle.linear(d.x, wq, wsf, d.bias), "after timeout m=%d" % m)


def test_grouped_wait_timeout_recovers(lib):
    g = workloads.grouped_from_counts([9, 0, 40, 3], n=256, k=512, seed=75)
    pw = lib.prepare_weight(to_dev_f32(g.w))
    x = to_dev_bf16(g.x_sorted)
    off = torch.from_numpy(g.offsets).cuda()
    lib.set_wait_limit_ns(1)
    try:
        lib.grouped_linear(x, off, pw)
        torch.cuda.synchronize()
    finally:
        lib.set_wait_limit_ns(0)
    assert lib.device_error() == TIMEOUT
    y = lib.grouped_linear(x, off, pw)
    torch.cuda.synchronize()
    assert lib.device_error() == 0
    wq = np.stack([oracle.quantize_rows(g.w[e])[0] for e in range(g.experts)])
    wsf = np.stack([oracle.quantize_rows(g.w[e])[1] for e in range(g.experts)])
    assert_close_to_oracle(y, oracle.grouped_linear(g.x_sorted, g.offsets, wq, wsf), "grouped after timeout")


def test_refit_in_place_under_cuda_graph(lib):
    d1 = workloads.dense(m=16, n=384, k=512, seed=80, bias=True)
    d2 = workloads.dense(m=16, n=384, k=512, seed=81, bias=True)
    pw, x, b = _dense_inputs(lib, d1)
    q_ptr, sf_ptr = pw.q.data_ptr(), pw.sf.data_ptr()
    ws = torch.empty(lib.linear_workspace_bytes(16, 512), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lib.linear(x, pw, b, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        y = lib.linear(x, pw, b, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    wq1, wsf1 = oracle_weight(d1.w)
    assert_close_to_oracle(y, oracle.linear(d1.x, wq1, wsf1, d1.bias), "before refit")
    lib.prepare_weight(to_dev_f32(d2.w), out=pw)       # refit: same buffers
    assert (pw.q.data_ptr(), pw.sf.data_ptr()) == (q_ptr, sf_ptr)
    g.replay()
    torch.cuda.synchronize()
    wq2, wsf2 = oracle_weight(d2.w)
    assert_close_to_oracle(y, oracle.linear(d1.x, wq2, wsf2, d1.bias), "after refit")
    q_ref, sf_ref = oracle.prepare_weight(d2.w)
    assert np.array_equal(pw.q[0].cpu().numpy(), q_ref) and np.array_equal(pw.sf[0].cpu().numpy(), sf_ref)
