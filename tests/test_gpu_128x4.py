"""GPU parity of the high-M 128x4 activation-scale path against the oracle:
the quantizer's bytes bit for bit (the scale layout is the prepared weights'
128x4 tiling), the GEMM and the whole layer within the layer tolerance,
including ragged M (a last tile with one 128-token scale tile) and M <= 128
(128-token tiles)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_close_to_oracle, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(1, 256), (7, 512), (130, 2048), (300, 1024), (1000, 768)])
def test_quantize_act_128x4_bytes(lib, shape):
    m, k = shape
    d = workloads.dense(m, 128, k, seed=m + k, bias=False)
    q, sf = lib.quantize_act_128x4(to_dev_bf16(d.x))
    torch.cuda.synchronize()
    q_ref, sf_ref = oracle.quantize_act_128x4(d.x)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert sf.numel() == len(sf_ref) == (m + 127) // 128 * 128 * (k // 32)
    assert np.array_equal(sf.cpu().numpy(), sf_ref)


def test_quantize_act_128x4_prefill_bytes(lib):
    d = workloads.prefill()
    q, sf = lib.quantize_act_128x4(to_dev_bf16(d.x))
    torch.cuda.synchronize()
    q_ref, sf_ref = oracle.quantize_act_128x4(d.x)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(sf.cpu().numpy(), sf_ref)


@pytest.mark.parametrize("shape", [(128, 512, 1024, True), (129, 640, 2048, False), (300, 384, 1024, True),
                                   (1000, 130, 512, True), (40, 256, 256, False)])
def test_linear_128x4_matches_oracle(lib, shape):
    m, n, k, bias = shape
    d = workloads.dense(m, n, k, seed=5 + m, bias=bias)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    b = None if d.bias is None else to_dev_bf16(d.bias)
    y = lib.linear_128x4(to_dev_bf16(d.x), pw, b)
    torch.cuda.synchronize()
    sched = lib.last_schedule()
    assert sched["split"] == -1 and sched["tokens_per_tile"] == (256 if m > 128 else 128)
    wq, wsf = oracle.quantize_rows(d.w)
    assert_close_to_oracle(y, oracle.linear(d.x, wq, wsf, d.bias), "linear_128x4 %s" % (shape,))
    # the GEMM on separately quantized activations gives the same bytes
    q, sf = lib.quantize_act_128x4(to_dev_bf16(d.x))
    y2 = lib.gemm_128x4(q, sf, pw, b)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


def test_linear_128x4_prefill_sampled_rows(lib):
    d = workloads.prefill()
    pw = lib.prepare_weight(to_dev_f32(d.w))
    y = lib.linear_128x4(to_dev_bf16(d.x), pw)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 255, 256, 4095, 8000, 8191])
    wq, wsf = oracle.quantize_rows(d.w)
    assert_close_to_oracle(y[torch.as_tensor(rows, device=y.device)], oracle.linear(d.x, wq, wsf, rows=rows),
                           "prefill 128x4")


def test_linear_128x4_dual_tiles(lib):
    """Large enough for the dual weight-tile kernel (two weight tiles x 176
    tokens per CTA tile), with M = 1000: token tiles that straddle two or
    three 128-row scale tiles and a last tile of 120 rows.  The result equals,
    bit for bit, the 8x4 layer forced to the same schedule (the same E4M3
    bytes and scale values, only the scale layout differs), and the oracle on
    every tile and scale-tile boundary row."""
    m, n, k = 1000, 8192, 256
    d = workloads.dense(m, n, k, seed=77, bias=True)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    x, b = to_dev_bf16(d.x), to_dev_bf16(d.bias)
    y = lib.linear_128x4(x, pw, b)
    torch.cuda.synchronize()
    sched = lib.last_schedule()
    assert sched["tokens_per_tile"] == 176 and sched["split"] == -2
    lib.set_schedule(176, -1, 0)
    try:
        y8 = lib.linear(x, pw, b)
    finally:
        lib.set_schedule(0, 0, -1)
    torch.cuda.synchronize()
    assert torch.equal(y, y8)
    rows = np.array([0, 1, 127, 128, 175, 176, 255, 256, 351, 352, 383, 384, 527, 528, 639, 640, 703, 704,
                     767, 768, 879, 880, 895, 896, 999])
    wq, wsf = oracle.quantize_rows(d.w)
    assert_close_to_oracle(y[torch.as_tensor(rows, device=y.device)],
                           oracle.linear(d.x, wq, wsf, d.bias, rows=rows), "linear_128x4 dual")
