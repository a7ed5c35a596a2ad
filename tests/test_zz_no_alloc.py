"""The scratch-free entry point, mxfp8_linear_static_scratch.

It serves callers that cannot allocate device memory and so cannot pass
mxfp8_linear a workspace (code inside a framework that owns every device
allocation, serving paths that must not allocate).  Its scratch is a fixed
array inside the library.  This test calls it through the C ABI and checks
  * each output against the CPU oracle, within the linear tolerance of the
    other GPU tests (|y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref));
  * each output bit for bit against mxfp8_gemm on mxfp8_quantize_act's
    output (the same unfused path with caller buffers);
  * two calls in a row on different inputs (the second reuses the array),
    a small M (where mxfp8_linear would fuse the quantization but this path
    does not), and the largest M that fits the array at K = 8192;
  * that one row more is refused before any launch.
The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import assert_close_to_oracle, to_dev_bf16, to_dev_f32


K_BIG = 8192
M_FITS = 1985   # ceil256(m*k) + ceil8(m)*k/32 <= 16 MiB at k = 8192; 1986 does not fit


def _static_call(mx, x, pw, bias):
    m = x.shape[0]
    y = torch.empty((m, pw.n), dtype=torch.bfloat16, device=x.device)
    st = mx.library().mxfp8_linear_static_scratch(
        ctypes.c_void_p(x.data_ptr()), m, ctypes.byref(pw.c),
        None if bias is None else ctypes.c_void_p(bias.data_ptr()),
        ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, mx.STATUS_NAMES.get(st, st)
    return y


def _unfused_reference(mx, x, pw, bias):
    q, sf = mx.quantize_act(x)
    return mx.gemm(q, sf, pw, bias)


def _check(mx, d, pw, b, rows=None):
    x = to_dev_bf16(d.x)
    y = _static_call(mx, x, pw, b)
    r = _unfused_reference(mx, x, pw, b)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), r.view(torch.int16)), d.name
    wq, wsf = oracle.quantize_rows(d.w)
    ref = oracle.linear(d.x, wq, wsf, d.bias, rows=rows)
    yy = y if rows is None else y[torch.as_tensor(rows, device=y.device)]
    assert_close_to_oracle(yy, ref, "static scratch " + d.name)
    return y


@pytest.mark.gpu
def test_static_scratch_two_calls_against_the_oracle(lib):
    d1 = workloads.dense(m=300, n=390, k=1024, seed=60, bias=True)
    d2 = workloads.dense(m=37, n=390, k=1024, seed=61, bias=True)
    d2.w = d1.w  # same weight, second input
    pw = lib.prepare_weight(to_dev_f32(d1.w))
    b = to_dev_bf16(d1.bias)
    d2.bias = d1.bias
    y1 = _check(lib, d1, pw, b)
    _check(lib, d2, pw, b)     # second call reuses the same array
    # the Python wrapper is the same call
    y1b = lib.linear_static_scratch(to_dev_bf16(d1.x), pw, b)
    torch.cuda.synchronize()
    assert torch.equal(y1b, y1)


@pytest.mark.gpu
def test_static_scratch_small_m(lib):
    """M = 16: mxfp8_linear fuses the quantization into the GEMM here; this
    entry point quantizes into its array first."""
    d = workloads.decode(m=16, n=1024, k=2048, seed=63)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    _check(lib, d, pw, to_dev_bf16(d.bias))


@pytest.mark.gpu
def test_static_scratch_largest_m_that_fits(lib):
    d = workloads.dense(m=M_FITS, n=128, k=K_BIG, seed=64, bias=False)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    rows = np.array([0, 1, 7, 8, 1000, M_FITS - 2, M_FITS - 1])
    _check(lib, d, pw, None, rows=rows)


@pytest.mark.gpu
def test_static_scratch_rejects_oversize(lib):
    lib_c = lib.library()
    d = workloads.dense(m=8, n=128, k=K_BIG, seed=62, bias=False)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    x = torch.zeros((1, K_BIG), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((1, 128), dtype=torch.bfloat16, device="cuda")
    # one row more than fits needs more than the array holds; nothing
    # launches, so the small x/y buffers are never touched.
    st = lib_c.mxfp8_linear_static_scratch(ctypes.c_void_p(x.data_ptr()), M_FITS + 1, ctypes.byref(pw.c),
                                           None, ctypes.c_void_p(y.data_ptr()), None)
    assert lib.STATUS_NAMES[st] == "MXFP8_ERR_WORKSPACE_TOO_SMALL"
    torch.cuda.synchronize()


def test_size_limit_arithmetic():
    """The limit quoted in include/mxfp8.h: M_FITS rows fit at K = 8192, one more does not."""
    def need(m, k):
        return (m * k + 255) // 256 * 256 + (m + 7) // 8 * 8 * (k // 32)
    cap = 16 << 20
    assert need(M_FITS, K_BIG) <= cap < need(M_FITS + 1, K_BIG)
    assert need(7943, 2048) <= cap < need(7944, 2048)
