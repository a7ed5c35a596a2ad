"""The scratch-free entry point, mxfp8_linear_static_scratch.

It serves callers that cannot allocate device memory and so cannot pass
mxfp8_linear a workspace (code inside a framework that owns every device
allocation, serving paths that must not allocate).  Its scratch is a fixed
array inside the library.  This test calls it through the C ABI on two
different inputs in a row and checks each output against mxfp8_linear's on
the same input, within the linear tolerance of the other GPU tests
(|y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref)); it also checks that a size
beyond the array is refused before any launch.  The file name sorts last so
that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_common import assert_close_to_oracle, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu


def _static_call(mx, x, pw, bias):
    m = x.shape[0]
    y = torch.empty((m, pw.n), dtype=torch.bfloat16, device=x.device)
    st = mx.library().mxfp8_linear_static_scratch(
        ctypes.c_void_p(x.data_ptr()), m, ctypes.byref(pw.c),
        None if bias is None else ctypes.c_void_p(bias.data_ptr()),
        ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, mx.STATUS_NAMES.get(st, st)
    return y


def test_static_scratch_matches_linear_on_two_calls(lib):
    d1 = workloads.dense(m=300, n=390, k=1024, seed=60, bias=True)
    d2 = workloads.dense(m=37, n=390, k=1024, seed=61, bias=True)
    pw = lib.prepare_weight(to_dev_f32(d1.w))
    b = to_dev_bf16(d1.bias)
    x1 = to_dev_bf16(d1.x)
    x2 = to_dev_bf16(d2.x)
    y1 = _static_call(lib, x1, pw, b)
    y2 = _static_call(lib, x2, pw, b)   # second call reuses the same array
    r1 = lib.linear(x1, pw, b)
    r2 = lib.linear(x2, pw, b)
    torch.cuda.synchronize()
    assert_close_to_oracle(y1, r1.float().cpu().numpy().astype(np.float64), "static scratch call 1")
    assert_close_to_oracle(y2, r2.float().cpu().numpy().astype(np.float64), "static scratch call 2")
    # the Python wrapper is the same call
    y1b = lib.linear_static_scratch(x1, pw, b)
    torch.cuda.synchronize()
    assert torch.equal(y1b, y1)


def test_static_scratch_rejects_oversize(lib):
    lib_c = lib.library()
    d = workloads.dense(m=8, n=128, k=8192, seed=62, bias=False)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    x = torch.zeros((1, 8192), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((1, 128), dtype=torch.bfloat16, device="cuda")
    # 1986 rows of K = 8192 need more than the array holds; nothing launches,
    # so the small x/y buffers are never touched.
    st = lib_c.mxfp8_linear_static_scratch(ctypes.c_void_p(x.data_ptr()), 1986, ctypes.byref(pw.c),
                                           None, ctypes.c_void_p(y.data_ptr()), None)
    assert lib.STATUS_NAMES[st] == "MXFP8_ERR_WORKSPACE_TOO_SMALL"
    torch.cuda.synchronize()
