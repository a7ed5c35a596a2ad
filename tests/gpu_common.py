"""Shared helpers of the GPU parity tests (device transfer, tolerance check).

The linear-layer tolerance, per output element, against the oracle's
double-precision result y_ref:
    |y - y_ref| <= 8e-3 * |y_ref| + 1e-3 * rms(y_ref)
(rms over the whole compared output).  The BF16 rounding of y alone is at most
2^-9 |y_ref| (~1.95e-3); the rest covers the FP32 accumulation order inside
the tensor cores and the split-K sum.  Quantized bytes and scales are compared
bit for bit.
"""
import numpy as np
import torch

REL_TOL = 8e-3
RMS_TOL = 1e-3


def to_dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda().to(torch.bfloat16)


def to_dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def assert_close_to_oracle(y, y_ref, what=""):
    y = y.float().cpu().numpy().astype(np.float64) if torch.is_tensor(y) else np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == y_ref.shape, (what, y.shape, y_ref.shape)
    assert np.isfinite(y).all(), "%s: non-finite output" % what
    rms = float(np.sqrt(np.mean(y_ref * y_ref))) if y_ref.size else 0.0
    bound = REL_TOL * np.abs(y_ref) + RMS_TOL * rms
    err = np.abs(y - y_ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError(
            "%s: %d/%d elements outside |y-y_ref| <= %g|y_ref| + %g rms (rms %.4g); first at %s: "
            "y=%.6g ref=%.6g; worst err/bound %.3g" %
            (what, int(bad.sum()), bad.size, REL_TOL, RMS_TOL, rms, i, y[i], y_ref[i],
             float(np.max(err / np.maximum(bound, 1e-300)))))


def oracle_weight(w):
    """The oracle's own quantization of a float weight: (q [n,k], sf [n,k/32])."""
    import oracle
    return oracle.quantize_rows(w)
