"""Child process of test_gpu_debug_build.py: loads the debug build of the
library (MXFP8_DEBUG_LIBRARY=1, every computed store index checked against
its buffer) and runs the five workloads of the layer through it, each
against the oracle, then asks the library whether any kernel computed an
out-of-bounds store.  Prints one line per workload and "DEBUG_BUILD_OK"."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import mxfp8_block_scaled_x4_gb300 as mx  # noqa: E402
import oracle  # noqa: E402
import oracle.moe as moe  # noqa: E402
import workloads  # noqa: E402
from gpu_common import assert_close_to_oracle, to_dev_bf16, to_dev_f32  # noqa: E402


def dense(d, rows=None):
    pw = mx.prepare_weight(to_dev_f32(d.w))
    b = None if d.bias is None else to_dev_bf16(d.bias)
    y = mx.linear(to_dev_bf16(d.x), pw, b)
    torch.cuda.synchronize()
    wq, wsf = oracle.quantize_rows(d.w)
    ref = oracle.linear(d.x, wq, wsf, d.bias, rows=rows)
    assert_close_to_oracle(y if rows is None else y[torch.as_tensor(rows, device=y.device)], ref, d.name)
    st = mx.device_error()
    assert st == 0, (d.name, mx.STATUS_NAMES.get(st, st))
    print("debug build:", d.name, "ok", flush=True)


def main():
    assert mx.debug_build(), "the debug library was not loaded"
    dense(workloads.tiny())
    dense(workloads.decode(m=1))
    dense(workloads.decode(m=16))
    dense(workloads.mid())
    dense(workloads.mid(n=130, bias=True))
    rng = np.random.default_rng(41)
    dense(workloads.prefill(), rows=np.unique(np.concatenate([[0, 191, 192, 8191], rng.integers(0, 8192, 12)])))
    g = workloads.grouped()
    pw = mx.prepare_weight(to_dev_f32(g.w))
    y = mx.grouped_linear(to_dev_bf16(g.x_sorted), torch.from_numpy(g.offsets).cuda(), pw)
    torch.cuda.synchronize()
    e = 8  # oracle on the rows of the first experts
    r1 = int(g.offsets[e])
    gq, gsf = moe.prepare_experts(g.w[:e])
    ref = oracle.grouped_linear(g.x_sorted[:r1], g.offsets[:e + 1], gq, gsf)
    assert_close_to_oracle(y[:r1], ref, "grouped")
    st = mx.device_error()
    assert st == 0, ("grouped", mx.STATUS_NAMES.get(st, st))
    print("debug build: grouped ok", flush=True)
    print("DEBUG_BUILD_OK", flush=True)


if __name__ == "__main__":
    main()
