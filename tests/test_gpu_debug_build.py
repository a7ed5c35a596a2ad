"""The debug build (MXFP8_DEBUG): every computed global store index of the
quantizers, the GEMM epilogues and the MoE kernels is checked against the
extent of its buffer; an out-of-range store is skipped and reported by
mxfp8_device_error() as MXFP8_ERR_OUT_OF_BOUNDS.  It stands in for the
sanitizer, which is not available here.  The five workloads of the layer run
through it in a process of their own (the environment variable selects the
library at load time) and must match the oracle with no bounds error."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_five_workloads_in_the_debug_build(lib):
    assert os.path.exists(os.path.join(os.path.dirname(lib.library_path()), "libmxfp8_gb300_debug.so"))
    env = dict(os.environ, MXFP8_DEBUG_LIBRARY="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_child.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "DEBUG_BUILD_OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


def test_normal_build_is_not_the_debug_build(lib):
    assert not lib.debug_build()
