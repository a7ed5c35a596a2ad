"""GPU parity: the activation quantizer (8x4 layout) and the weight
preparation, bit for bit against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_common import to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu


def _quant_and_compare(mx, x):
    m, k = x.shape
    q, sf = mx.quantize_act(to_dev_bf16(x))
    torch.cuda.synchronize()
    q_ref, sf_ref = oracle.quantize_act(x)
    q = q.cpu().numpy()
    sf = sf.cpu().numpy()
    assert sf.size == sf_ref.size == oracle.act_scale_bytes(m, k)
    bad_q = np.argwhere(q != q_ref)
    assert bad_q.size == 0, "E4M3 bytes differ at %s: gpu %s oracle %s" % (
        bad_q[:4].tolist(), q[tuple(bad_q[0])], q_ref[tuple(bad_q[0])])
    bad_s = np.flatnonzero(sf != sf_ref)
    assert bad_s.size == 0, "scale bytes differ at %s" % bad_s[:8].tolist()


def test_all_bf16_bit_patterns(lib):
    """Every BF16 bit pattern (NaN/Inf included), in sorted and shuffled
    blocks, gives the oracle's bytes: exercises every E4M3 rounding case,
    subnormals, saturation and the non-finite rule."""
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    vals = bits.view(np.float32)
    _quant_and_compare(lib, vals.reshape(256, 256))
    rng = np.random.default_rng(20)
    _quant_and_compare(lib, rng.permutation(vals).reshape(128, 512))
    # finite values only, shuffled, so most blocks take the normal path
    fin = vals[np.isfinite(vals)]
    fin = rng.permutation(fin)[:(fin.size // 1024) * 1024]
    _quant_and_compare(lib, fin.reshape(-1, 1024))


@pytest.mark.parametrize("m,k", [(1, 256), (7, 256), (9, 512), (16, 2048), (33, 768),
                                 (130, 256), (1000, 1024)])
def test_ragged_shapes(lib, m, k):
    rng = np.random.default_rng(m * 7 + k)
    x = workloads.bf16_round(rng.standard_normal((m, k)).astype(np.float32)
                             * np.exp2(rng.integers(-30, 30, (m, 1))).astype(np.float32))
    _quant_and_compare(lib, x)


def test_special_blocks(lib):
    x = np.zeros((8, 256), dtype=np.float32)
    x[1, :32] = -0.0                         # signed-zero block
    x[2, 32:64] = 2.0 ** -133                # smallest subnormal: clamped scale
    x[3, 0] = np.inf                         # non-finite block
    x[4, 64] = np.nan
    x[5, :] = 448.0
    x[6, 96:128] = [480.0, 464.0] * 16       # saturation
    x[7, :] = workloads.bf16_round(np.linspace(-1e3, 1e3, 256, dtype=np.float32))
    _quant_and_compare(lib, x)


@pytest.mark.parametrize("name", ["tiny", "decode1", "decode16", "mid", "grouped"])
def test_workload_activations(lib, name):
    if name == "tiny":
        x = workloads.tiny().x
    elif name == "decode1":
        x = workloads.decode(m=1).x
    elif name == "decode16":
        x = workloads.decode(m=16).x
    elif name == "mid":
        x = workloads.mid().x
    else:
        x = workloads.grouped(weights=False).x_sorted
    _quant_and_compare(lib, x)


def test_prefill_activations_full(lib):
    """The 8192 x 8192 prefill activations, every byte."""
    rng = np.random.default_rng(4)
    x = workloads.bf16_round(rng.standard_normal((8192, 8192), dtype=np.float32))
    _quant_and_compare(lib, x)


def test_quantize_m0_is_noop(lib):
    q = torch.empty((0, 256), dtype=torch.uint8, device="cuda")
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    st = lib.library().mxfp8_quantize_act(x.data_ptr() or 256, 0, 256, q.data_ptr() or 256,
                                          q.data_ptr() or 256, None)
    assert st == 0


def _prep_and_compare(mx, w, as_bf16=False):
    wt = to_dev_bf16(w) if as_bf16 else to_dev_f32(w)
    pw = mx.prepare_weight(wt)
    torch.cuda.synchronize()
    src = workloads.bf16_round(w) if as_bf16 else w
    e = src.shape[0] if src.ndim == 3 else 1
    src3 = src.reshape(e, src.shape[-2], src.shape[-1])
    q = pw.q.cpu().numpy()
    sf = pw.sf.cpu().numpy()
    for i in range(e):
        q_ref, sf_ref = oracle.prepare_weight(src3[i])
        assert np.array_equal(q[i], q_ref), "expert %d data" % i
        assert np.array_equal(sf[i], sf_ref), "expert %d scales" % i
    return pw


@pytest.mark.parametrize("n,k", [(130, 256), (128, 512), (1, 256), (300, 768), (5120, 2048)])
@pytest.mark.parametrize("as_bf16", [False, True])
def test_prepare_weight(lib, n, k, as_bf16):
    rng = np.random.default_rng(n + k)
    w = rng.standard_normal((n, k), dtype=np.float32) * np.float32(0.02)
    w[0, :32] = 0.0
    if n > 7:
        w[7, :] *= np.float32(1e3)
    _prep_and_compare(lib, w, as_bf16)


def test_prepare_weight_tiny_config(lib):
    _prep_and_compare(lib, workloads.tiny().w)


def test_prepare_weight_stacked_experts(lib):
    rng = np.random.default_rng(21)
    w = rng.standard_normal((5, 200, 512), dtype=np.float32) * np.float32(0.02)
    _prep_and_compare(lib, w)


def test_prepare_weight_prefill_full(lib):
    rng = np.random.default_rng(4)
    w = rng.standard_normal((8192, 8192), dtype=np.float32) * np.float32(0.02)
    _prep_and_compare(lib, w)
