"""GPU parity: the dense MXFP8 linear layer (quantize + block-scaled GEMM +
padded-N slice + bias) against the CPU oracle, per element within
|y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref) (see gpu_common)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads
from gpu_common import assert_close_to_oracle, oracle_weight, to_dev_bf16, to_dev_f32

pytestmark = pytest.mark.gpu


def _run_dense(mx, d, rows=None, schedule=(0, 0, -1), pipes=0):
    pw = mx.prepare_weight(to_dev_f32(d.w))
    x = to_dev_bf16(d.x)
    b = None if d.bias is None else to_dev_bf16(d.bias)
    mx.set_schedule(*schedule)
    mx.set_pipes(pipes)
    try:
        y = mx.linear(x, pw, b)
        if pipes:
            assert mx.last_schedule()["pipes"] == pipes
    finally:
        mx.set_schedule(0, 0, -1)
        mx.set_pipes(0)
    torch.cuda.synchronize()
    assert y.shape == (d.m, d.n) and y.is_contiguous()
    wq, wsf = oracle_weight(d.w)
    y_ref = oracle.linear(d.x, wq, wsf, d.bias, rows=rows)
    yy = y if rows is None else y[torch.as_tensor(rows, device=y.device)]
    assert_close_to_oracle(yy, y_ref, d.name)
    return y, pw


def test_tiny_config(lib):
    _run_dense(lib, workloads.tiny())


@pytest.mark.parametrize("m", [1, 16])
def test_decode_config(lib, m):
    _run_dense(lib, workloads.decode(m=m))


@pytest.mark.parametrize("n,bias", [(2048, False), (130, True)])
def test_mid_config(lib, n, bias):
    _run_dense(lib, workloads.mid(n=n, bias=bias))


def test_prefill_config_sampled_rows(lib):
    """8192^3: every column of 48 rows -- the first token tile's edges, the
    last row, and seeded random rows."""
    d = workloads.prefill()
    rng = np.random.default_rng(40)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, 4095, 8191],
                                     rng.integers(0, 8192, 40)]))
    _run_dense(lib, d, rows=rows)


@pytest.mark.parametrize("shape", [(1, 130, 256), (7, 256, 512), (128, 130, 768)])
def test_vllm_shapes_cosine_and_oracle(lib, shape):
    """The shapes and acceptance criterion of vLLM PR #52204's GPU test:
    cosine similarity > 0.98 against the unquantized product, output shape
    (m, n) and contiguous; plus the oracle tolerance."""
    m, n, k = shape
    torch.manual_seed(0)
    x = torch.randn((m, k), dtype=torch.bfloat16)
    w = torch.randn((n, k), dtype=torch.bfloat16)
    pw = lib.prepare_weight(w.cuda())
    y = lib.linear(x.cuda(), pw)
    ref = torch.mm(x.float(), w.float().t())
    cos = F.cosine_similarity(y.float().cpu().flatten(), ref.flatten(), dim=0)
    assert y.shape == (m, n) and y.is_contiguous()
    assert cos.item() > 0.98
    wq, wsf = oracle.quantize_rows(w.float().numpy())
    assert_close_to_oracle(y, oracle.linear(x.float().numpy(), wq, wsf), "vllm%s" % (shape,))


@pytest.mark.parametrize("tt,split,fuse", [
    (16, -1, 0), (16, 1, 1), (16, 4, 1), (16, 4, 0), (32, 2, 1), (32, 3, 0), (64, -1, 0),
    (64, 8, 1), (64, 8, 0), (128, -1, 0), (128, 4, 0), (128, 2, 1), (256, -1, 0), (192, -1, 0)])
def test_every_schedule(lib, tt, split, fuse):
    """Each token-tile size, persistent (-1) or one tile per cluster of `split`
    CTAs, with the activation quantization fused into the GEMM or not, on a
    shape with several weight tiles, a ragged N (N_pad > N) and a ragged token
    tail."""
    d = workloads.dense(m=300, n=390, k=1024, seed=30, bias=True)
    _run_dense(lib, d, schedule=(tt, split, fuse))


@pytest.mark.parametrize("tt,split,fuse,pipes", [
    (16, -1, 0, 2), (16, -1, 0, 4), (16, 2, 1, 2), (16, 4, 1, 4), (16, 1, 0, 4), (32, 2, 1, 2),
    (32, -1, 0, 2), (64, 4, 0, 2), (64, -1, 0, 2), (64, 2, 1, 2)])
def test_multi_pipe_schedules(lib, tt, split, fuse, pipes):
    """Several MMA pipelines per CTA (each every pipes-th K block, own
    accumulator, summed in pipe order), persistent and split-K, fused or not;
    K = 1024 gives 8 K blocks, also fewer than one per pipe under split 4."""
    d = workloads.dense(m=300, n=390, k=1024, seed=33, bias=True)
    _run_dense(lib, d, schedule=(tt, split, fuse), pipes=pipes)


@pytest.mark.parametrize("tt", [192, 176, 160, 144])
@pytest.mark.parametrize("m,n,k", [(300, 300, 1024), (1000, 640, 512), (193, 128, 256), (161, 256, 512)])
def test_dual_weight_tile_schedule(lib, m, n, k, tt):
    """Two weight tiles x 160 or 192 tokens per CTA tile (the large-M
    schedule): odd numbers of weight tiles (the pair's second tile out of
    range), ragged token tails, a single weight tile."""
    d = workloads.dense(m=m, n=n, k=k, seed=m + n, bias=True)
    _run_dense(lib, d, schedule=(tt, -1, 0))
    sched = lib.last_schedule()
    assert sched["split"] == -2 and sched["tokens_per_tile"] == tt, sched


def test_dual_schedule_unaligned_output(lib):
    """y only 2-byte aligned (the ABI's minimum): the epilogue must fall back
    from 16-byte stores."""
    d = workloads.dense(m=200, n=256, k=256, seed=35, bias=True)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    x = to_dev_bf16(d.x)
    # sentinel-filled around y: the element before it and the 7 after must stay
    sentinel = torch.tensor([-1234.5], dtype=torch.bfloat16).view(torch.int16).item()
    buf = torch.full((d.m * d.n + 8,), sentinel, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    y = buf[1:1 + d.m * d.n].view(d.m, d.n)  # 2-byte offset from a 256-byte aligned base
    import ctypes
    lib.set_schedule(192, -1, 0)  # the dual weight-tile kernel
    try:
        ws = torch.empty(lib.linear_workspace_bytes(d.m, d.k), dtype=torch.uint8, device="cuda")
        st = lib.library().mxfp8_linear(ctypes.c_void_p(x.data_ptr()), d.m, ctypes.byref(pw.c),
                                        ctypes.c_void_p(to_dev_bf16(d.bias).data_ptr()),
                                        ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                        ws.numel(), None)
        assert st == 0
        torch.cuda.synchronize()
    finally:
        lib.set_schedule(0, 0, -1)
    wq, wsf = oracle_weight(d.w)
    assert_close_to_oracle(y, oracle.linear(d.x, wq, wsf, d.bias), "unaligned y")
    raw = buf.view(torch.int16)
    assert raw[0].item() == sentinel and bool((raw[1 + d.m * d.n:] == sentinel).all())


def test_multi_pipe_fewer_k_blocks_than_pipes(lib):
    """K = 256 is 2 K blocks: with 4 pipelines two of them idle."""
    d = workloads.dense(m=40, n=256, k=256, seed=34, bias=True)
    _run_dense(lib, d, schedule=(16, -1, 0), pipes=4)
    _run_dense(lib, d, schedule=(16, 1, 1), pipes=4)


@pytest.mark.parametrize("m,n,k", [(1, 128, 256), (2, 130, 256), (17, 384, 512), (33, 260, 1024),
                                   (100, 1000, 768), (257, 256, 256), (511, 640, 512)])
def test_ragged_shapes(lib, m, n, k):
    _run_dense(lib, workloads.dense(m=m, n=n, k=k, seed=m + n + k, bias=(m % 2 == 1)))


@pytest.mark.parametrize("m,n,k,schedule", [
    (16, 1000, 16384, (0, 0, -1)),   # built-in choice: split-K clusters, fused quantization
    (16, 1000, 16384, (16, 1, 1)),   # one CTA walks all 128 K blocks: every stage reused many times
    (64, 520, 16384, (64, 2, 1)),    # 64-token tiles, fused, 64 K blocks per CTA
    (200, 260, 16384, (0, 0, -1)),   # persistent tiles, separate quantizer
    (8, 40960, 2048, (0, 0, -1)),    # 320 weight tiles: several waves of clusters
])
def test_long_k_and_wide_n(lib, m, n, k, schedule):
    """Long K (the fused quantizer refills pipeline stages the MMA has
    released) and wide N (more clusters than fit on the GPU at once), with
    ragged N and bias."""
    _run_dense(lib, workloads.dense(m=m, n=n, k=k, seed=m + n + k, bias=True), schedule=schedule)


def test_gemm_matches_linear_bitwise(lib):
    d = workloads.dense(m=77, n=520, k=512, seed=31)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    x = to_dev_bf16(d.x)
    b = to_dev_bf16(d.bias)
    y1 = lib.linear(x, pw, b)
    q, sf = lib.quantize_act(x)
    y2 = lib.gemm(q, sf, pw, b)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_deterministic(lib):
    d = workloads.decode(m=16)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    x = to_dev_bf16(d.x)
    b = to_dev_bf16(d.bias)
    ys = [lib.linear(x, pw, b) for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(ys[0], y) for y in ys[1:])


def test_closed_form_all_ones(lib):
    """x = W = 1: quantization is exact, y = K exactly (a power of two is
    exact in BF16), plus an exactly representable bias."""
    for k in (256, 2048):
        m, n = 20, 200
        pw = lib.prepare_weight(torch.ones((n, k), dtype=torch.float32, device="cuda"))
        x = torch.ones((m, k), dtype=torch.bfloat16, device="cuda")
        y = lib.linear(x, pw)
        assert torch.equal(y, torch.full((m, n), float(k), dtype=torch.bfloat16, device="cuda"))
        b = torch.arange(n, device="cuda", dtype=torch.float32).mul(0.5).to(torch.bfloat16)
        yb = lib.linear(x, pw, b)
        torch.cuda.synchronize()
        # K + bias rounded once to BF16
        ref = (float(k) + b.float()).to(torch.bfloat16).expand(m, n)
        assert torch.equal(yb, ref)


def test_leading_dims_and_m0(lib):
    d = workloads.dense(m=12, n=256, k=256, seed=32)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    x = to_dev_bf16(d.x).reshape(3, 4, 256)
    y = lib.linear(x, pw, to_dev_bf16(d.bias))
    assert y.shape == (3, 4, 256)
    y0 = lib.linear(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"), pw)
    assert y0.shape == (0, 256)


def test_no_device_timeout_recorded(lib):
    assert lib.device_error() == 0


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("mk", ["decode", "mid"])
def test_linear_host_buffers(lib, mk, pinned):
    """mxfp8_linear_host: host x in, host y out, one call; the result is the
    device call's, bit for bit, and within the oracle tolerance."""
    d = workloads.decode(m=16) if mk == "decode" else workloads.mid(n=130, bias=True)
    pw = lib.prepare_weight(to_dev_f32(d.w))
    b = None if d.bias is None else to_dev_bf16(d.bias)
    xh = torch.from_numpy(d.x).to(torch.bfloat16)
    if pinned:
        xh = xh.pin_memory()
    yh = torch.full((d.m, d.n), float("nan"), dtype=torch.bfloat16)
    if pinned:
        yh = yh.pin_memory()
    out = lib.linear_host(xh, pw, b, y_host=yh)
    torch.cuda.synchronize()
    assert out is yh
    y_dev = lib.linear(xh.cuda(), pw, b)
    torch.cuda.synchronize()
    assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))
    wq, wsf = oracle_weight(d.w)
    assert_close_to_oracle(yh, oracle.linear(d.x, wq, wsf, d.bias), d.name + "_host")
