"""The guard-byte checker the GPU tests run after every test (conftest),
exercised on CPU tensors: writes inside a buffer pass, a write one byte past
the end or one byte before the start is reported."""
import pytest
import torch

from conftest import GuardBytes


def test_writes_inside_pass():
    g = GuardBytes()
    y = g.alloc((3, 5), torch.bfloat16, "cpu")
    y.fill_(1.5)
    q = g.alloc((17,), torch.uint8, "cpu")
    q.fill_(7)
    g.check()
    assert g.live == []


@pytest.mark.parametrize("offset", [0, 1, GuardBytes.G - 1])
def test_write_past_the_end_is_reported(offset):
    g = GuardBytes()
    y = g.alloc((3, 5), torch.bfloat16, "cpu")
    raw = g.live[0][0]
    raw[GuardBytes.G + y.numel() * 2 + offset] ^= 0xFF
    with pytest.raises(AssertionError, match="past the end"):
        g.check()


def test_write_before_the_start_is_reported():
    g = GuardBytes()
    g.alloc((4, 4), torch.int32, "cpu")
    raw = g.live[0][0]
    raw[GuardBytes.G - 1] ^= 0x01
    with pytest.raises(AssertionError, match="before the start"):
        g.check()


def test_buffers_are_aligned_views():
    g = GuardBytes()
    y = g.alloc((2, 8), torch.bfloat16, "cpu")
    assert y.is_contiguous() and y.shape == (2, 8)
    assert (y.data_ptr() - g.live[0][0].data_ptr()) == GuardBytes.G
