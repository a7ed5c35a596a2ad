import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


class GuardBytes:
    """Places every device output and workspace the binding allocates between
    two 4 KiB guard regions of a fixed pseudo-random byte pattern, and checks
    after each test that no kernel wrote into them: a store past the end of
    an output (rows >= M, columns past N in the last row, 8x4 scale rows past
    ceil8(M), the workspace's tail) or before its start changes a guard byte.
    Buffers allocated while a CUDA graph is being captured are left plain."""
    G = 4096

    def __init__(self):
        self.live = []
        self.pattern = {}

    def _pattern(self, device):
        import torch
        key = str(device)
        if key not in self.pattern:
            g = torch.Generator().manual_seed(1234)
            self.pattern[key] = torch.randint(0, 256, (2 * self.G,), dtype=torch.uint8, generator=g).to(device)
        return self.pattern[key]

    def alloc(self, shape, dtype, device):
        import torch
        if torch.device(device).type == "cuda" and torch.cuda.is_current_stream_capturing():
            return torch.empty(shape, dtype=dtype, device=device)
        numel = 1
        for d in shape:
            numel *= int(d)
        nbytes = numel * torch.empty((), dtype=dtype).element_size()
        raw = torch.empty((2 * self.G + nbytes,), dtype=torch.uint8, device=device)
        pat = self._pattern(device)
        raw[:self.G].copy_(pat[:self.G])
        raw[self.G + nbytes:].copy_(pat[self.G:])
        self.live.append((raw, nbytes, tuple(int(d) for d in shape), dtype))
        return raw[self.G:self.G + nbytes].view(dtype).view(shape)

    def check(self):
        if not self.live:
            return
        import torch
        live, self.live = self.live, []
        if any(raw.is_cuda for raw, _, _, _ in live):
            torch.cuda.synchronize()
        for raw, nbytes, shape, dtype in live:
            pat = self._pattern(raw.device)
            head_bad = (raw[:self.G] != pat[:self.G]).nonzero()
            tail_bad = (raw[self.G + nbytes:] != pat[self.G:]).nonzero()
            if head_bad.numel() or tail_bad.numel():
                where = ("%d bytes before the start (first at -%d)" % (head_bad.numel(), self.G - int(head_bad[0]))
                         if head_bad.numel() else
                         "%d bytes past the end (first at +%d)" % (tail_bad.numel(), int(tail_bad[0])))
                raise AssertionError("guard bytes of a %s %s buffer (%d bytes) were overwritten: %s"
                                     % (dtype, shape, nbytes, where))


GUARDS = GuardBytes()


@pytest.fixture(scope="session")
def lib():
    """The CUDA library's Python binding (built in-tree by __graft_entry__.build),
    with every output and workspace it allocates placed between guard bytes."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp8_block_scaled_x4_gb300 as mx
    mx.set_allocator(GUARDS.alloc)
    return mx


@pytest.fixture(autouse=True)
def _check_guard_bytes():
    """After every test: the guard bytes around the buffers it had the
    binding allocate are intact."""
    yield
    GUARDS.check()


@pytest.fixture(autouse=True)
def _check_device_error(request):
    """After every test that used the CUDA library: no kernel of it gave up
    a bounded wait (a timeout skips that CTA's remaining tiles, which shows
    in a parity check only for the rows it happens to sample) and, in the
    debug build, none computed an out-of-bounds store index.  Reads and
    clears the device error words; tests that provoke a timeout read and
    clear it themselves."""
    yield
    if "lib" not in request.fixturenames:
        return
    import mxfp8_block_scaled_x4_gb300 as mx
    err = mx.device_error()
    assert err == 0, "device error after the test: %s" % mx.status_string(err)
