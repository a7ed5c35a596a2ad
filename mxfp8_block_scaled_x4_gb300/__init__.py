"""GB300 (sm_103a) MXFP8 block-scaled linear layer: Python binding.

A thin ctypes layer over the C ABI of ``include/mxfp8.h`` (the shared library
``_lib/libmxfp8_gb300.so``, built in-tree by ``_build.py``).  This module only
marshals arguments -- shapes, device pointers and the current CUDA stream --
and allocates outputs with PyTorch; every step of the layer runs in the
library's CUDA kernels.  There is no fallback: if the library is missing or
the device is not a GB300, calls raise.

The layer (vLLM PR #52204 "[Kernel] Add FlashInfer TRTLLM MXFP8 linear
backend"): weights are prepared once (MXFP8 quantization with one E8M0 scale
per 32 K elements, N padded to 128, GEMM layout); each call quantizes the BF16
activations with the 8x4 scale layout, runs the block-scaled GEMM with FP32
accumulation, slices the padded N and adds the bias, writing BF16.
"""
import ctypes
import os

import torch

__all__ = [
    "Mxfp8Error", "PreparedWeight", "prepare_weight", "quantize_act", "gemm",
    "linear", "linear_host", "linear_host_workspace_bytes", "grouped_linear", "act_scale_bytes", "weight_bytes",
    "weight_scale_bytes", "linear_workspace_bytes", "set_schedule",
    "device_error", "library", "library_path",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
# MXFP8_DEBUG_LIBRARY=1 in the environment selects the debug build (every
# computed store index checked; see mxfp8_device_error) for this process.
_LIB_PATH = os.path.join(_HERE, "_lib", "libmxfp8_gb300_debug.so" if os.environ.get("MXFP8_DEBUG_LIBRARY") == "1"
                         else "libmxfp8_gb300.so")

OK = 0
STATUS_NAMES = {
    0: "MXFP8_OK", 1: "MXFP8_ERR_INVALID_ARG", 2: "MXFP8_ERR_K_NOT_MULTIPLE_OF_256",
    3: "MXFP8_ERR_MISALIGNED", 4: "MXFP8_ERR_UNSUPPORTED_DEVICE",
    5: "MXFP8_ERR_WORKSPACE_TOO_SMALL", 6: "MXFP8_ERR_DEVICE_TIMEOUT", 7: "MXFP8_ERR_CUDA",
    8: "MXFP8_ERR_OUT_OF_BOUNDS",
}
IN_F32 = 0
IN_BF16 = 1


class Mxfp8Error(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = "%s: %s (%s)" % (where, STATUS_NAMES.get(status, status),
                               _lib_status_string(status))
        if status == 7:
            msg += ", cudaError %d" % library().mxfp8_last_cuda_error()
        super().__init__(msg)


class mxfp8_weight(ctypes.Structure):
    """Mirror of ``struct mxfp8_weight`` in include/mxfp8.h."""
    _fields_ = [("num_experts", ctypes.c_int64), ("n", ctypes.c_int64),
                ("n_pad", ctypes.c_int64), ("k", ctypes.c_int64),
                ("q", ctypes.c_void_p), ("sf", ctypes.c_void_p)]


_lib = None


_allocator = None


def _alloc(shape, dtype, device):
    """Every device output and workspace this module allocates comes from here."""
    if _allocator is not None:
        return _allocator(shape, dtype, device)
    return torch.empty(shape, dtype=dtype, device=device)


def set_allocator(fn=None) -> None:
    """Testing aid: allocate every device output and workspace of this module
    with fn(shape, dtype, device) instead of torch.empty (None restores it).
    The GPU tests use it to place each buffer between guard bytes."""
    global _allocator
    _allocator = fn


def library_path() -> str:
    return _LIB_PATH


def library():
    """The loaded C library (ctypes.CDLL) with argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            "MXFP8 CUDA library not built: %s is missing (run "
            "`python -c 'import __graft_entry__ as g; g.build()'` or "
            "`python mxfp8_block_scaled_x4_gb300/_build.py`)" % _LIB_PATH)
    lib = ctypes.CDLL(_LIB_PATH)
    i64, vp, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    W = ctypes.POINTER(mxfp8_weight)
    sig = {
        "mxfp8_act_scale_bytes": (sz, [i64, i64]),
        "mxfp8_weight_bytes": (sz, [i64, i64]),
        "mxfp8_weight_scale_bytes": (sz, [i64, i64]),
        "mxfp8_linear_workspace_bytes": (sz, [i64, i64]),
        "mxfp8_weight_view": (ctypes.c_int, [W, i64, i64, i64, vp, vp]),
        "mxfp8_prepare_weight": (ctypes.c_int, [vp, ctypes.c_int, W, vp]),
        "mxfp8_quantize_act": (ctypes.c_int, [vp, i64, i64, vp, vp, vp]),
        "mxfp8_gemm": (ctypes.c_int, [vp, vp, i64, W, vp, vp, vp]),
        "mxfp8_linear": (ctypes.c_int, [vp, i64, W, vp, vp, vp, sz, vp]),
        "mxfp8_grouped_linear": (ctypes.c_int, [vp, i64, vp, W, vp, vp, vp, sz, vp]),
        "mxfp8_linear_host_workspace_bytes": (sz, [i64, i64, i64]),
        "mxfp8_linear_host": (ctypes.c_int, [vp, i64, W, vp, vp, vp, sz, vp]),
        "mxfp8_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "mxfp8_last_cuda_error": (ctypes.c_int, []),
        "mxfp8_device_error": (ctypes.c_int, []),
        "mxfp8_set_schedule": (None, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
        "mxfp8_linear_static_scratch": (ctypes.c_int, [vp, i64, W, vp, vp, vp]),
        "mxfp8_last_schedule": (None, [ctypes.POINTER(ctypes.c_int)]),
        "mxfp8_set_wait_limit_ns": (None, [ctypes.c_uint64]),
        "mxfp8_set_pipes": (None, [ctypes.c_int]),
        "mxfp8_static_scratch_last_cuda_error": (ctypes.c_int, []),
        "mxfp8_act_scale_bytes_128x4": (sz, [i64, i64]),
        "mxfp8_linear_128x4_workspace_bytes": (sz, [i64, i64]),
        "mxfp8_quantize_act_128x4": (ctypes.c_int, [vp, i64, i64, vp, vp, vp]),
        "mxfp8_gemm_128x4": (ctypes.c_int, [vp, vp, i64, W, vp, vp, vp]),
        "mxfp8_linear_128x4": (ctypes.c_int, [vp, i64, W, vp, vp, vp, sz, vp]),
        "mxfp8_autotune_linear": (ctypes.c_int, [vp, i64, W, vp, vp, vp, sz, ctypes.c_int, vp, vp]),
        "mxfp8_autotune_grouped_linear": (ctypes.c_int, [vp, i64, vp, W, vp, vp, vp, sz, ctypes.c_int, vp, vp]),
        "mxfp8_tactic_get": (ctypes.c_int, [ctypes.c_int, i64, i64, i64, i64, vp]),
        "mxfp8_tactic_set": (ctypes.c_int, [ctypes.c_int, i64, i64, i64, i64, vp]),
        "mxfp8_tactic_clear": (None, []),
        "mxfp8_plan_tactic": (ctypes.c_int, [ctypes.c_int, i64, i64, i64, i64, ctypes.c_int, vp]),
        "mxfp8_tactic_count": (i64, []),
        "mxfp8_moe_route_workspace_bytes": (sz, [i64, i64, i64]),
        "mxfp8_moe_route": (ctypes.c_int, [vp, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp, vp, vp, sz, vp]),
        "mxfp8_prepare_gate_up_weight": (ctypes.c_int, [vp, ctypes.c_int, W, vp]),
        "mxfp8_moe_gate_up_workspace_bytes": (sz, [i64, i64]),
        "mxfp8_moe_gate_up_swiglu": (ctypes.c_int, [vp, vp, i64, vp, W, vp, vp, sz, vp]),
        "mxfp8_moe_finalize": (ctypes.c_int, [vp, vp, vp, i64, i64, i64, vp, vp]),
        "mxfp8_moe_workspace_bytes": (sz, [i64, i64, i64, i64, i64]),
        "mxfp8_moe_expert_mlp": (ctypes.c_int, [vp, vp, i64, i64, ctypes.c_int, W, W, vp, vp, sz, vp]),
        "mxfp8_debug_build": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _lib_status_string(status):
    try:
        return library().mxfp8_status_string(int(status)).decode()
    except Exception:  # noqa: BLE001 - message formatting only
        return "?"


def status_string(status: int) -> str:
    return library().mxfp8_status_string(int(status)).decode()


def last_cuda_error() -> int:
    """cudaError_t of this thread's last call that returned MXFP8_ERR_CUDA."""
    return library().mxfp8_last_cuda_error()


def _check(status, where):
    if status != OK:
        raise Mxfp8Error(status, where)


def _stream(t: torch.Tensor):
    """The current stream of t's device.  The library launches on the
    current CUDA device, so t must live there."""
    if t.device.index != torch.cuda.current_device():
        raise ValueError("tensor on %s but the current CUDA device is cuda:%d (use torch.cuda.device)"
                         % (t.device, torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


# ----------------------------------------------------------------- sizes
def act_scale_bytes(m: int, k: int) -> int:
    return library().mxfp8_act_scale_bytes(m, k)


def weight_bytes(n: int, k: int) -> int:
    return library().mxfp8_weight_bytes(n, k)


def weight_scale_bytes(n: int, k: int) -> int:
    return library().mxfp8_weight_scale_bytes(n, k)


def linear_workspace_bytes(m: int, k: int) -> int:
    return library().mxfp8_linear_workspace_bytes(m, k)


# ----------------------------------------------------------------- weights
class PreparedWeight:
    """A prepared MXFP8 weight: device buffers + the C struct viewing them.

    q  : uint8 [num_experts, n_pad, k]    E4M3 data (rows >= n are zero)
    sf : uint8 [num_experts, n_pad*k/32]  E8M0 scales, 128x4 tiles
    n  : logical output features (the padded N is sliced away per call)."""

    def __init__(self, q: torch.Tensor, sf: torch.Tensor, n: int):
        e, n_pad, k = q.shape
        self.q, self.sf, self.n, self.k, self.num_experts = q, sf, n, k, e
        self.n_pad = n_pad
        self.c = mxfp8_weight()
        _check(library().mxfp8_weight_view(ctypes.byref(self.c), e, n, k, _ptr(q), _ptr(sf)),
               "mxfp8_weight_view")

    @property
    def device(self):
        return self.q.device


def prepare_weight(w: torch.Tensor, out: PreparedWeight = None) -> PreparedWeight:
    """Quantize + pad + lay out a weight [n, k] (or stacked experts
    [e, n, k]) given as float32 or bfloat16 on the GPU.

    out: an existing PreparedWeight of the same shape to re-prepare in place
    (a weight refit: its buffers keep their addresses, so CUDA graphs that
    captured calls on it stay valid and see the new weight on replay)."""
    _need(w.is_cuda, "weight must be a CUDA tensor")
    _need(w.dtype in (torch.float32, torch.bfloat16), "weight must be float32 or bfloat16")
    w3 = w.unsqueeze(0) if w.dim() == 2 else w
    _need(w3.dim() == 3, "weight must be [n, k] or [experts, n, k]")
    w3 = w3.contiguous()
    e, n, k = w3.shape
    n_pad = (n + 127) // 128 * 128
    if out is not None:
        _need((out.num_experts, out.n, out.k) == (e, n, k), "refit needs a weight of the same shape")
        pw = out
    else:
        q = _alloc((e, n_pad, k), torch.uint8, w.device)
        sf = _alloc((e, n_pad * (k // 32)), torch.uint8, w.device)
        pw = PreparedWeight(q, sf, n)
    dt = IN_BF16 if w3.dtype == torch.bfloat16 else IN_F32
    _check(library().mxfp8_prepare_weight(_ptr(w3), dt, ctypes.byref(pw.c), _stream(w)),
           "mxfp8_prepare_weight")
    return pw


# -------------------------------------------------------------- activations
def _out(t, shape, dtype, dev, what):
    """A caller-given output tensor (checked) or a new one."""
    if t is None:
        return _alloc(shape, dtype, dev)
    _need(t.is_cuda and t.dtype == dtype and t.is_contiguous() and t.numel() >= _numel(shape),
          "%s must be a contiguous %s CUDA tensor of at least %s elements" % (what, dtype, _numel(shape)))
    return t


def _numel(shape):
    n = 1
    for d in shape:
        n *= int(d)
    return n


def quantize_act(x: torch.Tensor, q=None, sf=None):
    """BF16 [m, k] -> (E4M3 bytes uint8 [m, k], 8x4 scales uint8 [ceil8(m)*k/32]).
    q, sf: optional caller buffers to write into."""
    _need(x.is_cuda and x.dtype == torch.bfloat16, "x must be a bfloat16 CUDA tensor")
    x2 = x.reshape(-1, x.shape[-1]).contiguous()
    m, k = x2.shape
    q = _out(q, (m, k), torch.uint8, x.device, "q")
    sf = _out(sf, (max(act_scale_bytes(m, k), 1),), torch.uint8, x.device, "sf")
    _check(library().mxfp8_quantize_act(_ptr(x2), m, k, _ptr(q), _ptr(sf), _stream(x)),
           "mxfp8_quantize_act")
    return q, sf[:act_scale_bytes(m, k)]


def gemm(qa: torch.Tensor, sfa: torch.Tensor, pw: PreparedWeight, bias=None, out=None) -> torch.Tensor:
    """Block-scaled GEMM on pre-quantized activations -> BF16 [m, n]
    (written into `out` when given)."""
    m = qa.shape[0]
    y = _out(out, (m, pw.n), torch.bfloat16, qa.device, "out")
    _check(library().mxfp8_gemm(_ptr(qa), _ptr(sfa), m, ctypes.byref(pw.c), _ptr(bias), _ptr(y),
                                _stream(qa)), "mxfp8_gemm")
    return y


def linear(x: torch.Tensor, pw: PreparedWeight, bias=None, workspace=None, out=None) -> torch.Tensor:
    """The layer: BF16 x [..., k] -> BF16 [..., n] (leading dims kept, as
    apply_weights does).  out: optional contiguous BF16 buffer for y."""
    _need(x.is_cuda and x.dtype == torch.bfloat16, "x must be a bfloat16 CUDA tensor")
    _need(x.shape[-1] == pw.k, "x's last dim must equal the weight's K")
    lead = x.shape[:-1]
    x2 = x.reshape(-1, pw.k).contiguous()
    m = x2.shape[0]
    if bias is not None:
        _need(bias.dtype == torch.bfloat16 and bias.numel() == pw.n, "bias must be bf16 [n]")
    ws_need = linear_workspace_bytes(m, pw.k)
    if workspace is None:
        workspace = _alloc((max(ws_need, 16),), torch.uint8, x.device)
    y = _out(out, (m, pw.n), torch.bfloat16, x.device, "out")
    _check(library().mxfp8_linear(_ptr(x2), m, ctypes.byref(pw.c), _ptr(bias), _ptr(y),
                                  _ptr(workspace), workspace.numel(), _stream(x)), "mxfp8_linear")
    return y.view(-1)[:m * pw.n].view(*lead, pw.n)


def linear_host_workspace_bytes(m: int, n: int, k: int) -> int:
    return library().mxfp8_linear_host_workspace_bytes(m, n, k)


def linear_host(x_host: torch.Tensor, pw: PreparedWeight, bias=None, y_host=None, workspace=None,
                stream=None) -> torch.Tensor:
    """The layer on host buffers: bf16 CPU x [m, k] -> bf16 CPU y [m, n].
    One library call enqueues the copy in, the layer and the copy out on
    `stream` (default: the current stream); y_host is valid after that
    stream has synchronised.  Pass page-locked tensors (pin_memory()) to
    keep the copies asynchronous."""
    _need(not x_host.is_cuda and x_host.dtype == torch.bfloat16 and x_host.is_contiguous(),
          "x_host must be a contiguous bfloat16 CPU tensor")
    _need(x_host.dim() == 2 and x_host.shape[1] == pw.k, "x_host must be [m, k]")
    m = x_host.shape[0]
    if y_host is None:
        y_host = torch.empty((m, pw.n), dtype=torch.bfloat16, pin_memory=x_host.is_pinned())
    _need(not y_host.is_cuda and y_host.dtype == torch.bfloat16 and y_host.is_contiguous()
          and tuple(y_host.shape) == (m, pw.n), "y_host must be a contiguous bfloat16 CPU tensor [m, n]")
    if bias is not None:
        _need(bias.is_cuda and bias.dtype == torch.bfloat16 and bias.numel() == pw.n, "bias must be bf16 CUDA [n]")
    if workspace is None:
        workspace = _alloc((max(linear_host_workspace_bytes(m, pw.n, pw.k), 16),), torch.uint8,
                           torch.device("cuda", torch.cuda.current_device()))
    _need(workspace.is_cuda and workspace.device.index == torch.cuda.current_device(),
          "workspace must be on the current CUDA device")
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    _check(library().mxfp8_linear_host(_ptr(x_host), m, ctypes.byref(pw.c), _ptr(bias), _ptr(y_host),
                                       _ptr(workspace), workspace.numel(), ctypes.c_void_p(stream.cuda_stream)),
           "mxfp8_linear_host")
    return y_host


def grouped_linear(x_sorted: torch.Tensor, offsets: torch.Tensor, pw: PreparedWeight,
                   bias=None, workspace=None, out=None) -> torch.Tensor:
    """Per-expert layer over expert-sorted rows: x_sorted bf16 [rows, k],
    offsets int32 [e+1] (device) -> bf16 [rows, n]."""
    _need(x_sorted.is_cuda and x_sorted.dtype == torch.bfloat16, "x_sorted must be bf16 CUDA")
    _need(offsets.dtype == torch.int32 and offsets.is_cuda, "offsets must be int32 CUDA")
    _need(offsets.numel() == pw.num_experts + 1, "offsets must have num_experts + 1 entries")
    rows = x_sorted.shape[0]
    x2 = x_sorted.contiguous()
    ws_need = linear_workspace_bytes(rows, pw.k)
    if workspace is None:
        workspace = _alloc((max(ws_need, 16),), torch.uint8, x_sorted.device)
    y = _out(out, (rows, pw.n), torch.bfloat16, x_sorted.device, "out")
    _check(library().mxfp8_grouped_linear(_ptr(x2), rows, _ptr(offsets.contiguous()),
                                          ctypes.byref(pw.c), _ptr(bias), _ptr(y),
                                          _ptr(workspace), workspace.numel(), _stream(x_sorted)),
           "mxfp8_grouped_linear")
    return y


def linear_static_scratch(x: torch.Tensor, pw: PreparedWeight, bias=None, out=None) -> torch.Tensor:
    """The layer with the library's own static scratch instead of a caller
    workspace (the library allocates nothing; calls whose kernels overlap on
    the GPU must not share it).  bf16 [m, k] -> bf16 [m, n]."""
    _need(x.is_cuda and x.dtype == torch.bfloat16, "x must be a bfloat16 CUDA tensor")
    _need(x.dim() == 2 and x.shape[1] == pw.k, "x must be [m, k]")
    if bias is not None:
        _need(bias.dtype == torch.bfloat16 and bias.numel() == pw.n, "bias must be bf16 [n]")
    x2 = x.contiguous()
    y = _out(out, (x2.shape[0], pw.n), torch.bfloat16, x.device, "out")
    _check(library().mxfp8_linear_static_scratch(_ptr(x2), x2.shape[0], ctypes.byref(pw.c), _ptr(bias),
                                                 _ptr(y), _stream(x)), "mxfp8_linear_static_scratch")
    return y


# -------------------------------------------------- 128x4 activation scales
def act_scale_bytes_128x4(m: int, k: int) -> int:
    return library().mxfp8_act_scale_bytes_128x4(m, k)


def linear_128x4_workspace_bytes(m: int, k: int) -> int:
    return library().mxfp8_linear_128x4_workspace_bytes(m, k)


def quantize_act_128x4(x: torch.Tensor, q=None, sf=None):
    """BF16 [m, k] -> (E4M3 bytes [m, k], scales in the 128x4 layout
    [ceil128(m) * k/32]); q, sf: optional caller buffers."""
    _need(x.is_cuda and x.dtype == torch.bfloat16, "x must be a bfloat16 CUDA tensor")
    x2 = x.reshape(-1, x.shape[-1]).contiguous()
    m, k = x2.shape
    nsf = library().mxfp8_act_scale_bytes_128x4(m, k)
    q = _out(q, (m, k), torch.uint8, x.device, "q")
    sf = _out(sf, (max(nsf, 1),), torch.uint8, x.device, "sf")
    _check(library().mxfp8_quantize_act_128x4(_ptr(x2), m, k, _ptr(q), _ptr(sf), _stream(x)),
           "mxfp8_quantize_act_128x4")
    return q, sf[:nsf]


def gemm_128x4(qa: torch.Tensor, sfa: torch.Tensor, pw: PreparedWeight, bias=None, out=None) -> torch.Tensor:
    m = qa.shape[0]
    y = _out(out, (m, pw.n), torch.bfloat16, qa.device, "out")
    _check(library().mxfp8_gemm_128x4(_ptr(qa.contiguous()), _ptr(sfa.contiguous()), m, ctypes.byref(pw.c),
                                      _ptr(bias), _ptr(y), _stream(qa)), "mxfp8_gemm_128x4")
    return y


def linear_128x4(x: torch.Tensor, pw: PreparedWeight, bias=None, workspace=None, out=None) -> torch.Tensor:
    """The layer with 128x4 activation scales (the high-M variant)."""
    _need(x.is_cuda and x.dtype == torch.bfloat16, "x must be bf16 CUDA")
    lead = x.shape[:-1]
    x2 = x.reshape(-1, x.shape[-1]).contiguous()
    m = x2.shape[0]
    need = library().mxfp8_linear_128x4_workspace_bytes(m, pw.k)
    if workspace is None:
        workspace = _alloc((max(need, 16),), torch.uint8, x.device)
    y = _out(out, (m, pw.n), torch.bfloat16, x.device, "out")
    _check(library().mxfp8_linear_128x4(_ptr(x2), m, ctypes.byref(pw.c), _ptr(bias), _ptr(y), _ptr(workspace),
                                        workspace.numel(), _stream(x)), "mxfp8_linear_128x4")
    return y.view(-1)[:m * pw.n].view(*lead, pw.n)


# ----------------------------------------------------------------- tactics
KIND_LINEAR, KIND_GEMM, KIND_GROUPED, KIND_GATED = 0, 1, 2, 3


def _tactic_array(t=None):
    a = (ctypes.c_int32 * 4)()
    if t is not None:
        for i, v in enumerate(t):
            a[i] = int(v)
    return a


def autotune_linear(x: torch.Tensor, pw: PreparedWeight, bias=None, iters: int = 20, workspace=None):
    """Time every valid tactic for this linear call on these buffers, store
    the fastest in the tactic table and return it (tokens per tile, split_k,
    fuse_quant, pipes).  Synchronous."""
    _need(x.is_cuda and x.dtype == torch.bfloat16, "x must be bf16 CUDA")
    x2 = x.reshape(-1, x.shape[-1]).contiguous()
    m = x2.shape[0]
    if workspace is None:
        workspace = _alloc((max(linear_workspace_bytes(m, pw.k), 16),), torch.uint8, x.device)
    y = _alloc((m, pw.n), torch.bfloat16, x.device)
    out = _tactic_array()
    _check(library().mxfp8_autotune_linear(_ptr(x2), m, ctypes.byref(pw.c), _ptr(bias), _ptr(y), _ptr(workspace),
                                           workspace.numel(), iters, _stream(x), out), "mxfp8_autotune_linear")
    return tuple(out)


def autotune_grouped_linear(x_sorted: torch.Tensor, offsets: torch.Tensor, pw: PreparedWeight, bias=None,
                            iters: int = 20, workspace=None):
    """autotune_linear for the grouped (MoE expert) layer."""
    _need(x_sorted.is_cuda and x_sorted.dtype == torch.bfloat16, "x_sorted must be bf16 CUDA")
    x2 = x_sorted.contiguous()
    rows = x2.shape[0]
    if workspace is None:
        workspace = _alloc((max(linear_workspace_bytes(rows, pw.k), 16),), torch.uint8, x_sorted.device)
    y = _alloc((rows, pw.n), torch.bfloat16, x_sorted.device)
    out = _tactic_array()
    _check(library().mxfp8_autotune_grouped_linear(_ptr(x2), rows, _ptr(offsets.contiguous()), ctypes.byref(pw.c),
                                                   _ptr(bias), _ptr(y), _ptr(workspace), workspace.numel(), iters,
                                                   _stream(x_sorted), out), "mxfp8_autotune_grouped_linear")
    return tuple(out)


def tactic_get(kind: int, m: int, n: int, k: int, experts: int = 1):
    """The stored tactic for a call class, or None."""
    out = _tactic_array()
    st = library().mxfp8_tactic_get(kind, m, n, k, experts, out)
    return tuple(out) if st == OK else None


def tactic_set(kind: int, m: int, n: int, k: int, experts: int, tactic) -> None:
    _check(library().mxfp8_tactic_set(kind, m, n, k, experts, _tactic_array(tactic)), "mxfp8_tactic_set")


def plan_tactic(kind: int, m: int, n: int, k: int, experts: int = 1, sms: int = 0):
    """The tactic (tokens_per_tile, split_k, fuse_quant, pipes) a call of
    this kind and shape would run now: the table's entry, else the built-in
    heuristic's choice.  sms <= 0 means the current device's SM count."""
    out = (ctypes.c_int32 * 4)()
    _check(library().mxfp8_plan_tactic(kind, m, n, k, experts, sms, out), "mxfp8_plan_tactic")
    return tuple(out)


def tactic_clear() -> None:
    library().mxfp8_tactic_clear()


def tactic_count() -> int:
    return int(library().mxfp8_tactic_count())


# -------------------------------------------------------------------- MoE
ROUTE_RENORMALIZE = 0
ROUTE_RENORMALIZE_NAIVE = 1


class Routing:
    """Device outputs of moe_route: topk ids/weights [t, k], expert offsets
    [e+1], sorted_token [t*k] (token of each expert-sorted row) and row_of
    [t*k] (sorted row of pair (t, s) at t*k + s)."""

    def __init__(self, ids, weights, offsets, sorted_token, row_of):
        self.ids, self.weights, self.offsets = ids, weights, offsets
        self.sorted_token, self.row_of = sorted_token, row_of


def moe_route(logits: torch.Tensor, topk: int, method: int = ROUTE_RENORMALIZE) -> Routing:
    """Top-k routing of float32 logits [tokens, experts] and the stable
    expert-sorted order of the (token, slot) pairs."""
    _need(logits.is_cuda and logits.dtype == torch.float32 and logits.dim() == 2,
          "logits must be a float32 CUDA tensor [tokens, experts]")
    lg = logits.contiguous()
    t, e = lg.shape
    dev = logits.device
    ids = _alloc((t, topk), torch.int32, dev)
    w = _alloc((t, topk), torch.float32, dev)
    off = _alloc((e + 1,), torch.int32, dev)
    stok = _alloc((max(t * topk, 1),), torch.int32, dev)
    row_of = _alloc((max(t * topk, 1),), torch.int32, dev)
    nws = library().mxfp8_moe_route_workspace_bytes(t, e, topk)
    ws = _alloc((max(nws, 16),), torch.uint8, dev)
    _check(library().mxfp8_moe_route(_ptr(lg), t, e, topk, method, _ptr(ids), _ptr(w), _ptr(off),
                                     _ptr(stok), _ptr(row_of), _ptr(ws), ws.numel(), _stream(logits)),
           "mxfp8_moe_route")
    return Routing(ids, w, off, stok[:t * topk], row_of[:t * topk])


def prepare_gate_up_weight(w13: torch.Tensor, out: PreparedWeight = None) -> PreparedWeight:
    """GEMM1 weights [experts, 2*I, k] (rows [gate; up]) -> prepared with the
    gated-row reorder (tile j = gate rows 64j.. then up rows I+64j..)."""
    _need(w13.is_cuda and w13.dtype in (torch.float32, torch.bfloat16) and w13.dim() == 3,
          "w13 must be a float32/bfloat16 CUDA tensor [experts, 2I, k]")
    w3 = w13.contiguous()
    e, n, k = w3.shape
    if out is not None:
        _need((out.num_experts, out.n, out.k) == (e, n, k), "refit needs a weight of the same shape")
        pw = out
    else:
        q = _alloc((e, n, k), torch.uint8, w13.device)
        sf = _alloc((e, n * (k // 32)), torch.uint8, w13.device)
        pw = PreparedWeight(q, sf, n)
    dt = IN_BF16 if w3.dtype == torch.bfloat16 else IN_F32
    _check(library().mxfp8_prepare_gate_up_weight(_ptr(w3), dt, ctypes.byref(pw.c), _stream(w13)),
           "mxfp8_prepare_gate_up_weight")
    return pw


def moe_gate_up_swiglu(x: torch.Tensor, routing: Routing, w13: PreparedWeight, out=None, workspace=None) -> torch.Tensor:
    """h [t*k, I] bf16 = silu(gate) * up of GEMM1 on the expert-sorted,
    MXFP8-quantized token rows."""
    _need(x.is_cuda and x.dtype == torch.bfloat16, "x must be bf16 CUDA")
    x2 = x.contiguous()
    rows = routing.sorted_token.numel()
    h = _out(out, (rows, w13.n // 2), torch.bfloat16, x.device, "out")
    nws = library().mxfp8_moe_gate_up_workspace_bytes(rows, w13.k)
    ws = workspace if workspace is not None else _alloc((max(nws, 16),), torch.uint8, x.device)
    _check(library().mxfp8_moe_gate_up_swiglu(_ptr(x2), _ptr(routing.sorted_token), rows,
                                              _ptr(routing.offsets), ctypes.byref(w13.c), _ptr(h),
                                              _ptr(ws), ws.numel(), _stream(x)),
           "mxfp8_moe_gate_up_swiglu")
    return h


def moe_finalize(y2: torch.Tensor, routing: Routing, out=None) -> torch.Tensor:
    """out [t, hidden] bf16 = per token, the routing-weighted sum of its k
    expert outputs y2 [t*k, hidden] (expert-sorted rows)."""
    t, k = routing.ids.shape
    hidden = y2.shape[1]
    out = _out(out, (t, hidden), torch.bfloat16, y2.device, "out")
    _check(library().mxfp8_moe_finalize(_ptr(y2.contiguous()), _ptr(routing.row_of), _ptr(routing.weights),
                                        t, k, hidden, _ptr(out), _stream(y2)),
           "mxfp8_moe_finalize")
    return out


def moe_expert_mlp(x: torch.Tensor, logits: torch.Tensor, topk: int, w13: PreparedWeight,
                   w2: PreparedWeight, method: int = ROUTE_RENORMALIZE, workspace=None, out=None) -> torch.Tensor:
    """The whole expert MLP: route -> gate_up + SwiGLU -> down -> finalize."""
    _need(x.is_cuda and x.dtype == torch.bfloat16, "x must be bf16 CUDA")
    _need(logits.is_cuda and logits.dtype == torch.float32, "logits must be float32 CUDA")
    t, hdim = x.shape
    e = w13.num_experts
    nws = library().mxfp8_moe_workspace_bytes(t, e, topk, hdim, w13.n // 2)
    if workspace is None:
        workspace = _alloc((max(nws, 16),), torch.uint8, x.device)
    out = _out(out, (t, hdim), torch.bfloat16, x.device, "out")
    _check(library().mxfp8_moe_expert_mlp(_ptr(x.contiguous()), _ptr(logits.contiguous()), t, topk, method,
                                          ctypes.byref(w13.c), ctypes.byref(w2.c), _ptr(out),
                                          _ptr(workspace), workspace.numel(), _stream(x)),
           "mxfp8_moe_expert_mlp")
    return out


def moe_workspace_bytes(tokens, experts, topk, hidden, inter) -> int:
    return library().mxfp8_moe_workspace_bytes(tokens, experts, topk, hidden, inter)


# ------------------------------------------------------------------ hooks
def set_schedule(tokens_per_tile: int = 0, split_k: int = 0, fuse_quant: int = -1) -> None:
    """Pin the GEMM schedule (testing/benchmarking).  tokens_per_tile 0 = auto,
    16..256, or 144 / 160 / 176 / 192 = two weight tiles per CTA tile (dense); split_k 0 =
    auto, -1 = persistent, >0 = one tile per cluster of split_k CTAs;
    fuse_quant -1 = auto, 0 = off, 1 = on where possible."""
    library().mxfp8_set_schedule(int(tokens_per_tile), int(split_k), int(fuse_quant))


def set_pipes(pipes: int = 0) -> None:
    """MMA pipelines per CTA for later launches (0 = automatic; testing aid)."""
    library().mxfp8_set_pipes(int(pipes))


def last_schedule() -> dict:
    """Schedule of this thread's last GEMM launch (testing aid)."""
    out = (ctypes.c_int * 5)()
    library().mxfp8_last_schedule(out)
    return {"tokens_per_tile": out[0] % 1000, "pipes": out[0] // 1000 + 1, "split": out[1],
            "fused": bool(out[2]), "grid": out[3], "stages": out[4]}


def set_wait_limit_ns(ns: int = 0) -> None:
    """Limit of every pipeline wait in later GEMM launches (0 = default 4 s).
    Testing aid for the timeout path."""
    library().mxfp8_set_wait_limit_ns(int(ns))


def device_error() -> int:
    """Synchronise and read/clear the kernels' device-side error words
    (timeout; out-of-bounds store in the debug build)."""
    return library().mxfp8_device_error()


def debug_build() -> bool:
    """True when the loaded library is the debug build."""
    return bool(library().mxfp8_debug_build())
