"""Python binding of ``libfa.so`` (argument marshalling only).

Every function here checks tensor properties, picks output buffers and calls the C ABI
declared in ``include/fa.h`` through ctypes. All arithmetic happens in the CUDA kernels of
``libfa.so``; if that library is missing the functions raise ``FaLibraryMissing`` rather
than compute anything another way.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_ALIGNMENT = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5

# Every symbol include/fa.h declares.
EXPORTS = ("fa_forward", "fa_forward_ex", "fa_forward_splitkv_workspace_bytes",
           "fa_forward_splitkv", "fa_forward_choose_splits", "fa_backward_workspace_bytes",
           "fa_backward",
           "fa_backward_ex", "fa_backward_noalloc", "fa_noalloc_scratch_bytes",
           "fa_forward_backward_host_device_bytes", "fa_naive_softmax",
           "fa_forward_backward_host", "fa_selftest_wait_timeout", "fa_status_string",
           "fa_last_cuda_error", "fa_device_error")



class FaLibraryMissing(RuntimeError):
    pass


class FaError(RuntimeError):
    def __init__(self, status: int, what: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        name = status_string(status) if _LIB is not None else str(status)
        extra = f" (cudaError {cuda_error})" if status == FA_ERR_CUDA else ""
        super().__init__(f"{what} failed: {name}{extra}")


_LIB = None
_LOCK = threading.Lock()


def library(path: str | None = None):
    """Load libfa.so once and declare the C signatures."""
    global _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise FaLibraryMissing(
                f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_forward.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P]
        lib.fa_forward.restype = I
        lib.fa_forward_ex.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, P]
        lib.fa_forward_ex.restype = I
        lib.fa_forward_splitkv_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.fa_forward_splitkv_workspace_bytes.restype = Z
        lib.fa_forward_splitkv.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, I, F, I, P, P]
        lib.fa_forward_splitkv.restype = I
        lib.fa_forward_choose_splits.argtypes = [I, I, I, I, I, I]
        lib.fa_forward_choose_splits.restype = I
        lib.fa_backward_workspace_bytes.argtypes = [I, I, I, I]
        lib.fa_backward_workspace_bytes.restype = Z
        lib.fa_backward.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, P]
        lib.fa_backward.restype = I
        lib.fa_backward_ex.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, P, P]
        lib.fa_backward_ex.restype = I
        lib.fa_backward_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, P]
        lib.fa_backward_noalloc.restype = I
        lib.fa_naive_softmax.argtypes = [P, P, P, ctypes.c_longlong, I, I, F, P]
        lib.fa_naive_softmax.restype = I
        lib.fa_noalloc_scratch_bytes.argtypes = []
        lib.fa_noalloc_scratch_bytes.restype = Z
        lib.fa_forward_backward_host_device_bytes.argtypes = [I, I, I, I, I, I, I]
        lib.fa_forward_backward_host_device_bytes.restype = Z
        lib.fa_forward_backward_host.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I,
                                                 I, F, I, P, P]
        lib.fa_forward_backward_host.restype = I
        lib.fa_selftest_wait_timeout.argtypes = [ctypes.c_uint, P]
        lib.fa_selftest_wait_timeout.restype = I
        lib.fa_status_string.argtypes = [I]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_last_cuda_error.argtypes = []
        lib.fa_last_cuda_error.restype = I
        lib.fa_device_error.argtypes = [P, ctypes.POINTER(I)]
        lib.fa_device_error.restype = I
        _LIB = lib
        return lib


def status_string(status: int) -> str:
    return library().fa_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != FA_OK:
        lib = library()
        raise FaError(status, what, lib.fa_last_cuda_error() if status == FA_ERR_CUDA else 0)


# ---- raw entry points (plain integers as pointers; used by tests and the bench) ----------

def forward_raw(q: int, k: int, v: int, o: int, lse: int, B: int, H: int, N: int, d: int,
                causal: int, scale: float, stream: int) -> int:
    return library().fa_forward(q, k, v, o, lse, B, H, N, d, causal, scale, stream)


def forward_ex_raw(q: int, k: int, v: int, o: int, lse: int, B: int, Hq: int, Hkv: int, Tq: int,
                   Tk: int, d: int, causal: int, window: int, scale: float, stream: int) -> int:
    """fa_forward_ex: grouped KV heads, query offset Tk - Tq, optional sliding window."""
    return library().fa_forward_ex(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, window, scale,
                                   stream)


def forward_splitkv_raw(q: int, k: int, v: int, o: int, lse: int, B: int, Hq: int, Hkv: int,
                        Tq: int, Tk: int, d: int, causal: int, window: int, scale: float,
                        nsplit: int, workspace: int, stream: int) -> int:
    """fa_forward_splitkv: the key range of every query block cut into `nsplit` chunks."""
    return library().fa_forward_splitkv(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, causal, window,
                                        scale, nsplit, workspace, stream)


def splitkv_workspace_bytes(B: int, Hq: int, Tq: int, d: int, nsplit: int) -> int:
    return int(library().fa_forward_splitkv_workspace_bytes(B, Hq, Tq, d, nsplit))


def backward_ex_raw(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d, causal, window,
                    scale, workspace, stream) -> int:
    return library().fa_backward_ex(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d,
                                    causal, window, scale, workspace, stream)


def backward_raw(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale, workspace,
                 stream) -> int:
    return library().fa_backward(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale,
                                 workspace, stream)


def backward_noalloc_raw(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale,
                         stream) -> int:
    """fa_backward_noalloc: the backward with the library's own fixed device workspace, for
    callers that may not allocate device memory at call time (see include/fa.h)."""
    return library().fa_backward_noalloc(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal,
                                         scale, stream)


def noalloc_scratch_bytes() -> int:
    """Size of the library's own backward workspace (FA_NOALLOC_SCRATCH_BYTES), read from
    libfa.so so that callers never carry a second copy of the constant."""
    return int(library().fa_noalloc_scratch_bytes())


def backward_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(library().fa_backward_workspace_bytes(B, H, N, d))


MAX_HOST_CHUNKS = 16  # FA_MAX_HOST_CHUNKS in include/fa.h


def host_step_device_bytes(B: int, Hq: int, Hkv: int, Tq: int, Tk: int, d: int,
                           nchunks: int = 0) -> int:
    return int(library().fa_forward_backward_host_device_bytes(B, Hq, Hkv, Tq, Tk, d, nchunks))


def forward_backward_host_raw(q, k, v, dout, o, lse, dq, dk, dv, B, Hq, Hkv, Tq, Tk, d, causal,
                              window, scale, nchunks, device_buffer, stream) -> int:
    """fa_forward_backward_host: one forward + backward step on host buffers."""
    return library().fa_forward_backward_host(q, k, v, dout, o, lse, dq, dk, dv, B, Hq, Hkv, Tq,
                                              Tk, d, causal, window, scale, nchunks,
                                              device_buffer, stream)


def selftest_wait_timeout(limit_us: int, stream: int | None = None) -> None:
    """Launch the failure-path diagnostic (a bounded wait that runs out; see include/fa.h)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    _check(library().fa_selftest_wait_timeout(int(limit_us), stream), "fa_selftest_wait_timeout")


def device_error(stream: int | None = None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error word."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    code = ctypes.c_int(0)
    st = library().fa_device_error(stream, ctypes.byref(code))
    if st not in (FA_OK, FA_ERR_TIMEOUT):
        _check(st, "fa_device_error")
    return code.value


# ---- torch-facing wrappers ----------------------------------------------------------------

def _check_tensor(name, t, shape=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _shapes(q, k, v):
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t)
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D")
    B, Hq, Tq, d = q.shape
    _, Hkv, Tk, _ = k.shape
    if tuple(k.shape) != (B, Hkv, Tk, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k, v must both be [B, Hkv, Tk, d] = {(B, Hkv, Tk, d)}")
    return B, Hq, Hkv, Tq, Tk, d


MAX_SPLITS = 64  # FA_MAX_SPLITS in include/fa.h


def choose_splits(B: int, Hq: int, Hkv: int, Tq: int, Tk: int, num_sms: int) -> int:
    """Key-range splits for the forward: the library's cost model (fa_forward_choose_splits)."""
    return int(library().fa_forward_choose_splits(B, Hq, Hkv, Tq, Tk, num_sms))


def forward(q, k, v, causal: bool = False, scale: float | None = None, window: int = -1,
            out=None, lse=None, nsplit: int | None = None, workspace=None, stream=None):
    """O, LSE = attention(q, k, v).

    q is bf16 [B, Hq, Tq, d]; k and v are bf16 [B, Hkv, Tk, d] with Hq % Hkv == 0. Query row i
    sits at key position Tk - Tq + i; ``window`` >= 0 (causal only) keeps keys no more than
    ``window`` positions before it. Multi-head attention is Hkv = Hq, Tq = Tk.
    ``nsplit``: key-range splits (flash-decoding); None picks them from the shape
    (``choose_splits``), 1 disables them.
    """
    import torch
    B, Hq, Hkv, Tq, Tk, d = _shapes(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
    _check_tensor("out", out, q.shape)
    _check_tensor("lse", lse, (B, Hq, Tq))
    if nsplit is None:
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        nsplit = choose_splits(B, Hq, Hkv, Tq, Tk, sms)
    ws_ptr = 0
    if nsplit > 1:
        need = splitkv_workspace_bytes(B, Hq, Tq, d, nsplit)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if workspace is not None:
            if workspace.numel() * workspace.element_size() < need:
                raise ValueError(f"workspace needs {need} bytes")
            ws_ptr = workspace.data_ptr()
    s = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = forward_splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 lse.data_ptr(), B, Hq, Hkv, Tq, Tk, d, int(bool(causal)),
                                 int(window), float(scale), int(nsplit), ws_ptr, s)
    _check(st, "fa_forward_splitkv")
    return out, lse


def backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
             window: int = -1, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of sum(O * dO) given the forward's O and LSE (shapes as ``forward``)."""
    import torch
    B, Hq, Hkv, Tq, Tk, d = _shapes(q, k, v)
    for name, t in (("o", o), ("dout", dout)):
        _check_tensor(name, t, q.shape)
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
    _check_tensor("lse", lse, (B, Hq, Tq))
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensor("dq", dq, q.shape)
    _check_tensor("dk", dk, k.shape)
    _check_tensor("dv", dv, v.shape)
    need = backward_workspace_bytes(B, Hq, Tq, d)
    if workspace is None and need > 0:
        # torch's caching allocator keeps the block between calls (a stream-ordered
        # allocation inside the library would be returned to the driver at every sync)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = 0
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < need:
            raise ValueError(f"workspace needs {need} bytes")
        ws_ptr = workspace.data_ptr()
    s = stream if stream is not None else torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = backward_ex_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                             dv.data_ptr(), B, Hq, Hkv, Tq, Tk, d, int(bool(causal)), int(window),
                             float(scale), ws_ptr, s)
    _check(st, "fa_backward_ex")
    return dq, dk, dv


def _check_host(name, t, shape=None, dtype=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")


def forward_backward_host(q, k, v, dout, causal: bool = False, scale: float | None = None,
                          window: int = -1, nchunks: int = 0, out=None, device_buffer=None,
                          device=None, stream=None):
    """One forward + backward step on host tensors (pinned for overlap): returns host
    (O, LSE, dQ, dK, dV). Shapes as ``forward``; ``out`` = optional tuple of the five output
    tensors; ``device_buffer`` = optional uint8 CUDA tensor of ``host_step_device_bytes`` bytes.
    The call is asynchronous on ``stream`` (synchronise before reading the outputs)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        _check_host(name, t, dtype=torch.bfloat16)
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D")
    B, Hq, Tq, d = q.shape
    _, Hkv, Tk, _ = k.shape
    if tuple(k.shape) != (B, Hkv, Tk, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k, v must both be [B, Hkv, Tk, d] = {(B, Hkv, Tk, d)}")
    _check_host("dout", dout, q.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        pin = q.is_pinned()
        def alloc(shape, dt):
            return torch.empty(shape, dtype=dt, pin_memory=pin)
        out = (alloc(q.shape, torch.bfloat16), alloc((B, Hq, Tq), torch.float32),
               alloc(q.shape, torch.bfloat16), alloc(k.shape, torch.bfloat16),
               alloc(k.shape, torch.bfloat16))
    o, lse, dq, dk, dv = out
    _check_host("o", o, q.shape, torch.bfloat16)
    _check_host("lse", lse, (B, Hq, Tq), torch.float32)
    _check_host("dq", dq, q.shape, torch.bfloat16)
    _check_host("dk", dk, k.shape, torch.bfloat16)
    _check_host("dv", dv, k.shape, torch.bfloat16)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    need = host_step_device_bytes(B, Hq, Hkv, Tq, Tk, d, nchunks)
    if device_buffer is None and need > 0:
        device_buffer = torch.empty(need, dtype=torch.uint8, device=dev)
    buf_ptr = 0
    if device_buffer is not None:
        _check_tensor("device_buffer", device_buffer)
        if device_buffer.numel() * device_buffer.element_size() < need:
            raise ValueError(f"device_buffer needs {need} bytes")
        buf_ptr = device_buffer.data_ptr()
    s = stream if stream is not None else torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.device(dev):
        st = forward_backward_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr(),
                                       o.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                       dv.data_ptr(), B, Hq, Hkv, Tq, Tk, d, int(bool(causal)),
                                       int(window), float(scale), int(nchunks), buf_ptr, s)
    _check(st, "fa_forward_backward_host")
    return o, lse, dq, dk, dv


# ---- autograd -----------------------------------------------------------------------------

def _autograd_function():
    import torch

    class _FlashAttention(torch.autograd.Function):
        """Forward saves (q, k, v, o, lse); backward recomputes through fa_backward_ex."""

        @staticmethod
        def forward(ctx, q, k, v, causal, scale, window):
            o, lse = forward(q, k, v, causal=causal, scale=scale, window=window)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.causal, ctx.scale, ctx.window = causal, scale, window
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o, lse = ctx.saved_tensors
            dq, dk, dv = backward(q, k, v, o, lse, do.contiguous(), causal=ctx.causal,
                                  scale=ctx.scale, window=ctx.window)
            return dq, dk, dv, None, None, None

    return _FlashAttention


_FN = None


def attention(q, k, v, causal: bool = False, scale: float | None = None, window: int = -1):
    """Differentiable O = attention(q, k, v) (shapes as ``forward``); gradients through the
    recompute backward."""
    global _FN
    if _FN is None:
        _FN = _autograd_function()
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _FN.apply(q, k, v, bool(causal), float(scale), int(window))
