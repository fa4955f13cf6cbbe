"""Python binding of the GB300 tiled exact attention library (include/fa.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libfa_gb300.so``.  There is no CPU or PyTorch fallback -- if the
library cannot be loaded, every entry point raises.

Entry points mirror the C ABI:
    fa_forward(Q, K, V, causal, scale=None, window=0)            -> (O, L)
    fa_backward(Q, K, V, O, dO, L, causal, scale=None, window=0)  -> (dQ, dK, dV)
    fa_backward_workspace_bytes(...), fa_backward_workspace_min_bytes(...), fa_status_string(code),
    fa_last_device_status()
plus ``FlashAttention`` (a torch.autograd.Function that keeps only Q, K, V, O
and L for the backward pass) and ``attention`` (its functional form).

Tensors are CUDA bf16, contiguous, [B, H, T, d]; L is fp32 [B, Hq, Tq].
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)

EXPORTED_SYMBOLS = ("fa_forward", "fa_backward", "fa_backward_stages", "fa_backward_workspace_bytes",
                    "fa_backward_workspace_min_bytes", "fa_backward_noalloc", "fa_status_string",
                    "fa_last_device_status", "fa_last_launch_count")
FA_ERR_SCRATCH_TOO_SMALL = 5
FA_NOALLOC_SCRATCH_BYTES = 32 << 20
FA_BWD_PRE, FA_BWD_MAIN, FA_BWD_CAST, FA_BWD_ALL = 1, 2, 4, 7


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


class FaDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("Tq", ctypes.c_int),
                ("Tk", ctypes.c_int), ("d", ctypes.c_int), ("dv", ctypes.c_int), ("causal", ctypes.c_int),
                ("scale", ctypes.c_float), ("window", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load (building first if needed) the shared library; raises if that fails."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.build()
            if not os.path.exists(p):
                raise RuntimeError(f"CUDA attention library missing: {p}")
            lib = ctypes.CDLL(p)
            vp, dp = ctypes.c_void_p, ctypes.POINTER(FaDims)
            lib.fa_forward.argtypes = [dp, vp, vp, vp, vp, vp, vp]
            lib.fa_forward.restype = ctypes.c_int
            lib.fa_backward.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
            lib.fa_backward.restype = ctypes.c_int
            lib.fa_backward_stages.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t,
                                               ctypes.c_int, vp]
            lib.fa_backward_stages.restype = ctypes.c_int
            lib.fa_backward_noalloc.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.fa_backward_noalloc.restype = ctypes.c_int
            lib.fa_backward_workspace_bytes.argtypes = [dp]
            lib.fa_backward_workspace_bytes.restype = ctypes.c_size_t
            lib.fa_backward_workspace_min_bytes.argtypes = [dp]
            lib.fa_backward_workspace_min_bytes.restype = ctypes.c_size_t
            lib.fa_status_string.argtypes = [ctypes.c_int]
            lib.fa_status_string.restype = ctypes.c_char_p
            lib.fa_last_device_status.argtypes = [vp]
            lib.fa_last_device_status.restype = ctypes.c_int
            lib.fa_last_launch_count.argtypes = []
            lib.fa_last_launch_count.restype = ctypes.c_int
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().fa_status_string(int(code)).decode()


fa_status_string = status_string


def make_dims(B, Hq, Hkv, Tq, Tk, d, dv, causal, scale, window: int = 0) -> FaDims:
    return FaDims(int(B), int(Hq), int(Hkv), int(Tq), int(Tk), int(d), int(dv), int(bool(causal)),
                  float(scale) if scale is not None else 0.0, int(window))


def _dims_of(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, causal, scale, window: int = 0) -> FaDims:
    if Q.dim() != 4 or K.dim() != 4 or V.dim() != 4:
        raise ValueError("Q, K, V must be [B, H, T, d]")
    B, Hq, Tq, d = Q.shape
    Bk, Hkv, Tk, dk = K.shape
    Bv, Hv, Tv, dv = V.shape
    if not (B == Bk == Bv and Hkv == Hv and Tk == Tv and d == dk):
        raise ValueError(f"inconsistent shapes Q{tuple(Q.shape)} K{tuple(K.shape)} V{tuple(V.shape)}")
    return make_dims(B, Hq, Hkv, Tq, Tk, d, dv, causal, scale, window)


def _check(t: torch.Tensor, name: str, dtype=torch.bfloat16):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def _check_all(device, specs):
    """The library sees only pointers, so every size it relies on is checked
    here: each (tensor, name, shape, dtype) must have exactly that shape, be a
    contiguous CUDA tensor of that dtype and live on ``device``.  Shapes are
    checked first so a mismatch is reported as such on any device."""
    for t, name, shape, _ in specs:
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    for t, name, _, dtype in specs:
        _check(t, name, dtype)
        if t.device != device:
            raise ValueError(f"{name} is on {t.device}, expected {device} (all tensors on one GPU)")


def _stream_ptr(stream=None, device=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    if device is not None and s.device != device:
        raise ValueError(f"stream belongs to {s.device}, the tensors to {device}")
    return s.cuda_stream


def _raise(code: int, where: str):
    if code != FA_OK:
        raise FAError(code, where)


def fa_backward_workspace_bytes(dims: FaDims) -> int:
    """Workspace for the backward's fastest schedule (what fa_backward allocates)."""
    return int(load().fa_backward_workspace_bytes(ctypes.byref(dims)))


def fa_backward_workspace_min_bytes(dims: FaDims) -> int:
    """The least workspace fa_backward accepts (then no work item is split)."""
    return int(load().fa_backward_workspace_min_bytes(ctypes.byref(dims)))


def fa_forward(Q, K, V, causal: bool, scale: float | None = None, O=None, L=None, stream=None, window: int = 0):
    """O, L = attention forward.  Optional preallocated O / L are written in place.
    ``window=W`` (causal only) lets each row see at most its last W keys."""
    dims = _dims_of(Q, K, V, causal, scale, window)
    bf, f32 = torch.bfloat16, torch.float32
    specs = [(Q, "Q", Q.shape, bf), (K, "K", K.shape, bf), (V, "V", V.shape, bf)]
    if O is not None:
        specs.append((O, "O", (dims.B, dims.Hq, dims.Tq, dims.dv), bf))
    if L is not None:
        specs.append((L, "L", (dims.B, dims.Hq, dims.Tq), f32))
    _check_all(Q.device, specs)
    if O is None:
        O = torch.empty(dims.B, dims.Hq, dims.Tq, dims.dv, dtype=bf, device=Q.device)
    if L is None:
        L = torch.empty(dims.B, dims.Hq, dims.Tq, dtype=f32, device=Q.device)
    lib = load()
    with torch.cuda.device(Q.device):
        code = lib.fa_forward(ctypes.byref(dims), Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                              L.data_ptr(), _stream_ptr(stream, Q.device))
    _raise(code, "fa_forward")
    return O, L


def fa_backward(Q, K, V, O, dO, L, causal: bool, scale: float | None = None, dQ=None, dK=None, dV=None,
                workspace=None, stream=None, stages: int = FA_BWD_ALL, window: int = 0):
    """dQ, dK, dV = attention backward from the saved O and L.

    ``stages`` selects which of the three backward kernels to launch (see
    fa_backward_stages in include/fa.h); the default runs all of them.
    """
    dims, dQ, dK, dV = _backward_operands(Q, K, V, O, dO, L, causal, scale, window, dQ, dK, dV)
    lib = load()
    need = fa_backward_workspace_bytes(dims)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=Q.device)
    elif not workspace.is_cuda or workspace.device != Q.device or not workspace.is_contiguous():
        raise ValueError(f"workspace must be a contiguous CUDA tensor on {Q.device}")
    nbytes = workspace.numel() * workspace.element_size()
    args = (ctypes.byref(dims), Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), dO.data_ptr(),
            L.data_ptr(), dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), workspace.data_ptr(), nbytes)
    with torch.cuda.device(Q.device):
        if stages == FA_BWD_ALL:
            code = lib.fa_backward(*args, _stream_ptr(stream, Q.device))
        else:
            code = lib.fa_backward_stages(*args, int(stages), _stream_ptr(stream, Q.device))
    _raise(code, "fa_backward")
    return dQ, dK, dV


def _backward_operands(Q, K, V, O, dO, L, causal, scale, window, dQ, dK, dV):
    """Dims of a backward call, its gradient buffers (allocated when not given)
    and the shape / dtype / device checks of all eleven tensors."""
    dims = _dims_of(Q, K, V, causal, scale, window)
    bf, f32 = torch.bfloat16, torch.float32
    qv, rows = (dims.B, dims.Hq, dims.Tq, dims.dv), (dims.B, dims.Hq, dims.Tq)
    specs = [(Q, "Q", Q.shape, bf), (K, "K", K.shape, bf), (V, "V", V.shape, bf),
             (O, "O", qv, bf), (dO, "dO", qv, bf), (L, "L", rows, f32)]
    specs += [(t, n, like.shape, bf) for t, n, like in ((dQ, "dQ", Q), (dK, "dK", K), (dV, "dV", V))
              if t is not None]
    _check_all(Q.device, specs)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    return dims, dQ, dK, dV


def fa_backward_noalloc(Q, K, V, O, dO, L, causal: bool, scale: float | None = None, dQ=None, dK=None, dV=None,
                        stream=None, window: int = 0):
    """fa_backward without a workspace, for callers that cannot allocate device
    memory: the library's fixed scratch array (FA_NOALLOC_SCRATCH_BYTES per
    GPU) is used instead.  Pass preallocated dQ / dK / dV to allocate nothing
    at all; calls that could overlap on the GPU must be ordered by the caller."""
    dims, dQ, dK, dV = _backward_operands(Q, K, V, O, dO, L, causal, scale, window, dQ, dK, dV)
    lib = load()
    with torch.cuda.device(Q.device):
        code = lib.fa_backward_noalloc(ctypes.byref(dims), Q.data_ptr(), K.data_ptr(), V.data_ptr(),
                                       O.data_ptr(), dO.data_ptr(), L.data_ptr(), dQ.data_ptr(), dK.data_ptr(),
                                       dV.data_ptr(), _stream_ptr(stream, Q.device))
    _raise(code, "fa_backward_noalloc")
    return dQ, dK, dV


def fa_last_device_status(stream=None) -> int:
    return int(load().fa_last_device_status(_stream_ptr(stream)))


def last_launch_count() -> int:
    return int(load().fa_last_launch_count())


class FlashAttention(torch.autograd.Function):
    """Autograd wrapper: saves Q, K, V (inputs) plus O and L -- nothing quadratic."""

    @staticmethod
    def forward(ctx, Q, K, V, causal=False, scale=None, window=0):
        O, L = fa_forward(Q, K, V, causal, scale, window=window)
        ctx.save_for_backward(Q, K, V, O, L)
        ctx.causal, ctx.scale, ctx.window = causal, scale, window
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, L = ctx.saved_tensors
        dQ, dK, dV = fa_backward(Q, K, V, O, dO.contiguous(), L, ctx.causal, ctx.scale, window=ctx.window)
        return dQ, dK, dV, None, None, None


def attention(Q, K, V, causal=False, scale=None, window=0):
    return FlashAttention.apply(Q, K, V, causal, scale, window)
