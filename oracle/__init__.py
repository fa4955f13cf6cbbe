"""Float64 CPU oracle for tiled exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never calls it and the two share
no code: this side is plain C++ in float64 (``fa_oracle.cpp``) plus this ctypes
wrapper.

What is computed (see the header of ``fa_oracle.cpp`` for the row-by-row
definition and the hand-derived gradients):

* ``forward``  -- O = softmax(scale * Q K^T + mask) V and L = logsumexp of the
  scaled scores ("What Ordinary Autograd Saves", section "The implementation
  under test": `dense_attention` and the `L = mi + log(li)` statistic of the
  tiled forward; "Backward Pass Implementation", `standard_attention`).
* ``backward`` -- dQ, dK, dV (and D) of the loss <O, dO>.
* ``saved_bytes`` -- bytes kept for the backward pass by the dense, the
  checkpointed and the keep-O-and-L strategies ("What Ordinary Autograd
  Saves", sections "The measurement" and "Why this is FlashAttention's second
  idea").

Every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "libfa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle source into a shared library (g++, OpenMP, IEEE double)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _f64(a) -> np.ndarray:
    """Any array-like (numpy, torch CPU tensor of any float dtype) -> contiguous float64 numpy."""
    if hasattr(a, "detach"):  # torch tensor: upcast exactly (bf16/fp32 -> fp64 is exact)
        import torch

        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(Q, K, V):
    B, Hq, Tq, d = Q.shape
    B2, Hkv, Tk, d2 = K.shape
    B3, Hkv3, Tk3, dv = V.shape
    if not (B == B2 == B3 and Hkv == Hkv3 and Tk == Tk3 and d == d2 and Hkv > 0 and Hq % Hkv == 0):
        raise ValueError("inconsistent shapes")
    return B, Hq, Hkv, Tq, Tk, d, dv


def default_scale(d: int) -> float:
    return 1.0 / float(np.sqrt(d))


STRATEGIES = {"dense": 0, "checkpoint": 1, "keep_o_l": 2}


class OracleLib:
    """ctypes view of one build of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        lib.fa_oracle_forward.argtypes = [dp, dp, dp, i, i, i, i, i, i, i, i, i, ctypes.c_double, i, i, dp, dp, i]
        lib.fa_oracle_forward.restype = None
        lib.fa_oracle_backward.argtypes = [dp, dp, dp, dp, i, i, i, i, i, i, i, i, i, ctypes.c_double,
                                           dp, dp, dp, dp, i]
        lib.fa_oracle_backward.restype = None
        lib.fa_oracle_saved_bytes.argtypes = [i] * 11
        lib.fa_oracle_saved_bytes.restype = ctypes.c_int64
        self.lib = lib
        self.path = path

    def forward(self, Q, K, V, causal: bool, scale: float | None = None, rows: tuple[int, int] | None = None,
                nthreads: int = 0, window: int = 0):
        """Return (O, L) as float64 numpy arrays [B,Hq,Tq,dv] / [B,Hq,Tq].

        ``rows=(lo, hi)`` computes only query rows lo..hi-1 of every head (others are NaN).
        ``window=W`` (causal only) limits each row to its last W keys; 0 = no limit.
        """
        Q, K, V = _f64(Q), _f64(K), _f64(V)
        B, Hq, Hkv, Tq, Tk, d, dv = _dims(Q, K, V)
        scale = default_scale(d) if scale is None or scale <= 0 else float(scale)
        lo, hi = rows if rows is not None else (0, Tq)
        O = np.full((B, Hq, Tq, dv), np.nan)
        L = np.full((B, Hq, Tq), np.nan)
        self.lib.fa_oracle_forward(_ptr(Q), _ptr(K), _ptr(V), B, Hq, Hkv, Tq, Tk, d, dv, int(bool(causal)),
                                   int(window), scale, int(lo), int(hi), _ptr(O), _ptr(L), int(nthreads))
        return O, L

    def backward(self, Q, K, V, dO, causal: bool, scale: float | None = None, nthreads: int = 0, window: int = 0):
        """Return (dQ, dK, dV, D) as float64 numpy arrays for the loss <O, dO>."""
        Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
        B, Hq, Hkv, Tq, Tk, d, dv = _dims(Q, K, V)
        if dO.shape != (B, Hq, Tq, dv):
            raise ValueError("dO shape")
        scale = default_scale(d) if scale is None or scale <= 0 else float(scale)
        dQ = np.empty((B, Hq, Tq, d))
        dK = np.empty((B, Hkv, Tk, d))
        dV = np.empty((B, Hkv, Tk, dv))
        D = np.zeros((B, Hq, Tq))
        self.lib.fa_oracle_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, Hq, Hkv, Tq, Tk, d, dv,
                                    int(bool(causal)), int(window), scale, _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(D),
                                    int(nthreads))
        return dQ, dK, dV, D

    def saved_bytes(self, strategy: str, B, Hq, Hkv, Tq, Tk, d, dv, elem_bytes, stat_bytes=4,
                    prob_bytes=None) -> int:
        """Bytes retained for the backward pass by ``strategy`` (dense / checkpoint / keep_o_l)."""
        prob_bytes = elem_bytes if prob_bytes is None else prob_bytes
        return int(self.lib.fa_oracle_saved_bytes(STRATEGIES[strategy], B, Hq, Hkv, Tq, Tk, d, dv, elem_bytes,
                                                  stat_bytes, prob_bytes))


def default() -> OracleLib:
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
    return _lib


def forward(*a, **k):
    return default().forward(*a, **k)


def backward(*a, **k):
    return default().backward(*a, **k)


def saved_bytes(*a, **k):
    return default().saved_bytes(*a, **k)
