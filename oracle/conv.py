"""fp64 CPU oracle for the 2-D convolution derivatives (ctypes binding of
conv_oracle.c).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The CUDA product path never touches it.

What the functions compute is written out at the top of ``conv_oracle.c``:
the input and weight gradients of a channels-last 2-D convolution
(cross-correlation, zero padding, one stride and one padding for both spatial
axes), the derivative nodes behind the convolution-derivative kernels of
"Meganeura: Portable GPU Training and Inference through Vulkan and Metal"
(Sections 3.1 and 7.3).

Parity pins (``tests/test_conv_oracle_pins.py``, no GPU): central finite
differences of sum(G * Y) for both gradients, the adjoint identity between the
forward and both gradients, 1x1 convolutions as numpy matrix products, torch's
float64 conv2d and its input/weight gradients, the sampled (gather) forms
against the full (scatter) forms, and a hand-derived integer example
(``tests/golden/conv_tiny.json``)."""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_LIB = os.path.join(_HERE, "libconv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile conv_oracle.c into libconv_oracle.so next to it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lp = ctypes.POINTER(ctypes.c_long)
            L, I = ctypes.c_long, ctypes.c_int
            dims = [L] * 9 + [I]
            for name in ("conv_oracle_fwd", "conv_oracle_grad_input", "conv_oracle_grad_weight"):
                f = getattr(lib, name)
                f.argtypes = [dp, dp, dp] + dims
                f.restype = I
            for name in ("conv_oracle_grad_input_at", "conv_oracle_grad_weight_at"):
                f = getattr(lib, name)
                f.argtypes = [dp, dp, lp, L, dp] + dims
                f.restype = I
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def out_size(H: int, W: int, R: int, S: int, stride: int, pad: int):
    """(P, Q): output rows and columns of the convolution."""
    return (H + 2 * pad - R) // stride + 1, (W + 2 * pad - S) // stride + 1


def _dims(X_shape, Wt_shape):
    N, H, W, C = X_shape
    K, R, S, C2 = Wt_shape
    if C2 != C:
        raise ValueError("X [N,H,W,C] and Wt [K,R,S,C] must share C")
    return N, H, W, C, K, R, S


def conv2d_fwd(X, Wt, stride: int, pad: int, nthreads: int = 0) -> np.ndarray:
    """Y [N,P,Q,K] for X [N,H,W,C] and Wt [K,R,S,C]."""
    X, Wt = _f64(X), _f64(Wt)
    N, H, W, C, K, R, S = _dims(X.shape, Wt.shape)
    P, Q = out_size(H, W, R, S, stride, pad)
    Y = np.empty((N, P, Q, K))
    rc = _load().conv_oracle_fwd(_ptr(X), _ptr(Wt), _ptr(Y), N, H, W, C, K, R, S, stride, pad,
                                 nthreads)
    if rc:
        raise RuntimeError(f"conv_oracle_fwd failed ({rc})")
    return Y


def conv2d_grad_input(dY, Wt, H: int, W: int, stride: int, pad: int,
                      nthreads: int = 0) -> np.ndarray:
    """dX [N,H,W,C] for dY [N,P,Q,K] and Wt [K,R,S,C]."""
    dY, Wt = _f64(dY), _f64(Wt)
    N, P, Q, K = dY.shape
    K2, R, S, C = Wt.shape
    if K2 != K or out_size(H, W, R, S, stride, pad) != (P, Q):
        raise ValueError("dY does not match the convolution's output shape")
    dX = np.empty((N, H, W, C))
    rc = _load().conv_oracle_grad_input(_ptr(dY), _ptr(Wt), _ptr(dX), N, H, W, C, K, R, S,
                                        stride, pad, nthreads)
    if rc:
        raise RuntimeError(f"conv_oracle_grad_input failed ({rc})")
    return dX


def conv2d_grad_weight(X, dY, R: int, S: int, stride: int, pad: int,
                       nthreads: int = 0) -> np.ndarray:
    """dW [K,R,S,C] for X [N,H,W,C] and dY [N,P,Q,K]."""
    X, dY = _f64(X), _f64(dY)
    N, H, W, C = X.shape
    K = dY.shape[3]
    if dY.shape[:3] != (N,) + out_size(H, W, R, S, stride, pad):
        raise ValueError("dY does not match the convolution's output shape")
    dW = np.empty((K, R, S, C))
    rc = _load().conv_oracle_grad_weight(_ptr(X), _ptr(dY), _ptr(dW), N, H, W, C, K, R, S,
                                         stride, pad, nthreads)
    if rc:
        raise RuntimeError(f"conv_oracle_grad_weight failed ({rc})")
    return dW


def _idx(points) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(points, dtype=np.int64).reshape(-1, 4))
    return a


def conv2d_grad_input_at(dY, Wt, H: int, W: int, stride: int, pad: int, points,
                         nthreads: int = 0) -> np.ndarray:
    """dX at the (n, h, w, c) points (an [n_points, 4] integer array)."""
    dY, Wt = _f64(dY), _f64(Wt)
    N, P, Q, K = dY.shape
    _, R, S, C = Wt.shape
    idx = _idx(points)
    out = np.empty(len(idx))
    rc = _load().conv_oracle_grad_input_at(
        _ptr(dY), _ptr(Wt), idx.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), len(idx),
        _ptr(out), N, H, W, C, K, R, S, stride, pad, nthreads)
    if rc:
        raise RuntimeError(f"conv_oracle_grad_input_at failed ({rc})")
    return out


def conv2d_grad_weight_at(X, dY, R: int, S: int, stride: int, pad: int, points,
                          nthreads: int = 0) -> np.ndarray:
    """dW at the (k, r, s, c) points (an [n_points, 4] integer array)."""
    X, dY = _f64(X), _f64(dY)
    N, H, W, C = X.shape
    K = dY.shape[3]
    idx = _idx(points)
    out = np.empty(len(idx))
    rc = _load().conv_oracle_grad_weight_at(
        _ptr(X), _ptr(dY), idx.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), len(idx),
        _ptr(out), N, H, W, C, K, R, S, stride, pad, nthreads)
    if rc:
        raise RuntimeError(f"conv_oracle_grad_weight_at failed ({rc})")
    return out
