"""fp64 CPU oracle for attention forward + backward (ctypes binding of mg_oracle.c).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The CUDA product path never touches it.

What the functions compute is the definition written out at the top of
``mg_oracle.c`` (scaled dot-product attention and its chain-rule gradients, the
attention node of "Meganeura: Portable GPU Training and Inference through Vulkan
and Metal", Sections 3.1 and 3.3). Every input is converted to float64 exactly
(f32 and bf16 values are representable in f64) before the call.

Parity pins (checked by ``tests/test_oracle_pins.py`` without a GPU):
central finite differences of sum(dO*O) for dQ, dK, dV; softmax rows summing to
one; the causal first row; dV with dO = 1 giving the column sums of P; the
softmax-Jacobian invariant sum_j dK_j = 0; L = 1 and equal-key closed forms; the
key-shift metamorphic relation; torch float64 SDPA + autograd on tiny shapes.
For cross attention (Lq != Lk) and the two causal alignments: central finite
differences for every alignment, the alignments coinciding when Lq = Lk, a
single bottom-right query seeing every key, empty-softmax rows contributing
nothing, torch float64 SDPA with explicit boolean masks + autograd, and three
hand-derived worked examples with exact rationals (``tests/test_golden.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mg_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile mg_oracle.c into liboracle.so next to it (gcc, OpenMP)."""
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
            L, I, D = ctypes.c_long, ctypes.c_int, ctypes.c_double
            lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, L, L, I, I, D, I]
            lib.oracle_attn_fwd.restype = I
            lib.oracle_attn_fwd_rows.argtypes = [dp, dp, dp, lp, L, dp, dp, L, I, I, D, I]
            lib.oracle_attn_fwd_rows.restype = I
            lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                            L, L, I, I, D, I]
            lib.oracle_attn_bwd.restype = I
            lib.oracle_attn_fwd_ex.argtypes = [dp, dp, dp, dp, dp, L, L, L, I, I, D, I]
            lib.oracle_attn_fwd_ex.restype = I
            lib.oracle_attn_bwd_ex.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                               L, L, L, I, I, D, I]
            lib.oracle_attn_bwd_ex.restype = I
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = I
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shape(Q):
    if Q.ndim < 2:
        raise ValueError("expected [..., L, D]")
    L, D = Q.shape[-2], Q.shape[-1]
    BH = int(np.prod(Q.shape[:-2])) if Q.ndim > 2 else 1
    return BH, L, D


MASKS = {"none": 0, "causal": 1, "causal_bottom_right": 2}


def _mask_id(mask) -> int:
    if isinstance(mask, str):
        return MASKS[mask]
    if int(mask) not in MASKS.values():
        raise ValueError(f"unknown mask {mask}")
    return int(mask)


def _shape_ex(Q, K):
    if Q.ndim < 2 or K.ndim != Q.ndim or Q.shape[:-2] != K.shape[:-2] or Q.shape[-1] != K.shape[-1]:
        raise ValueError("expected Q [..., Lq, D] and K, V [..., Lk, D] with the same leading dims")
    BH = int(np.prod(Q.shape[:-2])) if Q.ndim > 2 else 1
    return BH, Q.shape[-2], K.shape[-2], Q.shape[-1]


def attn_fwd_ex(Q, K, V, mask, scale: float, nthreads: int = 0):
    """(O, LSE) in float64 for Q [..., Lq, D] and K, V [..., Lk, D]. ``mask``:
    "none", "causal" (top-left, j <= i) or "causal_bottom_right" (j <= i + Lk - Lq).
    Rows with no allowed key get O = 0 and LSE = -inf."""
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    if K.shape != V.shape:
        raise ValueError("K and V must share one shape")
    BH, Lq, Lk, D = _shape_ex(Q, K)
    O = np.empty_like(Q)
    LSE = np.empty(Q.shape[:-1], dtype=np.float64)
    rc = lib.oracle_attn_fwd_ex(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), BH, Lq, Lk, D,
                                _mask_id(mask), float(scale), int(nthreads))
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_ex failed ({rc})")
    return O, LSE


def attn_bwd_ex(Q, K, V, dO, mask, scale: float, nthreads: int = 0) -> dict:
    """Forward and backward in float64 for Q, dO [..., Lq, D] and K, V [..., Lk, D]:
    O, LSE, Dvec, dQ, dK, dV (see ``attn_fwd_ex`` for ``mask``)."""
    lib = _load()
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    if K.shape != V.shape or Q.shape != dO.shape:
        raise ValueError("K, V and Q, dO must share shapes")
    BH, Lq, Lk, D = _shape_ex(Q, K)
    out = {"O": np.empty_like(Q), "LSE": np.empty(Q.shape[:-1]), "Dvec": np.empty(Q.shape[:-1]),
           "dQ": np.empty_like(Q), "dK": np.empty_like(K), "dV": np.empty_like(K)}
    rc = lib.oracle_attn_bwd_ex(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(out["O"]),
                                _ptr(out["LSE"]), _ptr(out["Dvec"]), _ptr(out["dQ"]),
                                _ptr(out["dK"]), _ptr(out["dV"]), BH, Lq, Lk, D,
                                _mask_id(mask), float(scale), int(nthreads))
    if rc:
        raise RuntimeError(f"oracle_attn_bwd_ex failed ({rc})")
    return out


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def attn_fwd(Q, K, V, causal: bool, scale: float, nthreads: int = 0):
    """Return (O, LSE) in float64 for inputs shaped [..., L, D]."""
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    if not (Q.shape == K.shape == V.shape):
        raise ValueError("Q, K, V must share one shape")
    BH, L, D = _shape(Q)
    O = np.empty_like(Q)
    LSE = np.empty(Q.shape[:-1], dtype=np.float64)
    rc = lib.oracle_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                             BH, L, D, int(bool(causal)), float(scale), int(nthreads))
    if rc:
        raise RuntimeError(f"oracle_attn_fwd failed ({rc})")
    return O, LSE


def attn_fwd_rows(Q, K, V, rows, causal: bool, scale: float, nthreads: int = 0):
    """Forward for the query rows ``rows`` of ONE head ([L, D] inputs)."""
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    if Q.ndim != 2:
        raise ValueError("attn_fwd_rows takes one head: [L, D]")
    L, D = Q.shape
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    O = np.empty((r.size, D), dtype=np.float64)
    LSE = np.empty(r.size, dtype=np.float64)
    rc = lib.oracle_attn_fwd_rows(_ptr(Q), _ptr(K), _ptr(V),
                                  r.ctypes.data_as(ctypes.POINTER(ctypes.c_long)),
                                  r.size, _ptr(O), _ptr(LSE), L, D,
                                  int(bool(causal)), float(scale), int(nthreads))
    if rc:
        raise RuntimeError(f"oracle_attn_fwd_rows failed ({rc})")
    return O, LSE


def attn_bwd(Q, K, V, dO, causal: bool, scale: float, nthreads: int = 0):
    """Return dict(O, LSE, Dvec, dQ, dK, dV) in float64 for [..., L, D] inputs."""
    lib = _load()
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    if not (Q.shape == K.shape == V.shape == dO.shape):
        raise ValueError("Q, K, V, dO must share one shape")
    BH, L, D = _shape(Q)
    O = np.empty_like(Q)
    dQ = np.empty_like(Q)
    dK = np.empty_like(Q)
    dV = np.empty_like(Q)
    LSE = np.empty(Q.shape[:-1], dtype=np.float64)
    Dvec = np.empty(Q.shape[:-1], dtype=np.float64)
    rc = lib.oracle_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), _ptr(O), _ptr(LSE),
                             _ptr(Dvec), _ptr(dQ), _ptr(dK), _ptr(dV), BH, L, D,
                             int(bool(causal)), float(scale), int(nthreads))
    if rc:
        raise RuntimeError(f"oracle_attn_bwd failed ({rc})")
    return {"O": O, "LSE": LSE, "Dvec": Dvec, "dQ": dQ, "dK": dK, "dV": dV}


def attn_bwd_padded(Q, K, V, dO, kv_len, mask, scale: float, nthreads: int = 0) -> dict:
    """Per-batch key padding: Q, dO [B, H, Lq, D], K, V [B, H, Lk, D], kv_len B
    integers in [0, Lk]. Batch element b is the cross-attention problem with its
    first kv_len[b] keys only (the rows past it are padding and do not exist:
    ``attn_bwd_ex`` on the truncated K and V, so the bottom-right alignment uses
    kv_len[b] - Lq); the padding rows of dK and dV are 0. With kv_len[b] = 0 no
    key exists: every row of b has an empty softmax (O = 0, LSE = -inf) and all
    of b's gradients are 0. Returns O, LSE, Dvec, dQ, dK, dV in float64."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    if Q.ndim != 4 or K.shape != V.shape or Q.shape != dO.shape or K.shape[:2] != Q.shape[:2]:
        raise ValueError("expected Q, dO [B, H, Lq, D] and K, V [B, H, Lk, D]")
    B, H, Lq, D = Q.shape
    Lk = K.shape[2]
    lens = [int(n) for n in np.asarray(kv_len).reshape(-1)]
    if len(lens) != B or any(n < 0 or n > Lk for n in lens):
        raise ValueError("kv_len must hold B lengths in [0, Lk]")
    out = {"O": np.zeros_like(Q), "LSE": np.full((B, H, Lq), -np.inf),
           "Dvec": np.zeros((B, H, Lq)), "dQ": np.zeros_like(Q), "dK": np.zeros_like(K),
           "dV": np.zeros_like(K)}
    for b, n in enumerate(lens):
        if n == 0:
            continue
        r = attn_bwd_ex(Q[b], K[b, :, :n], V[b, :, :n], dO[b], mask, scale, nthreads)
        for k in ("O", "LSE", "Dvec", "dQ"):
            out[k][b] = r[k]
        out["dK"][b, :, :n] = r["dK"]
        out["dV"][b, :, :n] = r["dV"]
    return out


def attn_fwd_padded(Q, K, V, kv_len, mask, scale: float, nthreads: int = 0):
    """(O, LSE) of ``attn_bwd_padded`` without the backward."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    if Q.ndim != 4 or K.shape != V.shape or K.shape[:2] != Q.shape[:2]:
        raise ValueError("expected Q [B, H, Lq, D] and K, V [B, H, Lk, D]")
    B, H, Lq, D = Q.shape
    Lk = K.shape[2]
    lens = [int(n) for n in np.asarray(kv_len).reshape(-1)]
    if len(lens) != B or any(n < 0 or n > Lk for n in lens):
        raise ValueError("kv_len must hold B lengths in [0, Lk]")
    O = np.zeros_like(Q)
    LSE = np.full((B, H, Lq), -np.inf)
    for b, n in enumerate(lens):
        if n:
            O[b], LSE[b] = attn_fwd_ex(Q[b], K[b, :, :n], V[b, :, :n], mask, scale, nthreads)
    return O, LSE
