"""Python binding of libmgattn.so (ctypes): multi-head scaled-dot-product
attention forward + backward on one GB300 GPU.

Argument marshalling only. Every step of the computation runs in the CUDA
library; there is no Python, PyTorch or CPU fallback. If the library has not
been built, or the CUDA device is missing, the calls raise.

The function names mirror the C ABI in ``include/mg_attn.h``:

* ``mg_attn_fwd(Q, K, V, O, LSE, causal, scale, contract, stream=None)``
* ``mg_attn_bwd_workspace_bytes(B, H, L, D, contract)``
* ``mg_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, causal, scale, contract,
  workspace, stream=None)``
* ``mg_attn_fwd_ex``, ``mg_attn_bwd_workspace_bytes_ex``, ``mg_attn_bwd_ex`` (cross
  attention, Lq != Lk, with a mask)
* ``mg_attn_fwd_padded``, ``mg_attn_bwd_padded`` (per-batch key padding lengths)
* ``mg_attn_fwd_decode_workspace_bytes``, ``mg_attn_fwd_decode`` (split-key
  forward for at most 8 query rows)
* ``mg_conv2d_grad_input(dY, Wt, dX, stride, pad, contract)``,
  ``mg_conv2d_grad_weight(X, dY, dW, stride, pad, contract)`` (derivatives of a
  channels-last 2-D convolution: X [N, H, W, C], Wt [K, R, S, C], dY [N, P, Q, K])
* ``mg_status_string(status)``, ``mg_get_device_error(stream=None)``
* ``mg_attn_profile_enable``, ``mg_attn_profile_read``, ``mg_attn_kernel_name``

Tensors are PyTorch CUDA tensors, contiguous [B, H, L, D] (LSE [B, H, L]); the
shape is read from Q. ``contract`` is ``STRICT_F32`` (0), ``ACCEL_BF16`` (1) or
``ACCEL_F16`` (2), optionally OR-ed with ``OUT_16`` (16-bit outputs) and
``DS_HILO`` (hi/lo split of dS in the backward), or a name such as ``"accel"``,
``"accel_f16+out16"``, ``"accel+hilo"``.
``attention_fwd`` / ``attention_bwd`` are conveniences that allocate the
outputs with PyTorch and call the above.
"""
from __future__ import annotations

import ctypes
import os
import threading

STRICT_F32 = 0
ACCEL_BF16 = 1
ACCEL_F16 = 2
OUT_16 = 0x100  # flag: O, dQ, dK, dV in the inputs' 16-bit type
CONTRACTS = {"strict": STRICT_F32, "accel": ACCEL_BF16, "accel_f16": ACCEL_F16}
DS_HILO = 0x200  # flag: hi/lo split of dS in the backward (derivative precision)
FLAGS = {"out16": OUT_16, "hilo": DS_HILO}

MG_OK, MG_ERR_INVALID_ARG, MG_ERR_UNSUPPORTED, MG_ERR_WORKSPACE, MG_ERR_CUDA, MG_ERR_TIMEOUT = range(6)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmgattn.so")
_lock = threading.Lock()
_lib = None


class MgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {mg_status_string(status)} ({status})")


def load_library(path: str | None = None):
    """Load libmgattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(p)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.mg_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.mg_attn_fwd.restype = i
        lib.mg_attn_bwd_workspace_bytes.argtypes = [i, i, i, i, i]
        lib.mg_attn_bwd_workspace_bytes.restype = sz
        lib.mg_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i,
                                    vp, sz, vp]
        lib.mg_attn_bwd.restype = i
        lib.mg_attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.mg_attn_fwd_ex.restype = i
        lib.mg_attn_bwd_workspace_bytes_ex.argtypes = [i, i, i, i, i, i]
        lib.mg_attn_bwd_workspace_bytes_ex.restype = sz
        lib.mg_attn_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f,
                                       i, vp, sz, vp]
        lib.mg_attn_bwd_ex.restype = i
        lib.mg_attn_fwd_padded.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.mg_attn_fwd_padded.restype = i
        lib.mg_attn_bwd_padded.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i,
                                           i, i, f, i, vp, sz, vp]
        lib.mg_attn_bwd_padded.restype = i
        lib.mg_attn_fwd_decode_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.mg_attn_fwd_decode_workspace_bytes.restype = sz
        lib.mg_attn_fwd_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz,
                                           vp]
        lib.mg_attn_fwd_decode.restype = i
        lib.mg_status_string.argtypes = [i]
        lib.mg_status_string.restype = ctypes.c_char_p
        lib.mg_get_device_error.argtypes = [vp]
        lib.mg_get_device_error.restype = i
        lib.mg_attn_profile_enable.argtypes = [i, i]
        lib.mg_attn_profile_enable.restype = i
        lib.mg_attn_profile_read.argtypes = [i, ctypes.POINTER(i), ctypes.POINTER(ctypes.c_double)]
        lib.mg_attn_profile_read.restype = i
        lib.mg_attn_kernel_count.argtypes = []
        lib.mg_attn_kernel_count.restype = i
        lib.mg_attn_kernel_name.argtypes = [i]
        lib.mg_attn_kernel_name.restype = ctypes.c_char_p
        for name in ("mg_conv2d_grad_input", "mg_conv2d_grad_weight"):
            fn = getattr(lib, name)
            fn.argtypes = [vp, vp, vp] + [i] * 10 + [vp]
            fn.restype = i
        _lib = lib
        return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dims(Q):
    if Q.dim() != 4:
        raise ValueError("expected a [B, H, L, D] tensor")
    return tuple(int(x) for x in Q.shape)


def _contract(c) -> int:
    """A contract as its int value: an int, or a name such as "accel_f16+out16"
    (base contract, then "+"-joined flags)."""
    if not isinstance(c, str):
        return int(c)
    base, *flags = c.split("+")
    v = CONTRACTS[base]
    for f in flags:
        v |= FLAGS[f]
    return v


def _out_dtype(contract):
    """torch dtype of O, dQ, dK, dV under a contract."""
    import torch
    c = _contract(contract)
    if not c & OUT_16:
        return torch.float32
    return torch.float16 if (c & 0xFF) == ACCEL_F16 else torch.bfloat16


def mg_status_string(status: int) -> str:
    return load_library().mg_status_string(int(status)).decode()


def mg_attn_fwd(Q, K, V, O, LSE, causal, scale, contract, stream=None) -> int:
    B, H, L, D = _dims(Q)
    rc = load_library().mg_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, L, D,
                                    int(bool(causal)), float(scale), _contract(contract),
                                    _stream(stream))
    if rc != MG_OK:
        raise MgError(rc, "mg_attn_fwd")
    return rc


def mg_attn_bwd_workspace_bytes(B, H, L, D, contract) -> int:
    return int(load_library().mg_attn_bwd_workspace_bytes(B, H, L, D, _contract(contract)))


def mg_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, causal, scale, contract, workspace,
                stream=None) -> int:
    B, H, L, D = _dims(Q)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load_library().mg_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE),
                                    _ptr(dQ), _ptr(dK), _ptr(dV), B, H, L, D,
                                    int(bool(causal)), float(scale), _contract(contract),
                                    _ptr(workspace), ws_bytes, _stream(stream))
    if rc != MG_OK:
        raise MgError(rc, "mg_attn_bwd")
    return rc


MASKS = {"none": 0, "causal": 1, "causal_bottom_right": 2}


def _mask(m) -> int:
    return MASKS[m] if isinstance(m, str) else int(m)


def mg_attn_fwd_ex(Q, K, V, O, LSE, mask, scale, contract, stream=None) -> int:
    """Cross-attention forward: Q, O [B, H, Lq, D]; K, V [B, H, Lk, D]; LSE [B, H, Lq];
    mask "none", "causal" (top-left) or "causal_bottom_right"."""
    B, H, Lq, D = _dims(Q)
    Lk = int(K.shape[2])
    rc = load_library().mg_attn_fwd_ex(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H, Lq,
                                       Lk, D, _mask(mask), float(scale), _contract(contract),
                                       _stream(stream))
    if rc != MG_OK:
        raise MgError(rc, "mg_attn_fwd_ex")
    return rc


def mg_attn_bwd_workspace_bytes_ex(B, H, Lq, Lk, D, contract) -> int:
    return int(load_library().mg_attn_bwd_workspace_bytes_ex(B, H, Lq, Lk, D, _contract(contract)))


def mg_attn_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, mask, scale, contract, workspace,
                   stream=None) -> int:
    """Cross-attention backward (shapes as in mg_attn_fwd_ex; dQ like Q, dK and dV like K)."""
    B, H, Lq, D = _dims(Q)
    Lk = int(K.shape[2])
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load_library().mg_attn_bwd_ex(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(LSE),
                                       _ptr(dQ), _ptr(dK), _ptr(dV), B, H, Lq, Lk, D,
                                       _mask(mask), float(scale), _contract(contract),
                                       _ptr(workspace), ws_bytes, _stream(stream))
    if rc != MG_OK:
        raise MgError(rc, "mg_attn_bwd_ex")
    return rc


def mg_attn_fwd_padded(Q, K, V, O, LSE, kv_len, mask, scale, contract, stream=None) -> int:
    """Forward with per-batch key padding: kv_len is a CUDA int32 tensor of B
    lengths (or None); shapes and mask as in mg_attn_fwd_ex."""
    B, H, Lq, D = _dims(Q)
    Lk = int(K.shape[2])
    rc = load_library().mg_attn_fwd_padded(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE),
                                           _ptr(kv_len), B, H, Lq, Lk, D, _mask(mask),
                                           float(scale), _contract(contract), _stream(stream))
    if rc != MG_OK:
        raise MgError(rc, "mg_attn_fwd_padded")
    return rc


def mg_attn_bwd_padded(Q, K, V, O, dO, LSE, dQ, dK, dV, kv_len, mask, scale, contract,
                       workspace, stream=None) -> int:
    """Backward with per-batch key padding (shapes as in mg_attn_bwd_ex)."""
    B, H, Lq, D = _dims(Q)
    Lk = int(K.shape[2])
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load_library().mg_attn_bwd_padded(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO),
                                           _ptr(LSE), _ptr(dQ), _ptr(dK), _ptr(dV),
                                           _ptr(kv_len), B, H, Lq, Lk, D, _mask(mask),
                                           float(scale), _contract(contract), _ptr(workspace),
                                           ws_bytes, _stream(stream))
    if rc != MG_OK:
        raise MgError(rc, "mg_attn_bwd_padded")
    return rc


def mg_attn_fwd_decode_workspace_bytes(B, H, Lq, Lk, D, contract) -> int:
    return int(load_library().mg_attn_fwd_decode_workspace_bytes(B, H, Lq, Lk, D,
                                                                  _contract(contract)))


def mg_attn_fwd_decode(Q, K, V, O, LSE, mask, scale, contract, workspace, stream=None) -> int:
    """Split-key forward for Lq <= 8 query rows (decoding); shapes and mask as in
    mg_attn_fwd_ex, plus a workspace of mg_attn_fwd_decode_workspace_bytes() bytes."""
    B, H, Lq, D = _dims(Q)
    Lk = int(K.shape[2])
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load_library().mg_attn_fwd_decode(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(LSE), B, H,
                                           Lq, Lk, D, _mask(mask), float(scale),
                                           _contract(contract), _ptr(workspace), ws_bytes,
                                           _stream(stream))
    if rc != MG_OK:
        raise MgError(rc, "mg_attn_fwd_decode")
    return rc


def _conv_dims(X_shape, Wt_shape, stride: int, pad: int):
    N, H, W, C = (int(x) for x in X_shape)
    K, R, S, C2 = (int(x) for x in Wt_shape)
    if C2 != C:
        raise ValueError("X [N,H,W,C] and Wt [K,R,S,C] must share C")
    return N, H, W, C, K, R, S


def conv_out_size(H: int, W: int, R: int, S: int, stride: int, pad: int):
    """(P, Q): output rows and columns of the convolution."""
    return (H + 2 * pad - R) // stride + 1, (W + 2 * pad - S) // stride + 1


def mg_conv2d_grad_input(dY, Wt, dX, stride: int, pad: int, contract="accel",
                         stream=None) -> int:
    """dX [N,H,W,C] (f32, overwritten) from dY [N,P,Q,K] and Wt [K,R,S,C] (16-bit)."""
    N, H, W, C, K, R, S = _conv_dims(dX.shape, Wt.shape, stride, pad)
    if tuple(dY.shape) != (N,) + conv_out_size(H, W, R, S, stride, pad) + (K,):
        raise ValueError("dY does not match the convolution's output shape")
    rc = load_library().mg_conv2d_grad_input(_ptr(dY), _ptr(Wt), _ptr(dX), N, H, W, C, K, R, S,
                                             int(stride), int(pad), _contract(contract),
                                             _stream(stream))
    if rc != MG_OK:
        raise MgError(rc, "mg_conv2d_grad_input")
    return rc


def mg_conv2d_grad_weight(X, dY, dW, stride: int, pad: int, contract="accel",
                          stream=None) -> int:
    """dW [K,R,S,C] (f32, overwritten) from X [N,H,W,C] and dY [N,P,Q,K] (16-bit)."""
    N, H, W, C, K, R, S = _conv_dims(X.shape, dW.shape, stride, pad)
    if tuple(dY.shape) != (N,) + conv_out_size(H, W, R, S, stride, pad) + (K,):
        raise ValueError("dY does not match the convolution's output shape")
    rc = load_library().mg_conv2d_grad_weight(_ptr(X), _ptr(dY), _ptr(dW), N, H, W, C, K, R, S,
                                              int(stride), int(pad), _contract(contract),
                                              _stream(stream))
    if rc != MG_OK:
        raise MgError(rc, "mg_conv2d_grad_weight")
    return rc


def mg_get_device_error(stream=None) -> int:
    return int(load_library().mg_get_device_error(_stream(stream)))


def mg_attn_profile_enable(enable: bool, capacity: int = 4096) -> None:
    rc = load_library().mg_attn_profile_enable(int(bool(enable)), int(capacity))
    if rc != MG_OK:
        raise MgError(rc, "mg_attn_profile_enable")


def mg_attn_profile_read(kernel: int):
    n = ctypes.c_int(0)
    ms = ctypes.c_double(0.0)
    rc = load_library().mg_attn_profile_read(int(kernel), ctypes.byref(n), ctypes.byref(ms))
    if rc != MG_OK:
        raise MgError(rc, "mg_attn_profile_read")
    return n.value, ms.value


def mg_attn_kernel_count() -> int:
    return int(load_library().mg_attn_kernel_count())


def mg_attn_kernel_name(kernel: int) -> str:
    return load_library().mg_attn_kernel_name(int(kernel)).decode()


# ------------------------------------------------------------ conveniences
def attention_fwd(Q, K, V, causal: bool, scale: float, contract, stream=None):
    """Allocate O (f32, or 16-bit under MG_OUT_16) and LSE (f32) with PyTorch
    and run mg_attn_fwd."""
    import torch
    B, H, L, D = _dims(Q)
    O = torch.empty((B, H, L, D), dtype=_out_dtype(contract), device=Q.device)
    LSE = torch.empty((B, H, L), dtype=torch.float32, device=Q.device)
    mg_attn_fwd(Q, K, V, O, LSE, causal, scale, contract, stream)
    return O, LSE


def attention_bwd(Q, K, V, O, dO, LSE, causal: bool, scale: float, contract, stream=None,
                  workspace=None):
    """Allocate dQ, dK, dV (f32, or 16-bit under MG_OUT_16) and the workspace
    with PyTorch; run mg_attn_bwd."""
    import torch
    B, H, L, D = _dims(Q)
    dQ = torch.empty((B, H, L, D), dtype=_out_dtype(contract), device=Q.device)
    dK = torch.empty_like(dQ)
    dV = torch.empty_like(dQ)
    if workspace is None:
        nbytes = mg_attn_bwd_workspace_bytes(B, H, L, D, contract)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=Q.device)
    mg_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, causal, scale, contract, workspace, stream)
    return dQ, dK, dV
