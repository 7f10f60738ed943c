"""Shared helpers of the parity tests: run the CUDA path through the C ABI on
seeded inputs and compare element by element with the fp64 oracle.

Error metric (per output tensor X in O, dQ, dK, dV):
    err(X) = max |X_gpu - X_ref| / max(max |X_ref|, 1e-2 * M)
where M is the largest max |Y_ref| over the outputs Y of the same call. The
floor only matters where the exact result is identically zero: L = 1 gives
dQ = dK = 0, which f32 reaches only up to the cancellation in dP - Dvec (two
equal dot products of length D); on every other case the denominator is
max |X_ref|.
Gates: STRICT_F32 <= 1e-4, ACCEL_BF16 <= 2e-2. LSE is compared by
max |LSE_gpu - LSE_ref| / max(1, max |LSE_ref|) with the same gates.
"""
from __future__ import annotations

import numpy as np

import attention_forward_backward_gb300 as mg
from attention_forward_backward_gb300 import synth

class _Tol(dict):
    """Parity gate per contract name; a name with flags ("accel+hilo+out16")
    takes its base contract's gate."""

    def __missing__(self, contract):
        return self[synth.base_contract(contract)]


TOL = _Tol({"strict": 1e-4, "accel": 2e-2, "accel_f16": 2e-2})


def rel_err(got, ref, floor: float = 0.0) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not ref.size:
        return 0.0
    if not np.all(np.isfinite(got)):
        return float("inf")
    denom = max(float(np.max(np.abs(ref))), floor, 1e-300)
    return float(np.max(np.abs(got - ref))) / denom


def lse_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if not np.all(np.isfinite(got)):
        return float("inf")
    return float(np.max(np.abs(got - ref))) / max(1.0, float(np.max(np.abs(ref))))


def device_inputs(host: dict, contract: str, device="cuda"):
    """Torch device tensors for the CUDA path and the f64-exact values the
    oracle consumes (bf16 values for ACCEL, f32 values for STRICT)."""
    import torch
    dev, vals = {}, {}
    base = synth.base_contract(contract)
    for k, x in host.items():
        if base == "strict":
            dev[k] = torch.from_numpy(x).to(device)
            vals[k] = x
        else:
            bits = np.ascontiguousarray(x["bits"]).view(np.int16)
            dt = torch.float16 if base == "accel_f16" else torch.bfloat16
            dev[k] = torch.from_numpy(bits).view(dt).to(device)
            vals[k] = x["values"]
    return dev, vals


def run_gpu(dev: dict, causal: bool, scale: float, contract: str, bwd: bool = True,
            poison: bool = True):
    """Forward (+ backward) through the C ABI. Output buffers start as NaN so
    that an element the kernels fail to write shows up as an error."""
    import torch
    Q, K, V, dO = dev["Q"], dev["K"], dev["V"], dev["dO"]
    B, H, L, D = Q.shape
    O = torch.full((B, H, L, D), float("nan") if poison else 0.0, device=Q.device,
                   dtype=mg._out_dtype(contract))
    LSE = torch.full((B, H, L), float("nan") if poison else 0.0, device=Q.device)
    mg.mg_attn_fwd(Q, K, V, O, LSE, causal, scale, contract)
    out = {"O": O, "LSE": LSE}
    if bwd:
        dQ = torch.full_like(O, float("nan") if poison else 0.0)
        dK = torch.full_like(O, float("nan") if poison else 0.0)
        dV = torch.full_like(O, float("nan") if poison else 0.0)
        nbytes = mg.mg_attn_bwd_workspace_bytes(B, H, L, D, contract)
        ws = torch.full((nbytes // 4,), float("nan"), device=Q.device)
        mg.mg_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, causal, scale, contract, ws)
        out.update(dQ=dQ, dK=dK, dV=dV)
    torch.cuda.synchronize()
    assert mg.mg_get_device_error() == mg.MG_OK
    return {k: v.float().cpu().numpy() for k, v in out.items()}


def compare(got: dict, ref: dict, contract: str, keys=("O", "dQ", "dK", "dV")):
    tol = TOL[contract]
    errs = {}
    present = [k for k in keys if k in got]
    scale = max((float(np.max(np.abs(ref[k]))) for k in present if ref[k].size), default=0.0)
    for k in present:
        errs[k] = rel_err(got[k], ref[k], floor=1e-2 * scale)
    if "LSE" in got and "LSE" in ref:
        errs["LSE"] = lse_err(got["LSE"], ref["LSE"])
    bad = {k: e for k, e in errs.items() if not (e <= tol)}
    return errs, bad


def workload_inputs(w: synth.Workload, contract: str):
    return synth.inputs(w, contract)


def run_gpu_ex(dev: dict, mask: str, scale: float, contract: str, bwd: bool = True):
    """Cross-attention forward (+ backward) through the _ex calls, outputs
    poisoned with NaN first. Q, dO [B, H, Lq, D]; K, V [B, H, Lk, D]."""
    import torch
    Q, K, V, dO = dev["Q"], dev["K"], dev["V"], dev["dO"]
    B, H, Lq, D = Q.shape
    Lk = K.shape[2]
    nan = float("nan")
    odt = mg._out_dtype(contract)
    O = torch.full((B, H, Lq, D), nan, device=Q.device, dtype=odt)
    LSE = torch.full((B, H, Lq), nan, device=Q.device)
    mg.mg_attn_fwd_ex(Q, K, V, O, LSE, mask, scale, contract)
    out = {"O": O, "LSE": LSE}
    if bwd:
        dQ = torch.full((B, H, Lq, D), nan, device=Q.device, dtype=odt)
        dK = torch.full((B, H, Lk, D), nan, device=Q.device, dtype=odt)
        dV = torch.full((B, H, Lk, D), nan, device=Q.device, dtype=odt)
        nbytes = mg.mg_attn_bwd_workspace_bytes_ex(B, H, Lq, Lk, D, contract)
        ws = torch.full((nbytes // 4,), nan, device=Q.device)
        mg.mg_attn_bwd_ex(Q, K, V, O, dO, LSE, dQ, dK, dV, mask, scale, contract, ws)
        out.update(dQ=dQ, dK=dK, dV=dV)
    torch.cuda.synchronize()
    assert mg.mg_get_device_error() == mg.MG_OK
    return {k: v.float().cpu().numpy() for k, v in out.items()}


def compare_ex(got: dict, ref: dict, contract: str):
    """compare() for results that may hold empty-softmax rows: LSE must be -inf
    exactly where the oracle's is, the finite LSE values are compared as usual."""
    errs, bad = compare({k: v for k, v in got.items() if k != "LSE"},
                        {k: v for k, v in ref.items() if k != "LSE"}, contract)
    if "LSE" in got:
        empty = np.isneginf(ref["LSE"])
        if not np.array_equal(np.isneginf(got["LSE"]), empty):
            errs["LSE"] = float("inf")
        else:
            errs["LSE"] = lse_err(got["LSE"][~empty], ref["LSE"][~empty]) if (~empty).any() else 0.0
        if not errs["LSE"] <= TOL[contract]:
            bad = dict(bad, LSE=errs["LSE"])
    return errs, bad


def run_gpu_decode(dev: dict, mask: str, scale: float, contract: str):
    """Split-key decode forward (mg_attn_fwd_decode), outputs and workspace
    poisoned with NaN first. Q [B, H, Lq, D] with Lq <= 8; K, V [B, H, Lk, D]."""
    import torch
    Q, K, V = dev["Q"], dev["K"], dev["V"]
    B, H, Lq, D = Q.shape
    Lk = K.shape[2]
    nan = float("nan")
    O = torch.full((B, H, Lq, D), nan, device=Q.device)
    LSE = torch.full((B, H, Lq), nan, device=Q.device)
    nbytes = mg.mg_attn_fwd_decode_workspace_bytes(B, H, Lq, Lk, D, contract)
    ws = torch.full((nbytes // 4,), nan, device=Q.device)
    mg.mg_attn_fwd_decode(Q, K, V, O, LSE, mask, scale, contract, ws)
    torch.cuda.synchronize()
    assert mg.mg_get_device_error() == mg.MG_OK
    return {"O": O.cpu().numpy(), "LSE": LSE.cpu().numpy()}
