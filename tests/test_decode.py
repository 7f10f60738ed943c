"""The split-key decode forward (mg_attn_fwd_decode: at most 8 query rows per
head, the key axis split over many CTAs and merged) against the fp64 oracle,
element by element: one to eight query rows, key lengths that are below, at and
just past one 32-key tile and span many splits, every mask (with empty rows under
the bottom-right alignment when Lq > Lk), every head dim, both contracts, and the
long-cache shape the benchmark times (B=1, H=8, Lq=1, Lk=32768, D=128)."""
import numpy as np
import pytest

import attention_forward_backward_gb300 as mg
import oracle
from attention_forward_backward_gb300 import synth
from parity_util import compare_ex, device_inputs, run_gpu_decode

pytestmark = pytest.mark.gpu

MASKS = ("none", "causal", "causal_bottom_right")


def _check(B, H, Lq, Lk, D, mask, contract, seed):
    host = synth.cross_inputs(B, H, Lq, Lk, D, contract, seed_cfg=seed)
    host.pop("dO")
    dev, vals = device_inputs(host, contract)
    scale = D ** -0.5
    got = run_gpu_decode(dev, mask, scale, contract)
    O, LSE = oracle.attn_fwd_ex(vals["Q"], vals["K"], vals["V"], mask, scale)
    errs, bad = compare_ex(got, {"O": O, "LSE": LSE}, contract)
    assert not bad, ((B, H, Lq, Lk, D, mask, contract), errs)
    return got, {"O": O, "LSE": LSE}


@pytest.mark.parametrize("contract", ["accel", "strict"])
@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Lk", [1, 31, 32, 33, 1000, 5000])
@pytest.mark.parametrize("Lq", [1, 3, 8])
def test_decode_parity(Lq, Lk, mask, contract):
    _check(1, 3, Lq, Lk, 64, mask, contract, seed=1100 + Lq + Lk % 97)


@pytest.mark.parametrize("contract", ["accel", "strict"])
@pytest.mark.parametrize("D", [32, 128])
@pytest.mark.parametrize("mask", MASKS)
def test_decode_head_dims(D, mask, contract):
    _check(2, 3, 5, 2000, D, mask, contract, seed=1110 + D)


@pytest.mark.parametrize("contract", ["accel", "strict"])
def test_decode_many_heads_few_splits(contract):
    """B*H = 256 heads: about two splits per head, each of thousands of keys."""
    _check(4, 64, 2, 4096, 128, "causal_bottom_right", contract, seed=1120)


@pytest.mark.parametrize("contract", ["accel", "strict"])
def test_decode_long_cache(contract):
    """The benchmarked decode shape: one new token against a 32768-key cache."""
    _check(1, 8, 1, 32768, 128, "causal_bottom_right", contract, seed=1130)


@pytest.mark.parametrize("contract", ["accel", "strict"])
def test_decode_empty_rows(contract):
    """Bottom-right with Lq = 8 > Lk = 3: rows 0..4 see no key (O = 0, LSE = -inf);
    top-left causal with Lk = 5000: row i sees keys 0..i only, so every split but
    the first is empty for every row and the merge must ignore them."""
    got, _ = _check(1, 2, 8, 3, 64, "causal_bottom_right", contract, seed=1140)
    assert np.all(np.isneginf(got["LSE"][:, :, :5])) and np.all(got["O"][:, :, :5] == 0)
    assert np.all(np.isfinite(got["LSE"][:, :, 5:]))
    _check(1, 2, 8, 5000, 64, "causal", contract, seed=1141)


def test_decode_rejects_nine_rows():
    import torch
    x = torch.zeros((1, 1, 9, 64), dtype=torch.float32, device="cuda")
    kv = torch.zeros((1, 1, 100, 64), dtype=torch.float32, device="cuda")
    O = torch.empty_like(x)
    LSE = torch.empty((1, 1, 9), device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(mg.MgError) as ei:
        mg.mg_attn_fwd_decode(x, kv, kv.clone(), O, LSE, "none", 0.125, "strict", ws)
    assert ei.value.status == mg.MG_ERR_UNSUPPORTED


@pytest.mark.parametrize("contract", ["accel", "strict"])
@pytest.mark.parametrize("Lk", [127, 128, 129, 255, 257, 1793])
def test_decode_tile_edges(Lk, contract):
    """Key lengths at and around the tensor-core kernel's 128-key tile."""
    _check(1, 2, 8, Lk, 128, "causal_bottom_right", contract, seed=1150 + Lk % 89)


@pytest.mark.parametrize("contract", ["accel", "strict"])
@pytest.mark.parametrize("mask", ["none", "causal_bottom_right"])
def test_decode_large_logits(mask, contract):
    """K scaled by 8 (logit standard deviation about 8 in base e): tile maxima
    move by far more than the lazy-rescale threshold from tile to tile, so the
    running reference and the accumulated output are rescaled many times."""
    B, H, Lq, Lk, D = 2, 2, 8, 3000, 128
    host = synth.cross_inputs(B, H, Lq, Lk, D, contract, seed_cfg=1160)
    host.pop("dO")
    base = synth.base_contract(contract)
    kv = host["K"] if base == "strict" else host["K"]["values"]
    host["K"] = synth.encode(np.ascontiguousarray(kv * np.float32(8.0)), contract)
    dev, vals = device_inputs(host, contract)
    scale = D ** -0.5
    got = run_gpu_decode(dev, mask, scale, contract)
    O, LSE = oracle.attn_fwd_ex(vals["Q"], vals["K"], vals["V"], mask, scale)
    errs, bad = compare_ex(got, {"O": O, "LSE": LSE}, contract)
    assert not bad, errs
