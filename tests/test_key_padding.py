"""Per-batch key padding (mg_attn_fwd_padded / mg_attn_bwd_padded): batch
element b keeps its first kv_len[b] key rows, the rest of K and V is padding.
Compared element by element with the fp64 oracle (``oracle.attn_bwd_padded``:
each batch element is the cross-attention problem with kv_len[b] keys). The
padding rows hold large finite values, so any leak into a result shows. Cases:
kv_len = 1, ragged lengths inside a key tile, the full length, a batch element
with no key at all (empty softmax on every row), every mask, Lq != Lk, head dims
32/64/128, both contracts, and the two-pass ACCEL backward."""
import numpy as np
import pytest

import attention_forward_backward_gb300 as mg
import oracle
from attention_forward_backward_gb300 import synth
from parity_util import compare_ex, device_inputs

pytestmark = pytest.mark.gpu

MASKS = ("none", "causal", "causal_bottom_right")


def padded_inputs(B, H, Lq, Lk, D, kv_len, contract, seed):
    """Seeded inputs whose padding rows of K and V are 300x the seeded values."""
    host = synth.cross_inputs(B, H, Lq, Lk, D, contract, seed_cfg=seed)
    for t in ("K", "V"):
        if contract == "strict":
            x = host[t]
            for b, n in enumerate(kv_len):
                x[b, :, n:] *= 300.0
        else:
            x = host[t]["values"].copy()
            for b, n in enumerate(kv_len):
                x[b, :, n:] *= 300.0
            bits = synth.round_to_bf16(x)
            host[t] = {"bits": bits, "values": synth.bf16_bits_to_f32(bits)}
    return host


def run_padded(dev, kv_len, mask, scale, contract):
    import torch
    Q, K, V, dO = dev["Q"], dev["K"], dev["V"], dev["dO"]
    B, H, Lq, D = Q.shape
    Lk = K.shape[2]
    nan = float("nan")
    lens = torch.tensor(kv_len, dtype=torch.int32, device=Q.device)
    O = torch.full((B, H, Lq, D), nan, device=Q.device)
    LSE = torch.full((B, H, Lq), nan, device=Q.device)
    mg.mg_attn_fwd_padded(Q, K, V, O, LSE, lens, mask, scale, contract)
    dQ = torch.full((B, H, Lq, D), nan, device=Q.device)
    dK = torch.full((B, H, Lk, D), nan, device=Q.device)
    dV = torch.full((B, H, Lk, D), nan, device=Q.device)
    nbytes = mg.mg_attn_bwd_workspace_bytes_ex(B, H, Lq, Lk, D, contract)
    ws = torch.full((nbytes // 4,), nan, device=Q.device)
    mg.mg_attn_bwd_padded(Q, K, V, O, dO, LSE, dQ, dK, dV, lens, mask, scale, contract, ws)
    torch.cuda.synchronize()
    assert mg.mg_get_device_error() == mg.MG_OK
    return {k: v.cpu().numpy() for k, v in dict(O=O, LSE=LSE, dQ=dQ, dK=dK, dV=dV).items()}


def check(B, H, Lq, Lk, D, kv_len, mask, contract, seed):
    host = padded_inputs(B, H, Lq, Lk, D, kv_len, contract, seed)
    dev, vals = device_inputs(host, contract)
    scale = D ** -0.5
    got = run_padded(dev, kv_len, mask, scale, contract)
    ref = oracle.attn_bwd_padded(vals["Q"], vals["K"], vals["V"], vals["dO"], kv_len, mask,
                                 scale)
    errs, bad = compare_ex(got, ref, contract)
    assert not bad, ((B, H, Lq, Lk, D, kv_len, mask, contract), errs)
    for b, n in enumerate(kv_len):
        assert np.all(got["dK"][b, :, n:] == 0) and np.all(got["dV"][b, :, n:] == 0)
        if n == 0:
            assert np.all(np.isneginf(got["LSE"][b])) and np.all(got["O"][b] == 0)
            assert np.all(got["dQ"][b] == 0)
    return got


@pytest.mark.parametrize("contract", ["accel", "strict"])
@pytest.mark.parametrize("mask", MASKS)
def test_padded_lengths(mask, contract):
    """kv_len = 1, 77 (inside a key tile), the full 200, and 0 in one batch."""
    check(4, 2, 150, 200, 64, [1, 77, 200, 0], mask, contract, seed=1100)


@pytest.mark.parametrize("contract", ["accel", "strict"])
@pytest.mark.parametrize("D", [32, 128])
@pytest.mark.parametrize("mask", MASKS)
def test_padded_head_dims(D, mask, contract):
    check(3, 2, 300, 513, D, [513, 129, 128], mask, contract, seed=1110 + D)


@pytest.mark.parametrize("contract", ["accel", "strict"])
def test_padded_text_conditioning(contract):
    """Text cross-attention: many query rows against a padded 77-key text."""
    check(3, 4, 640, 77, 64, [77, 12, 40], "none", contract, seed=1120)


@pytest.mark.parametrize("contract", ["accel", "strict"])
def test_null_lengths_are_the_ex_calls(contract):
    """kv_len = NULL is exactly mg_attn_fwd_ex / mg_attn_bwd_ex."""
    import torch
    from parity_util import run_gpu_ex
    host = synth.cross_inputs(2, 2, 130, 260, 64, contract, seed_cfg=1130)
    dev, _ = device_inputs(host, contract)
    a = run_gpu_ex(dev, "causal_bottom_right", 0.125, contract)
    Q, K, V, dO = dev["Q"], dev["K"], dev["V"], dev["dO"]
    O = torch.empty((2, 2, 130, 64), device=Q.device)
    LSE = torch.empty((2, 2, 130), device=Q.device)
    mg.mg_attn_fwd_padded(Q, K, V, O, LSE, None, "causal_bottom_right", 0.125, contract)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(O.cpu().numpy(), a["O"])
    np.testing.assert_array_equal(LSE.cpu().numpy(), a["LSE"])


def test_padded_two_pass_backward_in_child():
    """The two-pass ACCEL backward (MG_DQ_MODE=pass) under padding, in a child
    process because the mode is read once per process."""
    import os
    import subprocess
    import sys
    import textwrap
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {root!r}); sys.path.insert(0, {os.path.join(root, 'tests')!r})
        from test_key_padding import check, MASKS
        for mask in MASKS:
            for D in (64, 128):
                check(4, 2, 150, 200, D, [1, 77, 200, 0], mask, "accel", seed=1140)
        print("PADDED-PASS-OK")
    """)
    env = dict(os.environ, MG_DQ_MODE="pass")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "PADDED-PASS-OK" in r.stdout, r.stdout + r.stderr
