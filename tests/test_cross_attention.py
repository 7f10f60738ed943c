"""Cross attention (Lq query rows, Lk key rows) with no mask, the top-left and
the bottom-right causal alignment, through mg_attn_fwd_ex / mg_attn_bwd_ex,
against the fp64 oracle element by element. Includes rows with an empty softmax
(bottom-right, Lq > Lk: O = 0, LSE = -inf, dQ = 0), key blocks that no query
sees (top-left, Lk > Lq: dK = dV = 0), one query or one key, ragged lengths
across several tiles, and every head dim."""
import numpy as np
import pytest

import oracle
from attention_forward_backward_gb300 import synth
from parity_util import compare_ex, device_inputs, run_gpu_ex

pytestmark = pytest.mark.gpu

MASKS = ("none", "causal", "causal_bottom_right")
SHAPES = [(64, 200), (200, 64), (1, 300), (300, 1), (129, 129), (77, 513), (513, 77),
          (256, 384), (640, 256)]


def _check(B, H, Lq, Lk, D, mask, contract, seed):
    host = synth.cross_inputs(B, H, Lq, Lk, D, contract, seed_cfg=seed)
    dev, vals = device_inputs(host, contract)
    scale = D ** -0.5
    got = run_gpu_ex(dev, mask, scale, contract)
    ref = oracle.attn_bwd_ex(vals["Q"], vals["K"], vals["V"], vals["dO"], mask, scale)
    errs, bad = compare_ex(got, ref, contract)
    assert not bad, ((Lq, Lk, D, mask, contract), errs)
    return got, ref


@pytest.mark.parametrize("contract", ["accel", "strict"])
@pytest.mark.parametrize("mask", MASKS)
@pytest.mark.parametrize("Lq,Lk", SHAPES)
def test_cross_attention_parity(Lq, Lk, mask, contract):
    _check(1, 2, Lq, Lk, 64, mask, contract, seed=960 + Lq % 7 + 3 * (Lk % 5))


@pytest.mark.parametrize("contract", ["accel", "strict"])
@pytest.mark.parametrize("D", [32, 128])
@pytest.mark.parametrize("mask", MASKS)
def test_cross_attention_head_dims(D, mask, contract):
    _check(2, 2, 300, 170, D, mask, contract, seed=970 + D)
    _check(2, 2, 170, 300, D, mask, contract, seed=971 + D)


@pytest.mark.parametrize("contract", ["accel", "strict"])
def test_empty_rows_and_unseen_keys(contract):
    """Bottom-right with Lq > Lk: the first Lq - Lk rows are empty. Top-left with
    Lk > Lq: keys past Lq - 1 are seen by no query, their dK, dV are 0."""
    got, ref = _check(1, 2, 700, 90, 64, "causal_bottom_right", contract, seed=980)
    e = 700 - 90
    assert np.all(np.isneginf(got["LSE"][:, :, :e]))
    assert np.all(got["O"][:, :, :e] == 0) and np.all(got["dQ"][:, :, :e] == 0)
    got, ref = _check(1, 2, 90, 700, 64, "causal", contract, seed=981)
    assert np.all(got["dK"][:, :, 90:] == 0) and np.all(got["dV"][:, :, 90:] == 0)


@pytest.mark.parametrize("contract", ["accel", "strict"])
def test_square_bottom_right_equals_causal(contract):
    """With Lq = Lk the two alignments are the same mask and must give the same
    results as the self-attention calls."""
    import torch
    import attention_forward_backward_gb300 as mg
    w = synth.custom_workload(1, 2, 333, 64, True, seed_cfg=985)
    dev, _ = device_inputs(synth.inputs(w, contract), contract)
    a = run_gpu_ex(dev, "causal_bottom_right", w.scale, contract)
    b = run_gpu_ex(dev, "causal", w.scale, contract)
    O, LSE = mg.attention_fwd(dev["Q"], dev["K"], dev["V"], True, w.scale, contract)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(a["O"], b["O"])
    np.testing.assert_array_equal(a["LSE"], b["LSE"])
    np.testing.assert_array_equal(a["O"], O.cpu().numpy())
    np.testing.assert_array_equal(a["LSE"], LSE.cpu().numpy())


def test_cross_attention_two_pass_backward_in_child():
    """The same parity through the two-pass backward (MG_DQ_MODE=pass), in a
    child process because the mode is read once per process."""
    import os
    import subprocess
    import sys
    import textwrap
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {root!r}); sys.path.insert(0, {os.path.join(root, 'tests')!r})
        from test_cross_attention import _check, MASKS
        for (Lq, Lk) in ((64, 200), (200, 64), (1, 300), (300, 1), (700, 90), (90, 700)):
            for mask in MASKS:
                for D in (64, 128):
                    _check(1, 2, Lq, Lk, D, mask, "accel", seed=990 + Lq % 11)
        print("CROSS-PASS-OK")
    """)
    env = dict(os.environ, MG_DQ_MODE="pass")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "CROSS-PASS-OK" in r.stdout, r.stdout + r.stderr
