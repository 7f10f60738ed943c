"""ACCEL_BF16 parity: the tcgen05 kernels against the fp64 oracle, element by
element, through the C ABI (gate 2e-2, max-abs error over max-abs reference).

The oracle consumes the bf16-rounded inputs (upcast exactly), so only the
kernels' own arithmetic (bf16 P and dS operands, f32 accumulation, approximate
exp2) is measured, not the input quantisation."""
import numpy as np
import pytest

import oracle
from attention_forward_backward_gb300 import synth
from parity_util import compare, device_inputs, run_gpu

pytestmark = pytest.mark.gpu


def _full_check(w: synth.Workload, bwd=True):
    host = synth.inputs(w, "accel")
    dev, vals = device_inputs(host, "accel")
    got = run_gpu(dev, w.causal, w.scale, "accel", bwd=bwd)
    if bwd:
        ref = oracle.attn_bwd(vals["Q"], vals["K"], vals["V"], vals["dO"], w.causal, w.scale)
    else:
        O, LSE = oracle.attn_fwd(vals["Q"], vals["K"], vals["V"], w.causal, w.scale)
        ref = {"O": O, "LSE": LSE}
    errs, bad = compare(got, ref, "accel")
    assert not bad, (w.name, errs)
    return errs


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_accel_configs(cfg):
    _full_check(synth.WORKLOADS[cfg])


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("L", [1, 7, 64, 65, 128, 129, 197, 300])
@pytest.mark.parametrize("causal", [True, False])
def test_accel_edge_shapes(D, L, causal):
    """Sub-tile, exactly-one-tile and ragged sequence lengths for every head dim."""
    _full_check(synth.custom_workload(1, 2, L, D, causal, seed_cfg=950 + D))


def test_accel_forward_only_first():
    """Forward alone (no backward launched) on a multi-tile causal case."""
    _full_check(synth.custom_workload(2, 2, 640, 128, True, seed_cfg=960), bwd=False)


def test_accel_large_logits_noncausal():
    _full_check(synth.custom_workload(2, 3, 300, 64, False, seed_cfg=970, qk_gain=4.0))


def test_accel_long_sequence_sampled():
    """The long-sequence causal workload (B=2, H=32, L=8192, D=128) in the launch configuration
    the benchmark times: two heads in full (forward and backward) and every
    fifth head on sampled query rows (O and LSE)."""
    w = synth.WORKLOADS[5]
    host = synth.inputs(w, "accel")
    dev, vals = device_inputs(host, "accel")
    got = run_gpu(dev, w.causal, w.scale, "accel", bwd=True)
    BH = w.B * w.H
    flat = {k: v.reshape(BH, w.L, -1) if v.ndim == 4 else v.reshape(BH, w.L)
            for k, v in got.items()}
    vflat = {k: v.reshape(BH, w.L, w.D) for k, v in vals.items()}
    for h in (0, BH - 1):
        ref = oracle.attn_bwd(vflat["Q"][h], vflat["K"][h], vflat["V"][h], vflat["dO"][h],
                              True, w.scale)
        sub = {k: flat[k][h] for k in ("O", "LSE", "dQ", "dK", "dV")}
        errs, bad = compare(sub, ref, "accel")
        assert not bad, (h, errs)
    rows = np.array([0, 1, 127, 128, 255, 256, 4095, 8190, 8191])
    for h in range(0, BH, 5):
        O, LSE = oracle.attn_fwd_rows(vflat["Q"][h], vflat["K"][h], vflat["V"][h], rows, True,
                                      w.scale)
        errs, bad = compare({"O": flat["O"][h][rows], "LSE": flat["LSE"][h][rows]},
                            {"O": O, "LSE": LSE}, "accel")
        assert not bad, (h, errs)


def test_accel_causal_first_row():
    """Row 0 attends only key 0, so O[0] = V[0]. P = 1 enters the MMA exactly
    (bf16); the f32 row sum can differ from 1 by the rounding of one fused
    multiply-add, hence the 1e-6 relative tolerance."""
    w = synth.custom_workload(2, 2, 77, 64, True, seed_cfg=980)
    dev, vals = device_inputs(synth.inputs(w, "accel"), "accel")
    got = run_gpu(dev, True, w.scale, "accel", bwd=False)
    np.testing.assert_allclose(got["O"][:, :, 0, :], vals["V"][:, :, 0, :], rtol=1e-6, atol=0)


def test_accel_repeatable_forward():
    """The forward has no atomics: two calls give bit-identical O and LSE."""
    w = synth.custom_workload(1, 4, 513, 128, True, seed_cfg=985)
    dev, _ = device_inputs(synth.inputs(w, "accel"), "accel")
    a = run_gpu(dev, True, w.scale, "accel", bwd=False)
    b = run_gpu(dev, True, w.scale, "accel", bwd=False)
    np.testing.assert_array_equal(a["O"], b["O"])
    np.testing.assert_array_equal(a["LSE"], b["LSE"])


def test_accel_pass_dq_mode_in_child():
    """The two-pass backward (dK/dV kernel with two query blocks in flight, then
    the separate dQ pass; MG_DQ_MODE=pass) on the decoder, encoder and large-logit
    workloads and on sub-tile,
    one-tile and ragged lengths for every head dim, causal and not, in a child
    process because the mode is read once per process."""
    import os
    import subprocess
    import sys
    import textwrap
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {root!r}); sys.path.insert(0, {os.path.join(root, 'tests')!r})
        import oracle
        from attention_forward_backward_gb300 import synth
        from parity_util import compare, device_inputs, run_gpu
        cases = [synth.WORKLOADS[2], synth.WORKLOADS[3], synth.WORKLOADS[4],
                 synth.custom_workload(1, 3, 300, 128, True, seed_cfg=990)]
        for D in (32, 64, 128):
            for L in (1, 63, 64, 65, 200):
                for causal in (True, False):
                    cases.append(synth.custom_workload(1, 2, L, D, causal, seed_cfg=991 + D))
        for w in cases:
            dev, vals = device_inputs(synth.inputs(w, "accel"), "accel")
            got = run_gpu(dev, w.causal, w.scale, "accel")
            ref = oracle.attn_bwd(vals["Q"], vals["K"], vals["V"], vals["dO"], w.causal, w.scale)
            errs, bad = compare(got, ref, "accel")
            assert not bad, (w.name, errs)
        print("PASS-MODE-OK")
    """)
    env = dict(os.environ, MG_DQ_MODE="pass")
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0 and "PASS-MODE-OK" in res.stdout, res.stdout + res.stderr
