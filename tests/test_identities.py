"""Identities of the attention derivative that hold at any size, checked on
every head of the full-size long-sequence workload (B=2, H=32, L=8192, D=128,
causal) in the launch configuration the benchmark times. The element-by-element
oracle comparisons at this size sample heads and rows (test_parity_*); these
cover all heads and all key rows.

From the definitions (softmax rows sum to one over the allowed keys):
  sum_j dV_j = sum_j sum_i P_ij dO_i = sum_i dO_i
  sum_j dS_ij = dO_i . (sum_j P_ij V_j) - Dvec_i = dO_i . O_i - Dvec_i = 0,
  hence sum_j dK_j = scale * sum_i (sum_j dS_ij) Q_i = 0.
Each residual is compared with the root-sum-square of the terms it sums (what a
sum of unrelated vectors would give), so a dropped tile or a wrong sign shows
up at order one, while the rounding of P and dS to bf16 leaves about 2^-9.
The oracle satisfies both identities too (test_oracle_pins)."""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

from attention_forward_backward_gb300 import synth
from parity_util import device_inputs, run_gpu

TOL = {"strict": 1e-4, "accel": 2e-2}


def identity_residuals(got: dict, vals: dict, w) -> dict:
    """Largest normalised residual over heads of the two identities."""
    BH = w.B * w.H
    dK = got["dK"].reshape(BH, w.L, w.D).astype(np.float64)
    dV = got["dV"].reshape(BH, w.L, w.D).astype(np.float64)
    dO = vals["dO"].reshape(BH, w.L, w.D).astype(np.float64)
    rss_k = np.sqrt(np.sum(dK * dK, axis=(1, 2)))
    rss_v = np.sqrt(np.sum(dV * dV, axis=(1, 2)) + np.sum(dO * dO, axis=(1, 2)))
    res_k = np.linalg.norm(dK.sum(axis=1), axis=1) / rss_k
    res_v = np.linalg.norm(dV.sum(axis=1) - dO.sum(axis=1), axis=1) / rss_v
    return {"sum_dK": float(res_k.max()), "sum_dV_minus_sum_dO": float(res_v.max())}


def test_identity_check_flags_planted_mistakes():
    """The residuals are at rounding level on the oracle's gradients and of order
    one when a mistake is planted in them (a key tile dropped from dK, a sign
    flipped in dV), on a small causal case."""
    import oracle
    w = synth.custom_workload(1, 2, 300, 64, True, seed_cfg=1990)
    vals = synth.inputs(w, "strict")
    ref = oracle.attn_bwd(vals["Q"], vals["K"], vals["V"], vals["dO"], True, w.scale)
    got = {k: ref[k].astype(np.float32) for k in ("dK", "dV")}
    clean = identity_residuals(got, vals, w)
    assert max(clean.values()) < 1e-6, clean
    bad = {k: v.copy() for k, v in got.items()}
    bad["dK"][:, :, 128:256, :] = 0.0
    assert identity_residuals(bad, vals, w)["sum_dK"] > 0.05
    bad = {k: v.copy() for k, v in got.items()}
    bad["dV"][:, 1, :, :] *= -1.0
    assert identity_residuals(bad, vals, w)["sum_dV_minus_sum_dO"] > 0.05


@pytest.mark.gpu
@pytest.mark.parametrize("contract", ["accel", "strict"])
def test_long_sequence_identities_every_head(contract):
    w = synth.WORKLOADS[5]
    dev, vals = device_inputs(synth.inputs(w, contract), contract)
    got = run_gpu(dev, w.causal, w.scale, contract, bwd=True)
    res = identity_residuals(got, vals, w)
    assert all(v <= TOL[contract] for v in res.values()), res
    # O is a convex combination of V rows and LSE is finite on every row
    assert np.all(np.isfinite(got["LSE"]))
    assert np.abs(got["O"]).max() <= np.abs(vals["V"]).max() * (1 + 1e-3)


@pytest.mark.gpu
def test_long_sequence_identities_two_pass_backward_in_child():
    """The same identities through the two-pass backward (dK/dV kernel with two
    query blocks in flight, then the dQ pass; MG_DQ_MODE=pass), in a child
    process because the mode is read once per process."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {root!r}); sys.path.insert(0, {os.path.join(root, 'tests')!r})
        from attention_forward_backward_gb300 import synth
        from parity_util import device_inputs, run_gpu
        from test_identities import identity_residuals, TOL
        w = synth.WORKLOADS[5]
        dev, vals = device_inputs(synth.inputs(w, "accel"), "accel")
        got = run_gpu(dev, w.causal, w.scale, "accel", bwd=True)
        res = identity_residuals(got, vals, w)
        assert all(v <= TOL["accel"] for v in res.values()), res
        print("IDENTITIES-OK", res)
    """)
    env = dict(os.environ, MG_DQ_MODE="pass")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "IDENTITIES-OK" in r.stdout, r.stdout + r.stderr


@pytest.mark.gpu
@pytest.mark.parametrize("contract", ["accel", "strict"])
def test_long_single_head_identities_and_rows(contract):
    """One head of L = 32768 (D = 128, causal): 512 query blocks per key block in
    the backward and 256 key tiles per query tile in the forward. Sampled rows of
    O and LSE against the oracle, and both identities over the whole head."""
    import oracle
    from parity_util import compare
    w = synth.custom_workload(1, 1, 32768, 128, True, seed_cfg=1995)
    dev, vals = device_inputs(synth.inputs(w, contract), contract)
    got = run_gpu(dev, w.causal, w.scale, contract, bwd=True)
    res = identity_residuals(got, vals, w)
    assert all(v <= TOL[contract] for v in res.values()), res
    rows = np.array([0, 1, 127, 128, 16383, 16384, 32766, 32767])
    Q, K, V = (vals[k].reshape(w.L, w.D) for k in ("Q", "K", "V"))
    O, LSE = oracle.attn_fwd_rows(Q, K, V, rows, True, w.scale)
    errs, bad = compare({"O": got["O"].reshape(w.L, w.D)[rows], "LSE": got["LSE"].reshape(w.L)[rows]},
                        {"O": O, "LSE": LSE}, contract)
    assert not bad, errs
