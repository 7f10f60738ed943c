"""Failure detection without a GPU fault: a bounded wait is made to run out on
purpose and must come back as MG_ERR_TIMEOUT through the device error word,
with the CUDA context still usable afterwards.

The injection is on the host side of the kernel's inputs: with
MG_FAULT_INJECT=skip_k_tile the forward's TMA producer never issues the load
of key tile 1, so the MMA issuer's wait on that tile's barrier (limited to
MG_WAIT_TIMEOUT_MS) expires. Nothing traps, faults or spins without a bound;
the kernel drains its own copies and MMAs, frees tensor memory and returns.
The run happens in a child process because the library reads both variables
once per process."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    sys.path.insert(0, {tests!r})
    import numpy as np, torch
    import attention_forward_backward_gb300 as mg
    import oracle
    from attention_forward_backward_gb300 import synth
    from parity_util import compare, device_inputs, run_gpu

    w = synth.custom_workload(1, 2, 512, 64, True, seed_cfg=995)
    dev, _ = device_inputs(synth.inputs(w, "accel"), "accel")
    O = torch.zeros(w.shape, device="cuda")
    LSE = torch.zeros(w.shape[:3], device="cuda")
    mg.mg_attn_fwd(dev["Q"], dev["K"], dev["V"], O, LSE, True, w.scale, "accel")
    status = mg.mg_get_device_error()
    assert status == mg.MG_ERR_TIMEOUT, status
    assert mg.mg_get_device_error() == mg.MG_OK  # the word was cleared by the read

    # the context survived: a STRICT forward + backward still matches the oracle
    dev, vals = device_inputs(synth.inputs(w, "strict"), "strict")
    got = run_gpu(dev, True, w.scale, "strict")
    ref = oracle.attn_bwd(vals["Q"], vals["K"], vals["V"], vals["dO"], True, w.scale)
    errs, bad = compare(got, ref, "strict")
    assert not bad, errs
    print("FAULT-INJECTION-OK")
""")


def test_bounded_wait_times_out_and_context_survives():
    env = dict(os.environ, MG_FAULT_INJECT="skip_k_tile", MG_WAIT_TIMEOUT_MS="200")
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "FAULT-INJECTION-OK" in res.stdout
