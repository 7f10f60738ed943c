"""The hi/lo derivative-precision policy (MG_DS_HILO) of the accelerated backward.

"Meganeura: Portable GPU Training and Inference through Vulkan and Metal",
Section 3.1, attaches a precision bit to derivative regions so that the 16-bit
matrix promotion does not round small gradient operands. Here the policy splits
dS into hi = round16(dS) and lo = round16(dS - hi) and accumulates both products
for dK and dQ. Parity at the ACCEL gate is covered with the other precision
variants; this file checks what the split is for: with the exact O and LSE fed
to the backward (so that nothing upstream of dS carries a 16-bit rounding), the
dK and dQ errors against the fp64 oracle shrink by far more than the gate's
margin, while dV, whose operand P is not split, does not change materially."""
import numpy as np
import pytest

import attention_forward_backward_gb300 as mg
import oracle
from attention_forward_backward_gb300 import synth
from parity_util import device_inputs, rel_err

pytestmark = pytest.mark.gpu


def _bwd_from_exact_forward(w, contract, ref, dev):
    """Backward only, from the oracle's O (as f32) and LSE."""
    import torch
    O = torch.from_numpy(ref["O"].astype(np.float32)).cuda()
    LSE = torch.from_numpy(ref["LSE"].astype(np.float32)).cuda()
    dQ, dK, dV = mg.attention_bwd(dev["Q"], dev["K"], dev["V"], O, dev["dO"], LSE, w.causal,
                                  w.scale, contract)
    torch.cuda.synchronize()
    assert mg.mg_get_device_error() == mg.MG_OK
    return {"dQ": dQ.float().cpu().numpy(), "dK": dK.float().cpu().numpy(),
            "dV": dV.float().cpu().numpy()}


@pytest.mark.parametrize("cfg", [2, 4])
def test_hilo_shrinks_the_ds_rounding_error(cfg):
    w = synth.WORKLOADS[cfg]
    dev, vals = device_inputs(synth.inputs(w, "accel"), "accel")
    ref = oracle.attn_bwd(vals["Q"], vals["K"], vals["V"], vals["dO"], w.causal, w.scale)
    plain = _bwd_from_exact_forward(w, "accel", ref, dev)
    split = _bwd_from_exact_forward(w, "accel+hilo", ref, dev)
    e_plain = {k: rel_err(plain[k], ref[k]) for k in plain}
    e_split = {k: rel_err(split[k], ref[k]) for k in split}
    # one bf16 rounding of dS (relative 2^-9) against two (2^-17): the products
    # that take dS must come out at least 8x closer to the oracle
    for k in ("dQ", "dK"):
        assert e_split[k] * 8 <= e_plain[k], (k, e_plain, e_split)
    # dV's operand P is rounded the same way under both policies
    assert e_split["dV"] <= 2 * e_plain["dV"], (e_plain, e_split)


def test_hilo_runs_the_two_pass_backward():
    """The split needs both dS parts as tensor-memory operands of the dK and dQ
    products: the backward launches the dK/dV kernel and the dQ pass, not the
    fused kernel with dQ reductions."""
    import torch
    w = synth.custom_workload(1, 2, 300, 128, True, seed_cfg=1350)
    dev, _ = device_inputs(synth.inputs(w, "accel"), "accel")
    O, LSE = mg.attention_fwd(dev["Q"], dev["K"], dev["V"], True, w.scale, "accel+hilo")
    names = [mg.mg_attn_kernel_name(i) for i in range(mg.mg_attn_kernel_count())]
    mg.mg_attn_profile_enable(True, 64)
    try:
        mg.attention_bwd(dev["Q"], dev["K"], dev["V"], O, dev["dO"], LSE, True, w.scale,
                         "accel+hilo")
        torch.cuda.synchronize()
        launched = {names[i] for i in range(len(names)) if mg.mg_attn_profile_read(i)[0] > 0}
    finally:
        mg.mg_attn_profile_enable(False)
    assert launched == {"accel_dvec", "accel_dkdv", "accel_dq"}, launched
