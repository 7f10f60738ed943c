"""Precision variants of the accelerated contract against the fp64 oracle, element
by element at the ACCEL gate (2e-2, max-abs error over max-abs reference):

* ACCEL_F16 ("accel_f16"): f16 Q, K, V, dO, with P and dS rounded to f16 as MMA
  operands; the pages' own accelerated format ("Meganeura: Portable GPU Training
  and Inference through Vulkan and Metal", Section 4.2);
* MG_OUT_16 ("+out16"): O, dQ, dK, dV stored in the inputs' 16-bit type;
* MG_DS_HILO ("+hilo"): the backward's derivative-precision policy, dS split
  into a 16-bit hi and lo part (Section 3.1's precision bit on derivative
  regions), with bf16 and with f16 inputs and 16-bit outputs.

The oracle consumes the 16-bit-rounded inputs exactly, so only the kernels' own
arithmetic and the final rounding of 16-bit outputs are measured. Covered: the
decoder, encoder and large-logit workloads in full, the long-sequence workload on
two whole heads and sampled rows, ragged and sub-tile lengths for every head dim,
cross attention with key padding, both ACCEL backward modes, and the decode
forward with f16 inputs."""
import numpy as np
import pytest

import attention_forward_backward_gb300 as mg
import oracle
from attention_forward_backward_gb300 import synth
from parity_util import TOL, compare, compare_ex, device_inputs, run_gpu, run_gpu_decode

pytestmark = pytest.mark.gpu

VARIANTS = ["accel_f16", "accel+out16", "accel_f16+out16", "accel+hilo", "accel_f16+hilo+out16"]


def _full(w, contract, bwd=True):
    dev, vals = device_inputs(synth.inputs(w, contract), contract)
    got = run_gpu(dev, w.causal, w.scale, contract, bwd=bwd)
    ref = oracle.attn_bwd(vals["Q"], vals["K"], vals["V"], vals["dO"], w.causal, w.scale)
    if not bwd:
        ref = {"O": ref["O"], "LSE": ref["LSE"]}
    errs, bad = compare(got, ref, contract)
    assert not bad, (w.name, contract, errs)
    return got


@pytest.mark.parametrize("contract", VARIANTS)
@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_variant_configs(cfg, contract):
    _full(synth.WORKLOADS[cfg], contract)


@pytest.mark.parametrize("contract", VARIANTS)
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("L", [1, 65, 300])
@pytest.mark.parametrize("causal", [True, False])
def test_variant_edge_shapes(D, L, causal, contract):
    _full(synth.custom_workload(1, 2, L, D, causal, seed_cfg=1300 + D), contract)


@pytest.mark.parametrize("contract", VARIANTS)
def test_variant_long_sequence_sampled(contract):
    """B=2 H=32 L=8192 D=128 causal: two heads in full, every seventh head on
    sampled query rows (O and LSE)."""
    w = synth.WORKLOADS[5]
    host = synth.inputs(w, contract)
    dev, vals = device_inputs(host, contract)
    got = run_gpu(dev, w.causal, w.scale, contract, bwd=True)
    BH = w.B * w.H
    flat = {k: v.reshape(BH, w.L, -1) if v.ndim == 4 else v.reshape(BH, w.L)
            for k, v in got.items()}
    vflat = {k: v.reshape(BH, w.L, w.D) for k, v in vals.items()}
    for h in (1, BH - 2):
        ref = oracle.attn_bwd(vflat["Q"][h], vflat["K"][h], vflat["V"][h], vflat["dO"][h],
                              True, w.scale)
        errs, bad = compare({k: flat[k][h] for k in ("O", "LSE", "dQ", "dK", "dV")}, ref,
                            contract)
        assert not bad, (h, errs)
    rows = np.array([0, 1, 127, 128, 4095, 8191])
    for h in range(0, BH, 7):
        O, LSE = oracle.attn_fwd_rows(vflat["Q"][h], vflat["K"][h], vflat["V"][h], rows, True,
                                      w.scale)
        errs, bad = compare({"O": flat["O"][h][rows], "LSE": flat["LSE"][h][rows]},
                            {"O": O, "LSE": LSE}, contract)
        assert not bad, (h, errs)


@pytest.mark.parametrize("contract", VARIANTS)
def test_variant_outputs_have_the_requested_type(contract):
    import torch
    w = synth.custom_workload(1, 2, 130, 64, True, seed_cfg=1310)
    dev, _ = device_inputs(synth.inputs(w, contract), contract)
    O, LSE = mg.attention_fwd(dev["Q"], dev["K"], dev["V"], True, w.scale, contract)
    dQ, dK, dV = mg.attention_bwd(dev["Q"], dev["K"], dev["V"], O, dev["dO"], LSE, True,
                                  w.scale, contract)
    torch.cuda.synchronize()
    want = mg._out_dtype(contract)
    assert O.dtype == dQ.dtype == dK.dtype == dV.dtype == want and LSE.dtype == torch.float32


@pytest.mark.parametrize("contract", VARIANTS)
def test_variant_cross_attention_with_padding(contract):
    """Lq != Lk, bottom-right causal, per-batch key padding (lengths 0, 77, full)."""
    import torch
    B, H, Lq, Lk, D = 3, 2, 150, 200, 64
    kv_len = [0, 77, 200]
    host = synth.cross_inputs(B, H, Lq, Lk, D, contract, seed_cfg=1320)
    dev, vals = device_inputs(host, contract)
    scale = D ** -0.5
    odt = mg._out_dtype(contract)
    lens = torch.tensor(kv_len, dtype=torch.int32, device="cuda")
    O = torch.full((B, H, Lq, D), float("nan"), device="cuda", dtype=odt)
    LSE = torch.full((B, H, Lq), float("nan"), device="cuda")
    mg.mg_attn_fwd_padded(dev["Q"], dev["K"], dev["V"], O, LSE, lens, "causal_bottom_right",
                          scale, contract)
    dQ = torch.full((B, H, Lq, D), float("nan"), device="cuda", dtype=odt)
    dK = torch.full((B, H, Lk, D), float("nan"), device="cuda", dtype=odt)
    dV = torch.full_like(dK, float("nan"))
    ws = torch.empty(mg.mg_attn_bwd_workspace_bytes_ex(B, H, Lq, Lk, D, contract),
                     dtype=torch.uint8, device="cuda")
    mg.mg_attn_bwd_padded(dev["Q"], dev["K"], dev["V"], O, dev["dO"], LSE, dQ, dK, dV, lens,
                          "causal_bottom_right", scale, contract, ws)
    torch.cuda.synchronize()
    assert mg.mg_get_device_error() == mg.MG_OK
    got = {k: v.float().cpu().numpy() for k, v in dict(O=O, LSE=LSE, dQ=dQ, dK=dK, dV=dV).items()}
    ref = oracle.attn_bwd_padded(vals["Q"], vals["K"], vals["V"], vals["dO"], kv_len,
                                 "causal_bottom_right", scale)
    errs, bad = compare_ex(got, ref, contract)
    assert not bad, errs


def test_decode_with_f16_inputs():
    host = synth.cross_inputs(2, 4, 5, 3000, 128, "accel_f16", seed_cfg=1330)
    dev, vals = device_inputs(host, "accel_f16")
    scale = 128 ** -0.5
    got = run_gpu_decode(dev, "causal_bottom_right", scale, "accel_f16")
    O, LSE = oracle.attn_fwd_ex(vals["Q"], vals["K"], vals["V"], "causal_bottom_right", scale)
    errs, bad = compare_ex(got, {"O": O, "LSE": LSE}, "accel_f16")
    assert not bad, errs


def test_variants_two_pass_backward_in_child():
    """The two-pass ACCEL backward (MG_DQ_MODE=pass: its dQ pass stores dQ in the
    output type directly) for every variant, in a child process."""
    import os
    import subprocess
    import sys
    import textwrap
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {root!r}); sys.path.insert(0, {os.path.join(root, 'tests')!r})
        from attention_forward_backward_gb300 import synth
        from test_precision_variants import _full, VARIANTS
        for c in VARIANTS:
            for w in (synth.WORKLOADS[2], synth.custom_workload(1, 3, 300, 128, True, seed_cfg=1340),
                      synth.custom_workload(2, 2, 197, 64, False, seed_cfg=1341)):
                _full(w, c)
        print("VARIANT-PASS-OK")
    """)
    env = dict(os.environ, MG_DQ_MODE="pass")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "VARIANT-PASS-OK" in r.stdout, r.stdout + r.stderr
