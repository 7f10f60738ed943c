"""mg_attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (its Dvec scratch is a fixed array inside the library instead of a
caller workspace). Called through the C ABI and compared, twice in a row (so
that the shared array's leftover contents from the first call cannot leak into
the second), with mg_attn_bwd on the same inputs and with the fp64 oracle.
Collected last on purpose."""
import ctypes

import numpy as np
import pytest

import attention_forward_backward_gb300 as mg
import oracle
from attention_forward_backward_gb300 import synth
from parity_util import TOL, compare, device_inputs, rel_err

pytestmark = pytest.mark.gpu

MAX_ROWS = 1 << 20


def _lib():
    lib = mg.load_library()
    f = lib.mg_attn_bwd_noalloc
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, fl, i, vp]
    f.restype = i
    return lib


@pytest.mark.parametrize("contract", ["strict", "accel"])
def test_noalloc_matches_workspace_backward(contract):
    import torch
    lib = _lib()
    cases = [synth.custom_workload(2, 4, 300, 64, True, seed_cfg=870),
             synth.custom_workload(1, 3, 257, 128, False, seed_cfg=871)]
    stream = torch.cuda.current_stream().cuda_stream
    for w in cases:
        dev, vals = device_inputs(synth.inputs(w, contract), contract)
        B, H, L, D = w.shape
        O, LSE = mg.attention_fwd(dev["Q"], dev["K"], dev["V"], w.causal, w.scale, contract)
        ref = mg.attention_bwd(dev["Q"], dev["K"], dev["V"], O, dev["dO"], LSE, w.causal,
                               w.scale, contract)
        torch.cuda.synchronize()
        ref = [t.cpu().numpy() for t in ref]
        exact = oracle.attn_bwd(vals["Q"], vals["K"], vals["V"], vals["dO"], w.causal, w.scale)
        for _ in range(2):
            outs = [torch.full_like(O, float("nan")) for _ in range(3)]
            rc = lib.mg_attn_bwd_noalloc(
                dev["Q"].data_ptr(), dev["K"].data_ptr(), dev["V"].data_ptr(), O.data_ptr(),
                dev["dO"].data_ptr(), LSE.data_ptr(), outs[0].data_ptr(), outs[1].data_ptr(),
                outs[2].data_ptr(), B, H, L, D, int(w.causal), w.scale,
                mg.CONTRACTS[contract], stream)
            assert rc == mg.MG_OK, mg.mg_status_string(rc)
            torch.cuda.synchronize()
            assert mg.mg_get_device_error() == mg.MG_OK
            got = [t.cpu().numpy() for t in outs]
            for g, want in zip(got, ref):
                assert rel_err(g, want) <= TOL[contract]
            errs, bad = compare(dict(zip(("dQ", "dK", "dV"), got)), exact, contract,
                                keys=("dQ", "dK", "dV"))
            assert not bad, (w.name, errs)


def test_noalloc_rejects_beyond_the_fixed_scratch():
    lib = _lib()
    fake = 1 << 40  # never dereferenced: the size check comes first
    rc = lib.mg_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                 2, 1, MAX_ROWS // 2 + 1, 64, 1, 0.125, 0, None)
    assert rc == mg.MG_ERR_WORKSPACE
    rc = lib.mg_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, fake, fake,
                                 2, 32, 16385, 128, 1, 0.125, 1, None)
    assert rc == mg.MG_ERR_WORKSPACE


def test_noalloc_reports_argument_errors_before_the_size_limit():
    """A shape beyond the fixed array with an invalid head dim, mask flag or
    sequence length reports the same status as mg_attn_bwd, not MG_ERR_WORKSPACE."""
    lib = _lib()
    fake = 1 << 40  # never dereferenced: the argument checks come first
    args = [fake] * 9
    big = (2, 32, 16385)
    assert lib.mg_attn_bwd_noalloc(*args, *big, 96, 1, 0.125, 1, None) == mg.MG_ERR_UNSUPPORTED
    assert lib.mg_attn_bwd_noalloc(*args, *big, 128, 2, 0.125, 1, None) == mg.MG_ERR_INVALID_ARG
    assert lib.mg_attn_bwd_noalloc(*args, *big, 128, 1, 0.125, 7, None) == mg.MG_ERR_INVALID_ARG
    assert lib.mg_attn_bwd_noalloc(*args, 1, 1, (1 << 20) + 1, 64, 1, 0.125, 0,
                                   None) == mg.MG_ERR_INVALID_ARG
