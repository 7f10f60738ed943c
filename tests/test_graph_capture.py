"""The C-ABI calls inside a CUDA graph. Every call only enqueues work on the
caller's stream (no allocation, no synchronising call), so a sequence of calls
can be captured once and replayed, which is how a launch-bound sequence (the
convolution layer set, short attention steps) is best run. Each test captures a
step, poisons the outputs, replays the graph twice and compares with an eager
run of the same calls (bitwise where the kernels' order of additions is fixed)
and with the fp64 oracles."""
import numpy as np
import pytest

import attention_forward_backward_gb300 as mg
import oracle
from attention_forward_backward_gb300 import synth
from parity_util import compare, compare_ex, device_inputs, rel_err

pytestmark = pytest.mark.gpu


def _capture_and_replay(step, outs, stream):
    """Run `step` eagerly, then capture it, poison `outs`, replay twice; return
    the eager results (clones) and leave the replayed ones in `outs`."""
    import torch
    with torch.cuda.stream(stream):
        step()  # eager; also the library's one-time set-up, outside the capture
    torch.cuda.synchronize()
    assert mg.mg_get_device_error() == mg.MG_OK
    eager = {k: t.clone() for k, t in outs.items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    with torch.cuda.stream(stream):  # poison and replay in one stream order
        for t in outs.values():
            t.fill_(float("nan"))
        graph.replay()
        graph.replay()
    torch.cuda.synchronize()
    assert mg.mg_get_device_error() == mg.MG_OK
    return eager


@pytest.mark.parametrize("D", [64, 128])
def test_attention_step_replayed_from_a_graph(D):
    import torch
    w = synth.custom_workload(1, 3, 333, D, True, seed_cfg=880 + D)
    dev, vals = device_inputs(synth.inputs(w, "accel"), "accel")
    B, H, L, _ = w.shape
    s = torch.cuda.Stream()
    O = torch.empty((B, H, L, D), device="cuda")
    outs = {"O": O, "LSE": torch.empty((B, H, L), device="cuda"),
            "dQ": torch.empty_like(O), "dK": torch.empty_like(O), "dV": torch.empty_like(O)}
    ws = torch.empty(mg.mg_attn_bwd_workspace_bytes(B, H, L, D, "accel"), dtype=torch.uint8,
                     device="cuda")

    def step():
        mg.mg_attn_fwd(dev["Q"], dev["K"], dev["V"], outs["O"], outs["LSE"], w.causal, w.scale,
                       "accel", s.cuda_stream)
        mg.mg_attn_bwd(dev["Q"], dev["K"], dev["V"], outs["O"], dev["dO"], outs["LSE"],
                       outs["dQ"], outs["dK"], outs["dV"], w.causal, w.scale, "accel", ws,
                       s.cuda_stream)

    eager = _capture_and_replay(step, outs, s)
    # forward, dK and dV: one CTA owns each element, fixed order -> identical;
    # dQ: partial sums added by several CTAs -> compared within rounding
    for k in ("O", "LSE", "dK", "dV"):
        assert torch.equal(eager[k], outs[k]), k
    assert rel_err(outs["dQ"].cpu().numpy(), eager["dQ"].cpu().numpy()) <= 1e-5
    got = {k: t.cpu().numpy() for k, t in outs.items()}
    ref = oracle.attn_bwd(vals["Q"], vals["K"], vals["V"], vals["dO"], w.causal, w.scale)
    errs, bad = compare(got, ref, "accel")
    assert not bad, errs


def test_decode_replayed_from_a_graph():
    import torch
    B, H, Lq, Lk, D = 2, 4, 8, 3000, 128
    host = synth.cross_inputs(B, H, Lq, Lk, D, "accel", seed_cfg=884)
    host.pop("dO")
    dev, vals = device_inputs(host, "accel")
    scale = D ** -0.5
    s = torch.cuda.Stream()
    outs = {"O": torch.empty((B, H, Lq, D), device="cuda"),
            "LSE": torch.empty((B, H, Lq), device="cuda")}
    ws = torch.empty(mg.mg_attn_fwd_decode_workspace_bytes(B, H, Lq, Lk, D, "accel"),
                     dtype=torch.uint8, device="cuda")

    def step():
        mg.mg_attn_fwd_decode(dev["Q"], dev["K"], dev["V"], outs["O"], outs["LSE"],
                              "causal_bottom_right", scale, "accel", ws, s.cuda_stream)

    eager = _capture_and_replay(step, outs, s)
    for key in ("O", "LSE"):  # the merge adds the splits in a fixed order
        assert torch.equal(eager[key], outs[key]), key
    O, LSE = oracle.attn_fwd_ex(vals["Q"], vals["K"], vals["V"], "causal_bottom_right", scale)
    errs, bad = compare_ex({"O": outs["O"].cpu().numpy(), "LSE": outs["LSE"].cpu().numpy()},
                           {"O": O, "LSE": LSE}, "accel")
    assert not bad, errs


def test_convolution_pair_replayed_from_a_graph():
    import torch
    from oracle import conv as conv_oracle
    s = torch.cuda.Stream()
    for cw in (synth.custom_conv(2, 9, 9, 64, 72, 3, 3, 2, 1, cid=886),
               synth.custom_conv(2, 7, 7, 256, 64, 3, 3, 1, 1, cid=887)):
        ch = synth.conv_inputs(cw, "accel")
        cd = {k: torch.from_numpy(np.ascontiguousarray(v["bits"]).view(np.int16)).view(
            torch.bfloat16).cuda() for k, v in ch.items()}
        cv = {k: v["values"] for k, v in ch.items()}
        outs = {"dX": torch.empty((cw.N, cw.H, cw.W, cw.C), device="cuda"),
                "dW": torch.empty((cw.K, cw.R, cw.S, cw.C), device="cuda")}

        def step():
            mg.mg_conv2d_grad_input(cd["dY"], cd["Wt"], outs["dX"], cw.stride, cw.pad, "accel",
                                    s.cuda_stream)
            mg.mg_conv2d_grad_weight(cd["X"], cd["dY"], outs["dW"], cw.stride, cw.pad, "accel",
                                     s.cuda_stream)

        eager = _capture_and_replay(step, outs, s)
        for key in ("dX", "dW"):
            assert rel_err(outs[key].cpu().numpy(), eager[key].cpu().numpy()) <= 1e-5, key
        refs = {"dX": conv_oracle.conv2d_grad_input(cv["dY"], cv["Wt"], cw.H, cw.W, cw.stride,
                                                    cw.pad),
                "dW": conv_oracle.conv2d_grad_weight(cv["X"], cv["dY"], cw.R, cw.S, cw.stride,
                                                     cw.pad)}
        for key, ref in refs.items():
            assert rel_err(outs[key].cpu().numpy(), ref) <= 1e-3, (cw.name, key)
