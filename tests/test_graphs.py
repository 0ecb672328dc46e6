"""The library's calls captured in CUDA graphs (the launch-free form of a
decode loop or a training step) and replayed: every call only enqueues work
on the caller's stream, with caller-provided buffers, so a captured sequence
replays to the results of the same calls made directly.

  * a token through 8 layers of decode steps, each layer with its own state:
    the replayed states and outputs equal the direct calls bit for bit;
  * the forward (FUSED and TWOPASS, each with its own workspace): bit for bit;
  * the training pair (forward with checkpoints, backward from them): the
    gradients within the backward's float32 tolerance (its float32 atomic
    sums may add in another order), and the oracle's gradients too.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import synth

from test_parity_bwd import _compare, _dy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_02_gb300 import build
    build.build()
    oracle.build()


def _capture(fn):
    """Warm up on a side stream (first calls set kernel attributes), capture
    fn into a graph, return it."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_layers_in_a_graph():
    layers = 8
    p = synth.make_problem(16, 256, 16, 1, dtype="bf16", gate=True, seed=900)
    ins = [{k: (v.cuda() if v is not None else None) for k, v in synth.step_inputs(p, 0).items()}
           for _ in range(layers)]
    h0 = [synth.make_state(16, 256, 16, seed=901 + i).cuda() for i in range(layers)]
    states = [h.clone() for h in h0]
    ys = [torch.empty_like(ins[0]["x"]) for _ in range(layers)]

    def token():
        for i in range(layers):
            c = ins[i]
            ssm.scan_step(states[i], c["x"], c["delta"], c["A"], c["B"], c["C"], D=c["D"], z=c["z"],
                          dt_bias=c["dt_bias"], delta_softplus=p.delta_softplus, y=ys[i])

    g = _capture(token)                    # the warm-up ran one token
    for i in range(layers):
        states[i].copy_(h0[i])
    for _ in range(3):                     # three tokens replayed
        g.replay()
    torch.cuda.synchronize()
    got_s = [s.clone() for s in states]
    got_y = [y.clone() for y in ys]
    for i in range(layers):                # the same three tokens called directly
        states[i].copy_(h0[i])
    for _ in range(3):
        token()
    torch.cuda.synchronize()
    for i in range(layers):
        assert torch.equal(got_s[i], states[i]) and torch.equal(got_y[i], ys[i]), f"layer {i}"


@pytest.mark.parametrize("variant", ["fused", "twopass"])
def test_forward_in_a_graph(variant):
    p = synth.make_problem(2, 64, 16, 700, dtype="bf16", gate=True, seed=902)
    t = {k: (getattr(p, k).cuda() if getattr(p, k) is not None else None)
         for k in ("x", "delta", "A", "B", "C", "D", "z", "dt_bias")}
    ws = torch.empty(max(ssm.workspace_size(2, 64, 16, 700, torch.bfloat16, variant), 1), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty_like(t["x"])
    fs = torch.empty(2, 64, 16, device="cuda")

    def fwd():
        ssm.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"], dt_bias=t["dt_bias"],
                     return_final_state=True, variant=variant, y=y, final_state=fs, workspace=ws)

    g = _capture(fwd)
    y.zero_()
    fs.zero_()
    g.replay()
    torch.cuda.synchronize()
    gy, gfs = y.clone(), fs.clone()
    fwd()
    torch.cuda.synchronize()
    assert torch.equal(gy, y) and torch.equal(gfs, fs)


def test_training_pair_in_a_graph():
    p = synth.make_problem(2, 48, 16, 300, dtype="f32", gate=True, seed=903, A_mode="random")
    t = {k: (getattr(p, k).cuda() if getattr(p, k) is not None else None)
         for k in ("x", "delta", "A", "B", "C", "D", "z", "dt_bias")}
    dy = _dy(p, 26).cuda()
    out = {}

    def step():
        _, ck = ssm.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"], dt_bias=t["dt_bias"],
                             return_ckpt=True)
        out["g"] = ssm.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], dy, D=t["D"], z=t["z"],
                                dt_bias=t["dt_bias"], ckpt=ck)

    g = _capture(step)
    for v in out["g"].values():
        if v is not None:
            v.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.bwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"), dy.cpu().numpy(),
                     D=p.D.numpy(), z=p.f32("z"), dt_bias=p.dt_bias.numpy())
    _compare(out["g"], ref, "f32")
