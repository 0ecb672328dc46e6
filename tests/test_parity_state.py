"""GPU parity of the start-state forward and the single-token decode step
against the fp64 oracle (ssm_oracle_fwd_from, ssm_oracle_step), with the
forward's tolerances: |got - ref| <= 1e-4 (1 + |ref|) for float32 I/O and for
every state, 2e-2 (1 + |ref|) for bf16 y.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import synth

from test_parity import assert_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_02_gb300 import build
    build.build()
    oracle.build()


def _oracle_from(p, h0):
    y, fs = oracle.fwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
                       None if p.D is None else p.D.numpy(), p.f32("z"),
                       None if p.dt_bias is None else p.dt_bias.numpy(), p.delta_softplus,
                       h0=h0.numpy().astype(np.float64))
    return y.reshape(p.batch, p.dim, p.seqlen), fs.reshape(p.batch, p.dim, p.dstate)


def _gpu_from(p, h0, variant, in_place=False):
    t = to_dev(p)
    s = h0.cuda()
    fs = s if in_place else torch.empty_like(s)
    y, fs = ssm.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"], dt_bias=t["dt_bias"],
                         delta_softplus=p.delta_softplus, return_final_state=True, variant=variant,
                         initial_state=s, final_state=fs)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), fs.cpu().numpy()


@pytest.mark.parametrize("variant", ["fused", "twopass", "chunked"])
@pytest.mark.parametrize("shape,dtype,gate", [
    ((2, 37, 16, 300), "f32", True),
    ((1, 70, 5, 515), "bf16", False),
    ((3, 33, 64, 129), "bf16", True),
])
def test_start_state_matches_oracle(variant, shape, dtype, gate):
    seed = 200 + 10 * ["fused", "twopass", "chunked"].index(variant) + shape[2]
    p = synth.make_problem(*shape, dtype=dtype, gate=gate, seed=seed, A_mode="random")
    h0 = synth.make_state(*shape[:3], seed=7)
    y, fs = _gpu_from(p, h0, variant)
    yr, fr = _oracle_from(p, h0)
    assert_close(y, yr, dtype, f"y[{variant}]")
    assert_close(fs, fr, "f32", f"final_state[{variant}]")


@pytest.mark.parametrize("variant", ["fused", "twopass", "chunked"])
def test_resume_in_place_equals_one_pass(variant):
    """Three consecutive segments, the state advanced in place, against the
    oracle over the whole sequence."""
    p = synth.make_problem(2, 48, 16, 1000, dtype="f32", gate=True, seed=211)
    h0 = synth.make_state(2, 48, 16, seed=8)
    yr, fr = _oracle_from(p, h0)
    t = to_dev(p)
    state = h0.cuda()
    ys = []
    for a, b in ((0, 1), (1, 512), (512, 1000)):
        cut = lambda v: None if v is None else v[:, :, a:b].contiguous()
        y, _ = ssm.scan_fwd(cut(t["x"]), cut(t["delta"]), t["A"], cut(t["B"]), cut(t["C"]), D=t["D"],
                            z=cut(t["z"]), dt_bias=t["dt_bias"], return_final_state=True, variant=variant,
                            initial_state=state, final_state=state)
        ys.append(y)
    torch.cuda.synchronize()
    assert_close(torch.cat(ys, dim=2).cpu().numpy(), yr, "f32", "y (resumed)")
    assert_close(state.cpu().numpy(), fr, "f32", "state (resumed)")


def test_empty_sequence_keeps_the_start_state():
    p = synth.make_problem(2, 8, 16, 0, dtype="f32", seed=212)
    h0 = synth.make_state(2, 8, 16, seed=9).cuda()
    t = to_dev(p)
    _, fs = ssm.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], return_final_state=True, initial_state=h0)
    torch.cuda.synchronize()
    assert torch.equal(fs, h0)


def _oracle_steps(p, h0, T):
    h = h0.numpy().astype(np.float64)
    ys = []
    for t in range(T):
        s = synth.step_inputs(p, t)
        f = lambda v: None if v is None else v.float().numpy()
        h, y = oracle.step(h, f(s["x"]), f(s["delta"]), p.A.numpy(), f(s["B"]), f(s["C"]),
                           None if p.D is None else p.D.numpy(), f(s["z"]),
                           None if p.dt_bias is None else p.dt_bias.numpy(), p.delta_softplus)
        ys.append(y)
    return np.stack(ys, axis=-1), h


@pytest.mark.parametrize("batch,dim,dstate,dtype,gate", [
    (3, 45, 16, "f32", True),     # 4 lanes per channel, 16-byte state rows
    (2, 33, 5, "bf16", False),    # ragged state: element path
    (1, 17, 1, "f32", True),      # one state
    (2, 19, 64, "bf16", True),    # 16 lanes per channel
    (4, 7, 12, "f32", False),     # a lane without states
])
def test_step_matches_oracle(batch, dim, dstate, dtype, gate):
    T = 6
    p = synth.make_problem(batch, dim, dstate, T, dtype=dtype, gate=gate, seed=300 + dstate, A_mode="random")
    h0 = synth.make_state(batch, dim, dstate, seed=10)
    yr, hr = _oracle_steps(p, h0, T)
    state = h0.cuda()
    ys = []
    for t in range(T):
        s = {k: (v.cuda() if v is not None else None) for k, v in synth.step_inputs(p, t).items()}
        ys.append(ssm.scan_step(state, s["x"], s["delta"], s["A"], s["B"], s["C"], D=s["D"], z=s["z"],
                                dt_bias=s["dt_bias"]))
    torch.cuda.synchronize()
    assert_close(torch.stack(ys, dim=-1).float().cpu().numpy(), yr, dtype, "y (steps)")
    assert_close(state.cpu().numpy(), hr, "f32", "state (steps)")


def test_steps_continue_a_forward():
    """A forward over the prompt, then decode steps from its final state: the
    same result as the oracle over prompt and tokens together."""
    p = synth.make_problem(2, 64, 16, 200, dtype="bf16", gate=True, seed=213)
    t = to_dev(p)
    n_prompt = 190
    cut = lambda v: None if v is None else v[:, :, :n_prompt].contiguous()
    _, state = ssm.scan_fwd(cut(t["x"]), cut(t["delta"]), t["A"], cut(t["B"]), cut(t["C"]), D=t["D"],
                            z=cut(t["z"]), dt_bias=t["dt_bias"], return_final_state=True)
    ys = []
    for k in range(n_prompt, p.seqlen):
        s = {kk: (v.cuda() if v is not None else None) for kk, v in synth.step_inputs(p, k).items()}
        ys.append(ssm.scan_step(state, s["x"], s["delta"], s["A"], s["B"], s["C"], D=s["D"], z=s["z"],
                                dt_bias=s["dt_bias"]))
    torch.cuda.synchronize()
    yr, fr = oracle.fwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"), p.D.numpy(),
                        p.f32("z"), p.dt_bias.numpy(), True)
    yr = yr.reshape(p.batch, p.dim, p.seqlen)[:, :, n_prompt:]
    assert_close(torch.stack(ys, dim=-1).float().cpu().numpy(), yr, "bf16", "y (decode)")
    assert_close(state.cpu().numpy(), fr.reshape(p.batch, p.dim, p.dstate), "f32", "state (decode)")


def test_step_at_serving_size():
    """The benchmark's decode shape (256 sequences x 2048 channels x 16
    states, bf16), one step, every output against the oracle."""
    p = synth.make_problem(256, 2048, 16, 1, dtype="bf16", gate=True, seed=214)
    h0 = synth.make_state(256, 2048, 16, seed=11)
    yr, hr = _oracle_steps(p, h0, 1)
    s = {k: (v.cuda() if v is not None else None) for k, v in synth.step_inputs(p, 0).items()}
    state = h0.cuda()
    y = ssm.scan_step(state, s["x"], s["delta"], s["A"], s["B"], s["C"], D=s["D"], z=s["z"], dt_bias=s["dt_bias"])
    torch.cuda.synchronize()
    assert_close(y.float().cpu().numpy(), yr[..., 0], "bf16", "y (serving step)")
    assert_close(state.cpu().numpy(), hr, "f32", "state (serving step)")
