"""GPU parity of the convolution + scan call (ssm_scan_fwd_conv) against the
fp64 oracle chain: the oracle's causal depthwise convolution with SiLU, its
output fed as x to the oracle's serial forward recurrence.  Element by
element with the forward's tolerances (|y - ref| <= 1e-4 (1 + |ref|) for
float32 I/O, 2e-2 (1 + |ref|) for bf16; the final state at the float32
bound).

The fused mode keeps the convolution's output in float32; the separate mode
writes it in the I/O dtype first, so with bf16 I/O every scan input x carries
one more rounding (relative 2^-9).  Both are held to the unrounded oracle
chain, not to each other; for the separate mode with bf16 I/O the final state,
which sums those rounded inputs, is therefore held to the bf16 bound.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import synth

from test_parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_02_gb300 import build
    build.build()
    oracle.build()


def _reference(p, w, cb, state):
    xc, _ = oracle.conv1d(p.f32("x"), w.numpy(), None if cb is None else cb.numpy(),
                          None if state is None else state.float().numpy(), silu=True)
    return oracle.fwd(xc.astype(np.float32), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
                      None if p.D is None else p.D.numpy(), p.f32("z"),
                      None if p.dt_bias is None else p.dt_bias.numpy(), p.delta_softplus)


def _run(p, w, cb, state, mode, x=None):
    g = lambda t: None if t is None else t.cuda()
    y, fs = ssm.scan_fwd_conv(g(p.x) if x is None else x, g(w), g(p.delta), g(p.A), g(p.B), g(p.C),
                              conv_bias=g(cb), conv_state=g(state), D=g(p.D), z=g(p.z), dt_bias=g(p.dt_bias),
                              delta_softplus=p.delta_softplus, return_final_state=True, mode=mode)
    torch.cuda.synchronize()
    return y.float().cpu().numpy(), fs.cpu().numpy()


def _check(p, w, cb, state, mode, what, x=None):
    yg, fg = _run(p, w, cb, state, mode, x)
    yr, fr = _reference(p, w, cb, state)
    nch = p.batch * p.dim
    assert_close(yg.reshape(nch, p.seqlen), yr, p.dtype, f"y[{what}]")
    rounded_x = p.dtype == "bf16" and mode != "fused"
    assert_close(fg.reshape(nch, p.dstate), fr, "bf16" if rounded_x else "f32", f"final_state[{what}]")
    return yg.reshape(nch, p.seqlen), yr


CASES = [
    # batch, dim, dstate, L, dtype, gate, width, with history
    (2, 40, 16, 300, "f32", True, 4, True),      # ragged tiles and channel blocks
    (1, 37, 16, 333, "f32", False, 3, False),    # rows not 16-byte aligned: element loads
    (3, 50, 16, 1000, "bf16", True, 4, True),    # several tiles, bf16
    (1, 20, 64, 300, "bf16", True, 2, True),     # 64 states: 16-step tiles
    (2, 9, 5, 130, "f32", False, 1, False),      # one tap, odd dstate
    (1, 33, 32, 2100, "f32", True, 4, False),    # 32 states, many tiles
]


@pytest.mark.parametrize("mode", ["fused", "separate"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:4])) + f"-{c[4]}-g{int(c[5])}-k{c[6]}"
                         + ("-h" if c[7] else ""))
def test_conv_scan_matches_oracle(case, mode):
    b, d, n, L, dt, gate, k, hist = case
    p = synth.make_problem(b, d, n, L, dtype=dt, gate=gate, seed=700 + d + n + L, A_mode="random")
    w, cb = synth.make_conv(d, k, seed=701 + k)
    state = synth.make_conv_state(b, d, k, dtype=dt, seed=702) if hist else None
    _check(p, w, cb, state, mode, f"{mode}")


def test_wide_filters_run_separately():
    """More than four taps: the separate mode (and AUTO) runs them; the fused
    mode refuses the width before launching anything."""
    p = synth.make_problem(2, 24, 16, 200, dtype="f32", gate=True, seed=710)
    w, cb = synth.make_conv(24, 7, seed=711)
    state = synth.make_conv_state(2, 24, 7, dtype="f32", seed=712)
    _check(p, w, cb, state, "separate", "separate k=7")
    _check(p, w, cb, state, "auto", "auto k=7")
    with pytest.raises(ssm.ScanError):
        _run(p, w, cb, state, "fused")


def test_scan_only_rms_with_convolution():
    """No skip and no gate: y is the state contraction of the convolved input
    alone; its relative RMS error stays within 1e-3 (float32) and 3e-2 (bf16)
    in both modes."""
    for dt, tol in (("f32", 1e-3), ("bf16", 3e-2)):
        p = synth.make_problem(2, 48, 16, 700, dtype=dt, gate=False, use_D=False, seed=713)
        w, cb = synth.make_conv(48, 4, seed=714)
        for mode in ("fused", "separate"):
            yg, yr = _check(p, w, cb, None, mode, f"scan-only {mode} {dt}")
            rel = np.sqrt(np.mean((yg - yr) ** 2)) / np.sqrt(np.mean(yr ** 2))
            assert rel <= tol, (mode, dt, rel)


def test_mid_workload_all_elements():
    """The mid-size workload's shape (4 x 1536 x 16, 2048 steps, bf16, gate
    on) with a 4-tap filter and a history, in the AUTO mode (fused at this
    size): every element against the oracle chain."""
    p = synth.workload("mid_bf16")
    assert ssm.select_variant(p.batch, p.dim, p.dstate, p.seqlen, p.torch_dtype) == "fused"
    w, cb = synth.make_conv(p.dim, 4, seed=715)
    state = synth.make_conv_state(p.batch, p.dim, 4, dtype="bf16", seed=716)
    assert ssm.conv_scan_workspace_size(p.batch, p.dim, p.dstate, p.seqlen, 4, p.torch_dtype, "auto") == \
        ssm.conv_scan_workspace_size(p.batch, p.dim, p.dstate, p.seqlen, 4, p.torch_dtype, "fused")
    _check(p, w, cb, state, "auto", "mid auto")


def test_second_segment_with_history():
    """A sequence split in two: the second segment's convolution needs the
    last K-1 raw inputs of the first as its history (conv_state).  With them,
    the call on the second segment (its scan from a zero state) matches the
    oracle chain given the same history."""
    p = synth.make_problem(1, 64, 16, 512, dtype="f32", gate=True, seed=717)
    w, cb = synth.make_conv(64, 4, seed=718)
    hist = p.x[:, :, 253:256].contiguous()
    q = synth.make_problem(1, 64, 16, 256, dtype="f32", gate=True, seed=717)
    q.x = p.x[:, :, 256:].contiguous()
    for name in ("delta", "z", "B", "C"):
        setattr(q, name, getattr(p, name)[:, :, 256:].contiguous())
    _check(q, w, cb, hist, "fused", "second segment")


def test_conv_workspace_sizes():
    fused = ssm.conv_scan_workspace_size(4, 1536, 16, 2048, 4, torch.bfloat16, "fused")
    assert fused == ssm.workspace_size(4, 1536, 16, 2048, torch.bfloat16, "fused")
    sep = ssm.conv_scan_workspace_size(4, 1536, 16, 2048, 4, torch.bfloat16, "separate")
    xc = (4 * 1536 * 2048 * 2 + 255) // 256 * 256
    assert sep == xc + ssm.workspace_size(4, 1536, 16, 2048, torch.bfloat16, "auto")
