"""GPU parity of the causal depthwise convolution (ssm_conv1d_fwd) against the
fp64 oracle, element by element, with the forward's tolerances
(|y - ref| <= 1e-4 (1 + |ref|) for float32 I/O, 2e-2 (1 + |ref|) for bf16);
the state handed to the next segment is a copy of inputs and must match
exactly.
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


def _x(batch, dim, L, dtype, seed):
    t = torch.from_numpy(np.random.default_rng(seed).standard_normal((batch, dim, L)).astype(np.float32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def _run(x, w, b, state, silu):
    y, st = ssm.conv1d(x.cuda(), w.cuda(), None if b is None else b.cuda(),
                       state_in=None if state is None else state.cuda(), silu=silu, return_state=True)
    torch.cuda.synchronize()
    yr, sr = oracle.conv1d(x.float().numpy(), w.numpy(), None if b is None else b.numpy(),
                           None if state is None else state.float().numpy(), silu=silu)
    return y, st, yr, sr


@pytest.mark.parametrize("batch,dim,L,width,dtype,silu,hist", [
    (2, 37, 64, 4, "bf16", True, True),      # vector path, history in
    (1, 16, 77, 4, "f32", True, False),      # ragged tail: element path
    (3, 5, 3, 4, "f32", False, True),        # shorter than the history
    (2, 9, 40, 1, "bf16", True, False),      # one tap
    (2, 11, 48, 2, "f32", True, True),
    (1, 7, 35, 7, "bf16", False, True),      # seven taps, odd length
    (2, 8, 16, 8, "f32", True, True),
])
def test_conv_matches_oracle(batch, dim, L, width, dtype, silu, hist):
    x = _x(batch, dim, L, dtype, seed=500 + L + width)
    w, b = synth.make_conv(dim, width, seed=501 + width)
    state = synth.make_conv_state(batch, dim, width, dtype, seed=502) if hist else None
    y, st, yr, sr = _run(x, w, b, state, silu)
    assert_close(y.float().cpu().numpy(), yr, dtype, "y")
    if width > 1:
        assert np.array_equal(st.float().cpu().numpy().astype(np.float64), sr), "state_out"


def test_segments_continue():
    """Two calls over consecutive segments, the state of the first starting
    the second, give the oracle's output over the whole sequence."""
    x = _x(2, 24, 100, "f32", seed=510)
    w, b = synth.make_conv(24, 4, seed=511)
    yr, sr = oracle.conv1d(x.numpy(), w.numpy(), b.numpy())
    y1, s1 = ssm.conv1d(x[..., :37].contiguous().cuda(), w.cuda(), b.cuda(), return_state=True)
    y2, s2 = ssm.conv1d(x[..., 37:].contiguous().cuda(), w.cuda(), b.cuda(), state_in=s1, return_state=True)
    torch.cuda.synchronize()
    assert_close(torch.cat([y1, y2], dim=-1).cpu().numpy(), yr, "f32", "y (segments)")
    assert np.array_equal(s2.cpu().numpy().astype(np.float64), sr)


def test_empty_sequence_passes_the_history_through():
    x = torch.empty(2, 4, 0).cuda()
    w, b = synth.make_conv(4, 4, seed=512)
    state = synth.make_conv_state(2, 4, 4, seed=513).cuda()
    y, st = ssm.conv1d(x, w.cuda(), b.cuda(), state_in=state, return_state=True)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.equal(st, state)


def test_mid_size_shape():
    """The mid-size shape (4 x 1536 x 2048, bf16, 4 taps), every output."""
    x = _x(4, 1536, 2048, "bf16", seed=514)
    w, b = synth.make_conv(1536, 4, seed=515)
    y, st, yr, sr = _run(x, w, b, None, True)
    assert_close(y.float().cpu().numpy(), yr, "bf16", "y (mid)")
    assert np.array_equal(st.float().cpu().numpy().astype(np.float64), sr)
