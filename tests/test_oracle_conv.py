"""Pins of the oracle's causal depthwise convolution (no GPU).

Each channel's output before the gate is the causal part of a full linear
convolution with the reversed filter, which numpy.convolve computes
independently; special filters (a single tap at the newest input, at the
oldest) give the input itself and its delayed copy; the SiLU gate is checked
with scipy's expit; a sequence cut into two segments, the second started from
the state the first returns, gives the whole sequence's output exactly.
Planted mistakes in a copy of the source must fail these pins.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest
from scipy.special import expit

import oracle
from selective_state_space_02_gb300 import synth


def _x(batch, dim, L, seed):
    return np.random.default_rng(seed).standard_normal((batch, dim, L)).astype(np.float32)


@pytest.mark.parametrize("K", [1, 2, 4, 7])
def test_matches_numpy_convolve(K):
    x = _x(2, 5, 37, 1)
    w, b = (t.numpy() for t in synth.make_conv(5, K, seed=2))
    y, _ = oracle.conv1d(x, w, b, silu=False)
    for bb in range(2):
        for d in range(5):
            ref = np.convolve(x[bb, d].astype(np.float64), w[d, ::-1].astype(np.float64))[:37] + b[d]
            np.testing.assert_allclose(y[bb, d], ref, rtol=1e-13, atol=1e-13)


def test_newest_and_oldest_tap():
    x = _x(1, 3, 20, 3)
    w = np.zeros((3, 4), np.float32)
    w[:, 3] = 1.0
    y, _ = oracle.conv1d(x, w, None, silu=False)
    assert np.array_equal(y, x.astype(np.float64))
    w = np.zeros((3, 4), np.float32)
    w[:, 0] = 1.0
    y, _ = oracle.conv1d(x, w, None, silu=False)
    assert np.array_equal(y[..., 3:], x[..., :-3].astype(np.float64)) and not y[..., :3].any()


def test_gate():
    x = _x(2, 4, 15, 4)
    w, b = (t.numpy() for t in synth.make_conv(4, 4, seed=5))
    v, _ = oracle.conv1d(x, w, b, silu=False)
    y, _ = oracle.conv1d(x, w, b, silu=True)
    np.testing.assert_allclose(y, v * expit(v), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("cut", [0, 2, 10, 30])
def test_segments_continue_exactly(cut):
    x = _x(2, 3, 30, 6)
    w, b = (t.numpy() for t in synth.make_conv(3, 4, seed=7))
    s0 = synth.make_conv_state(2, 3, 4, seed=8).numpy()
    y, st = oracle.conv1d(x, w, b, state_in=s0)
    y1, st1 = oracle.conv1d(np.ascontiguousarray(x[..., :cut]), w, b, state_in=s0)
    y2, st2 = oracle.conv1d(np.ascontiguousarray(x[..., cut:]), w, b, state_in=st1.astype(np.float32))
    assert np.array_equal(np.concatenate([y1, y2], axis=-1), y) and np.array_equal(st2, st)
    # the returned state is the last three inputs
    assert np.array_equal(st, x[..., -3:].astype(np.float64))


def test_history_matches_numpy_convolve():
    """With a start history the output is the convolution of history
    followed by the sequence, from the first sequence step on (the reference
    the planted mistakes below are checked against)."""
    x = _x(1, 2, 12, 9)
    w, b = (t.numpy() for t in synth.make_conv(2, 4, seed=10))
    s0 = synth.make_conv_state(1, 2, 4, seed=11).numpy()
    y, _ = oracle.conv1d(x, w, b, state_in=s0, silu=False)
    full = np.concatenate([s0.astype(np.float64), x.astype(np.float64)], axis=-1)
    for dd in range(2):
        ref = np.convolve(full[0, dd], w[dd, ::-1].astype(np.float64))[3:15] + b[dd]
        np.testing.assert_allclose(y[0, dd], ref, rtol=1e-13, atol=1e-13)


SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")
MUTATIONS = {
    "tap_shifted": ("long src = t - (K - 1) + k;                      /* index into the sequence */",
                    "long src = t - K + k;                      /* index into the sequence */"),
    "bias_dropped": ("double acc = bias ? (double)bias[d] : 0.0;\n            for (long k = 0; k < K; ++k) {",
                     "double acc = 0.0;\n            for (long k = 0; k < K; ++k) {"),
    "history_ignored": ("double xv = src >= 0 ? (double)xr[src] : hist[K - 1 + src];", "double xv = src >= 0 ? (double)xr[src] : 0.0;"),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_pins_catch(name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "m.c")
        so = os.path.join(d, "libm.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", so, c, "-lm"],
                       check=True)
        lib = ctypes.CDLL(so)
        fp, dp = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
        lib.ssm_oracle_conv1d.argtypes = [fp, fp, fp, fp, ctypes.c_int, dp, dp] + [ctypes.c_long] * 4
        x = _x(1, 2, 12, 9)
        w, b = (t.numpy() for t in synth.make_conv(2, 4, seed=10))
        s0 = synth.make_conv_state(1, 2, 4, seed=11).numpy()
        y = np.empty((1, 2, 12))
        st = np.empty((1, 2, 3))
        P = lambda a, t: a.ctypes.data_as(t)
        lib.ssm_oracle_conv1d(P(x, fp), P(w, fp), P(b, fp), P(s0, fp), 0, P(y, dp), P(st, dp), 1, 2, 12, 4)
        full = np.concatenate([s0.astype(np.float64), x.astype(np.float64)], axis=-1)
        ref = np.stack([[np.convolve(full[0, dd], w[dd, ::-1].astype(np.float64))[3:15] + b[dd] for dd in range(2)]])
        assert np.max(np.abs(y - ref)) > 1e-6, f"mutation {name} was not caught"
