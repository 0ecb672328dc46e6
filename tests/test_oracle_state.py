"""Pins of the oracle's start-state forward and its one-token step (no GPU).

The start state h0 enters the recurrence h_t = a_t h_{t-1} + b_t linearly,
so three independent facts fix it:
  * with x = 0 the state only decays, h_t[n] = exp(A[n] * S_t) * h0[n] with
    S_t the prefix sum of Delta (a closed form evaluated here with numpy);
  * superposition: the run from (h0, x) is the run from (0, x) plus the run
    from (h0, 0);
  * resumption: running [0, k) and then [k, L) from the state reached at k
    is the run over [0, L) ("Mamba (part 2)", sect. 4.3: a segment restarts
    from the boundary state of the one before it).
The step is the recurrence for one token ("Mamba (part 2)", sect. 6-7:
inference advances the state one token at a time); L steps must reproduce
the forward exactly, and one step has a closed form.  Planted mistakes in a
copy of the oracle source must be caught by these pins.
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


def _args(p):
    return (p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
            None if p.D is None else p.D.numpy(), p.f32("z"),
            None if p.dt_bias is None else p.dt_bias.numpy(), p.delta_softplus)


def _delta(p):
    v = p.f32("delta").astype(np.float64)
    if p.dt_bias is not None:
        v = v + p.dt_bias.numpy().astype(np.float64)[None, :, None]
    return np.logaddexp(0.0, v) if p.delta_softplus else v


def _fwd(p, h0=None, x=None):
    a = list(_args(p))
    if x is not None:
        a[0] = x
    y, fs = oracle.fwd(*a, h0=h0)
    return y.reshape(p.batch, p.dim, p.seqlen), fs.reshape(p.batch, p.dim, p.dstate)


@pytest.mark.parametrize("gate", [False, True])
def test_zero_input_decays_the_start_state(gate):
    p = synth.make_problem(2, 3, 5, 40, gate=gate, seed=61, A_mode="random")
    h0 = synth.make_state(2, 3, 5, seed=62).numpy().astype(np.float64)
    y, fs = _fwd(p, h0=h0, x=np.zeros_like(p.f32("x")))
    S = np.cumsum(_delta(p), axis=-1)                               # [b, d, t]
    A = p.A.numpy().astype(np.float64)                              # [d, n]
    h = np.exp(A[None, :, :, None] * S[:, :, None, :]) * h0[..., None]   # [b, d, n, t]
    Cm = p.f32("C").astype(np.float64)                              # [b, n, t]
    yc = np.einsum("bnt,bdnt->bdt", Cm, h)
    if gate:
        z = p.f32("z").astype(np.float64)
        yc = yc * z * expit(z)
    np.testing.assert_allclose(y, yc, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(fs, h[..., -1], rtol=1e-11, atol=1e-13)


def test_superposition_of_start_state_and_input():
    p = synth.make_problem(2, 4, 6, 33, gate=False, seed=63, A_mode="random")
    h0 = synth.make_state(2, 4, 6, seed=64).numpy().astype(np.float64)
    y_both, f_both = _fwd(p, h0=h0)
    y_in, f_in = _fwd(p)
    y_st, f_st = _fwd(p, h0=h0, x=np.zeros_like(p.f32("x")))
    # the skip D x is linear in x, so it belongs to the input run only
    np.testing.assert_allclose(y_both, y_in + y_st, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(f_both, f_in + f_st, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("k", [1, 7, 32])
def test_resuming_from_the_boundary_state(k):
    p = synth.make_problem(1, 3, 4, 33, gate=True, seed=65)
    h0 = synth.make_state(1, 3, 4, seed=66).numpy().astype(np.float64)
    y, fs = _fwd(p, h0=h0)
    cut = lambda a, s: None if a is None else np.ascontiguousarray(a[:, :, s])
    a = _args(p)
    y1, f1 = oracle.fwd(cut(a[0], slice(0, k)), cut(a[1], slice(0, k)), a[2], cut(a[3], slice(0, k)),
                        cut(a[4], slice(0, k)), a[5], cut(a[6], slice(0, k)), a[7], a[8], h0=h0)
    y2, f2 = oracle.fwd(cut(a[0], slice(k, None)), cut(a[1], slice(k, None)), a[2], cut(a[3], slice(k, None)),
                        cut(a[4], slice(k, None)), a[5], cut(a[6], slice(k, None)), a[7], a[8],
                        h0=f1.reshape(1, 3, 4))
    # the same double arithmetic in the same order: exact
    assert np.array_equal(np.concatenate([y1, y2], axis=1).reshape(y.shape), y)
    assert np.array_equal(f2.reshape(fs.shape), fs)


def _steps(p, h0):
    h = h0.copy()
    ys = []
    for t in range(p.seqlen):
        s = synth.step_inputs(p, t)
        f = lambda v: None if v is None else v.float().numpy()
        h, y = oracle.step(h, f(s["x"]), f(s["delta"]), p.A.numpy(), f(s["B"]), f(s["C"]),
                           None if p.D is None else p.D.numpy(), f(s["z"]),
                           None if p.dt_bias is None else p.dt_bias.numpy(), p.delta_softplus)
        ys.append(y)
    return np.stack(ys, axis=-1), h


@pytest.mark.parametrize("gate,dtype", [(True, "bf16"), (False, "f32")])
def test_steps_reproduce_the_forward(gate, dtype):
    p = synth.make_problem(2, 5, 7, 19, dtype=dtype, gate=gate, seed=67, A_mode="random")
    h0 = synth.make_state(2, 5, 7, seed=68).numpy().astype(np.float64)
    y, fs = _fwd(p, h0=h0)
    ys, h = _steps(p, h0)
    assert np.array_equal(ys, y) and np.array_equal(h, fs)


def test_one_step_closed_form():
    p = synth.make_problem(3, 4, 6, 1, gate=True, seed=69, A_mode="random")
    h0 = synth.make_state(3, 4, 6, seed=70).numpy().astype(np.float64)
    s = synth.step_inputs(p, 0)
    f = lambda v: v.float().numpy().astype(np.float64)
    Delta = _delta(p)[:, :, 0]                                        # [b, d]
    A = p.A.numpy().astype(np.float64)
    h = np.exp(Delta[..., None] * A[None]) * h0 + (Delta * f(s["x"]))[..., None] * f(s["B"])[:, None, :]
    y = np.einsum("bn,bdn->bd", f(s["C"]), h) + p.D.numpy().astype(np.float64)[None] * f(s["x"])
    z = f(s["z"])
    y = y * z * expit(z)
    ho, yo = oracle.step(h0, s["x"].numpy(), s["delta"].numpy(), p.A.numpy(), s["B"].numpy(), s["C"].numpy(),
                         p.D.numpy(), s["z"].numpy(), p.dt_bias.numpy(), True)
    np.testing.assert_allclose(ho, h, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(yo, y, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- mutations
SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")
MUTATIONS = {
    "start_state_ignored": ("        if (h0)\n            for (long n = 0; n < dstate; ++n) h[n] = h0[(size_t)c * (size_t)dstate + (size_t)n];\n", ""),
    "start_state_other_channel": ("h[n] = h0[(size_t)c * (size_t)dstate + (size_t)n];",
                                  "h[n] = h0[(size_t)((c + 1) % nall) * (size_t)dstate + (size_t)n];"),
    "step_decay_next_state": ("double decay = exp(step * (double)A[(size_t)d * (size_t)dstate + (size_t)k]);",
                              "double decay = exp(step * (double)A[(size_t)d * (size_t)dstate + (size_t)((k + 1) % dstate)]);"),
    "step_inject_without_delta": ("double inject = step * (double)Bv[", "double inject = 1.0 * (double)Bv["),
    "step_skip_dropped": ("out = out + skip * xin;", ""),
    "step_output_before_update": ("            s[k] = decay * s[k] + inject;\n            out += (double)Cv[(size_t)bb * (size_t)dstate + (size_t)k] * s[k];",
                                  "            out += (double)Cv[(size_t)bb * (size_t)dstate + (size_t)k] * s[k];\n            s[k] = decay * s[k] + inject;"),
}


def _mutant(name, d):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    c = os.path.join(d, name + ".c")
    so = os.path.join(d, "lib" + name + ".so")
    open(c, "w").write(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", so, c, "-lm"],
                   check=True)
    lib = ctypes.CDLL(so)
    fp, dp, lp = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_long)
    lib.ssm_oracle_fwd_from.argtypes = [fp] * 8 + [ctypes.c_int, dp, dp, dp] + [ctypes.c_long] * 4 + \
        [lp, ctypes.c_long, ctypes.c_int]
    lib.ssm_oracle_step.argtypes = [dp] + [fp] * 8 + [ctypes.c_int, dp] + [ctypes.c_long] * 3
    return lib


def _ptr(a, t):
    return ctypes.cast(None, t) if a is None else a.ctypes.data_as(t)


def _mutant_fwd(lib, p, h0, x=None):
    fp, dp = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    a = [np.ascontiguousarray(v, np.float32) if v is not None else None for v in _args(p)[:8]]
    if x is not None:
        a[0] = np.ascontiguousarray(x, np.float32)
    y = np.empty((p.batch * p.dim, p.seqlen))
    fs = np.empty((p.batch * p.dim, p.dstate))
    h0 = np.ascontiguousarray(h0, np.float64)
    rc = lib.ssm_oracle_fwd_from(*[_ptr(v, fp) for v in a], int(p.delta_softplus), _ptr(h0, dp), _ptr(y, dp),
                                 _ptr(fs, dp), p.batch, p.dim, p.dstate, p.seqlen,
                                 ctypes.cast(None, ctypes.POINTER(ctypes.c_long)), 0, 1)
    assert rc == 0
    return y.reshape(p.batch, p.dim, p.seqlen), fs.reshape(p.batch, p.dim, p.dstate)


def _mutant_steps(lib, p, h0):
    fp, dp = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    h = np.ascontiguousarray(h0, np.float64).copy()
    ys = []
    for t in range(p.seqlen):
        s = synth.step_inputs(p, t)
        f = lambda v: None if v is None else np.ascontiguousarray(v.float().numpy(), np.float32)
        y = np.empty((p.batch, p.dim))
        A, D, bias = p.A.numpy(), p.D.numpy(), p.dt_bias.numpy()
        rc = lib.ssm_oracle_step(_ptr(h, dp), _ptr(f(s["x"]), fp), _ptr(f(s["delta"]), fp), _ptr(A, fp),
                                 _ptr(f(s["B"]), fp), _ptr(f(s["C"]), fp), _ptr(D, fp), _ptr(f(s["z"]), fp),
                                 _ptr(bias, fp), int(p.delta_softplus), _ptr(y, dp), p.batch, p.dim, p.dstate)
        assert rc == 0
        ys.append(y)
    return np.stack(ys, axis=-1), h


@pytest.fixture(scope="module")
def tmp():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name", ["start_state_ignored", "start_state_other_channel"])
def test_start_state_pins_catch(name, tmp):
    lib = _mutant(name, tmp)
    p = synth.make_problem(2, 3, 5, 40, gate=False, seed=61, A_mode="random")
    h0 = synth.make_state(2, 3, 5, seed=62).numpy().astype(np.float64)
    y, _ = _mutant_fwd(lib, p, h0, x=np.zeros_like(p.f32("x")))
    S = np.cumsum(_delta(p), axis=-1)
    h = np.exp(p.A.numpy().astype(np.float64)[None, :, :, None] * S[:, :, None, :]) * h0[..., None]
    yc = np.einsum("bnt,bdnt->bdt", p.f32("C").astype(np.float64), h)
    assert np.max(np.abs(y - yc)) > 1e-6, name


@pytest.mark.parametrize("name", [m for m in MUTATIONS if m.startswith("step_")])
def test_step_pins_catch(name, tmp):
    lib = _mutant(name, tmp)
    p = synth.make_problem(2, 5, 7, 19, gate=True, seed=67, A_mode="random")
    h0 = synth.make_state(2, 5, 7, seed=68).numpy().astype(np.float64)
    y, fs = _fwd(p, h0=h0)                # the shipped forward, pinned above
    ys, h = _mutant_steps(lib, p, h0)
    assert np.max(np.abs(ys - y)) > 1e-6 or np.max(np.abs(h - fs)) > 1e-6, name
