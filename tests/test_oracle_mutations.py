"""Planted mistakes: each plausible error in a copy of the oracle must be
caught by an independent pin (no GPU).

The test copies the oracle's C source, applies one textual mutation (a
dropped term, a flipped sign, a shifted or transposed index, swapped
composition operands), compiles the copy to a temporary library and checks
that the closed-form / brute-force pins reject it.  The shipped oracle is
never modified.
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
from test_oracle_forward import _closed_form

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")

MUTATIONS = {
    "flip_sign_of_b": ("h[n] = an * h[n] + bn;", "h[n] = an * h[n] - bn;"),
    "drop_skip": ("double yv = acc + Dd * xt;", "double yv = acc;"),
    "B_one_step_late": ("double bn = Delta * (double)Br[(size_t)n * (size_t)L + (size_t)t] * xt;",
                        "double bn = Delta * (double)Br[(size_t)n * (size_t)L + (size_t)(t > 0 ? t - 1 : 0)] * xt;"),
    "A_states_reversed": ("double an = exp(Delta * (double)Ar[n]);",
                          "double an = exp(Delta * (double)Ar[dstate - 1 - n]);"),
    "gate_dropped": ("if (zr) yv *= ssm_oracle_silu((double)zr[t]);", ""),
    "softplus_skipped": ("double Delta = softplus ? ssm_oracle_softplus(v) : v;\n            double acc",
                         "double Delta = v;\n            double acc"),
    "C_read_from_B": ("acc += (double)Cr[(size_t)n", "acc += (double)Br[(size_t)n"),
    "compose_swapped": ("*b_out = a2 * b1 + b2;", "*b_out = a1 * b2 + b1;"),
}


def _build_mutant(name, tmpdir):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    src = src.replace(old, new)
    cpath = os.path.join(tmpdir, f"{name}.c")
    lpath = os.path.join(tmpdir, f"lib{name}.so")
    with open(cpath, "w") as f:
        f.write(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", lpath, cpath, "-lm"], check=True)
    return ctypes.CDLL(lpath)


def _fwd_with(lib, p):
    fp = ctypes.POINTER(ctypes.c_float)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.ssm_oracle_fwd.restype = ctypes.c_int
    arrs = [p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
            p.D.numpy(), p.f32("z"), p.dt_bias.numpy()]
    arrs = [np.ascontiguousarray(a, np.float32) if a is not None else None for a in arrs]
    ptrs = [a.ctypes.data_as(fp) if a is not None else ctypes.cast(None, fp) for a in arrs]
    y = np.empty((p.batch * p.dim, p.seqlen))
    fs = np.empty((p.batch * p.dim, p.dstate))
    rc = lib.ssm_oracle_fwd(*ptrs, ctypes.c_int(1), y.ctypes.data_as(dp), fs.ctypes.data_as(dp),
                            ctypes.c_long(p.batch), ctypes.c_long(p.dim), ctypes.c_long(p.dstate),
                            ctypes.c_long(p.seqlen), ctypes.cast(None, ctypes.POINTER(ctypes.c_long)),
                            ctypes.c_long(0), ctypes.c_int(1))
    assert rc == 0
    return y.reshape(p.batch, p.dim, p.seqlen)


@pytest.fixture(scope="module")
def tmpdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name", [m for m in MUTATIONS if m != "compose_swapped"])
def test_forward_pin_catches(name, tmpdir):
    lib = _build_mutant(name, tmpdir)
    p = synth.make_problem(1, 3, 4, 24, gate=True, seed=30, A_mode="random")
    yc, _ = _closed_form(p)
    ym = _fwd_with(lib, p)
    assert np.max(np.abs(ym - yc)) > 1e-6, f"mutation {name} was not caught"


def test_unmutated_copy_passes(tmpdir):
    # control: the same harness with the real source agrees with the pin
    src = open(SRC).read()
    cpath = os.path.join(tmpdir, "control.c")
    lpath = os.path.join(tmpdir, "libcontrol.so")
    open(cpath, "w").write(src)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", lpath, cpath, "-lm"], check=True)
    p = synth.make_problem(1, 3, 4, 24, gate=True, seed=30, A_mode="random")
    yc, _ = _closed_form(p)
    np.testing.assert_allclose(_fwd_with(ctypes.CDLL(lpath), p), yc, rtol=1e-10, atol=1e-12)


def test_compose_pin_catches(tmpdir):
    lib = _build_mutant("compose_swapped", tmpdir)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.ssm_oracle_compose.argtypes = [ctypes.c_double] * 4 + [dp, dp]
    a, b = ctypes.c_double(), ctypes.c_double()
    lib.ssm_oracle_compose(2.0, 3.0, 5.0, 7.0, ctypes.byref(a), ctypes.byref(b))
    h = 1.5
    assert a.value * h + b.value != 2.0 * (5.0 * h + 7.0) + 3.0
