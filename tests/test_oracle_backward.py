"""Pins of the oracle's backward (no GPU).

The backward is checked against central finite differences of a forward
written independently here in numpy float64 (the plain recurrence, itself
checked against the pinned C forward first).  The loss is
    L = sum(wy * y) + sum(wf * final_state)
with random weights, so that its derivatives with respect to y and to the final
state are wy and wf, the dy and dfinal the backward takes.  Every gradient
(x, delta, z, A, B, C, D, dt_bias and the start state) is compared element by
element on small problems, with the gate and softplus on and off.  Planted
mistakes in a copy of the backward's source must fail the same comparison.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from selective_state_space_02_gb300 import synth


def fwd64(x, delta, A, B, C, D, z, bias, h0, softplus=True):
    """The forward recurrence in float64 (vectorised over batch, channel and
    state; serial in time).  Shapes as the oracle's; D, z, bias may be None."""
    Bt, Dm, L = x.shape
    N = A.shape[1]
    v = delta + (bias[None, :, None] if bias is not None else 0.0)
    Delta = np.logaddexp(0.0, v) if softplus else v
    h = np.zeros((Bt, Dm, N)) if h0 is None else h0.copy()
    y = np.empty((Bt, Dm, L))
    for t in range(L):
        a = np.exp(Delta[:, :, t, None] * A[None])                         # [b, d, n]
        h = a * h + (Delta[:, :, t] * x[:, :, t])[..., None] * B[:, None, :, t]
        q = np.einsum("bdn,bn->bd", h, C[:, :, t])
        if D is not None:
            q = q + D[None] * x[:, :, t]
        if z is not None:
            zt = z[:, :, t]
            q = q * zt / (1.0 + np.exp(-zt))
        y[:, :, t] = q
    return y, h


def _params(p, h0):
    g = lambda a: None if a is None else np.asarray(a, np.float64)
    return dict(x=g(p.f32("x")), delta=g(p.f32("delta")), A=g(p.A.numpy()), B=g(p.f32("B")), C=g(p.f32("C")),
                D=None if p.D is None else g(p.D.numpy()), z=g(p.f32("z")),
                bias=None if p.dt_bias is None else g(p.dt_bias.numpy()), h0=h0)


def _loss(prm, wy, wf, softplus):
    y, h = fwd64(prm["x"], prm["delta"], prm["A"], prm["B"], prm["C"], prm["D"], prm["z"], prm["bias"],
                 prm["h0"], softplus)
    return float(np.sum(wy * y) + np.sum(wf * h))


def _fd(prm, wy, wf, softplus, name):
    """Central differences with a relative step of 1e-4: the truncation error
    is O(1e-8) relative, and rounding costs about 1e-12 * |L| absolute."""
    base = prm[name]
    g = np.empty_like(base)
    for i in np.ndindex(base.shape):
        e = 1e-4 * max(1.0, abs(base[i]))
        keep = base[i]
        base[i] = keep + e
        lp = _loss(prm, wy, wf, softplus)
        base[i] = keep - e
        lm = _loss(prm, wy, wf, softplus)
        base[i] = keep
        g[i] = (lp - lm) / (2 * e)
    return g


ORACLE_NAME = {"x": "dx", "delta": "ddelta", "z": "dz", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
               "bias": "ddt_bias", "h0": "dh0"}


def _case(gate, softplus, start, seed):
    # without softplus Delta = delta itself must stay small: the "slow" recipe (delta ~ N(0, 0.1^2)) and no
    # dt_bias (the recipe's bias is the inverse softplus of the step size, meaningless without softplus)
    p = synth.make_problem(2, 3, 4, 9, gate=gate, seed=seed, A_mode="random", delta_softplus=softplus,
                           delta="logu" if softplus else "slow", use_dt_bias=softplus)
    h0 = synth.make_state(2, 3, 4, seed=seed + 1).numpy().astype(np.float64) if start else None
    rng = np.random.default_rng(seed + 2)
    wy = rng.standard_normal((2, 3, 9))
    wf = rng.standard_normal((2, 3, 4))
    return p, h0, wy, wf


def test_numpy_forward_matches_the_pinned_oracle():
    p = synth.make_problem(2, 3, 5, 17, gate=True, seed=90, A_mode="random")
    h0 = synth.make_state(2, 3, 5, seed=91).numpy().astype(np.float64)
    prm = _params(p, h0)
    y, h = fwd64(prm["x"], prm["delta"], prm["A"], prm["B"], prm["C"], prm["D"], prm["z"], prm["bias"], h0)
    yo, fo = oracle.fwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"), p.D.numpy(),
                        p.f32("z"), p.dt_bias.numpy(), True, h0=h0)
    np.testing.assert_allclose(y.reshape(yo.shape), yo, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h.reshape(fo.shape), fo, rtol=1e-12, atol=1e-13)


def _oracle_grads(p, h0, wy, wf, lib=None):
    if lib is None:
        return oracle.bwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"), wy,
                          D=None if p.D is None else p.D.numpy(), z=p.f32("z"),
                          dt_bias=None if p.dt_bias is None else p.dt_bias.numpy(),
                          delta_softplus=p.delta_softplus, h0=h0, dfinal=wf)
    return _mutant_bwd(lib, p, h0, wy, wf)


@pytest.mark.parametrize("gate,softplus,start", [(True, True, True), (False, True, False), (True, False, True),
                                                 (False, False, False)])
def test_backward_matches_finite_differences(gate, softplus, start):
    p, h0, wy, wf = _case(gate, softplus, start, seed=93 + 4 * gate + 2 * softplus + start)
    prm = _params(p, h0)
    got = _oracle_grads(p, h0, wy, wf)
    names = ["x", "delta", "A", "B", "C", "D"] + (["bias"] if softplus else []) + (["z"] if gate else []) + \
        (["h0"] if start else [])
    atol = 1e-8 + 1e-10 * abs(_loss(prm, wy, wf, softplus))
    for name in names:
        fd = _fd(prm, wy, wf, softplus, name)
        np.testing.assert_allclose(got[ORACLE_NAME[name]], fd, rtol=1e-6, atol=atol, err_msg=name)


def test_gradients_without_a_loss_on_the_state_are_those_of_y_alone():
    p, h0, wy, _ = _case(True, True, False, seed=97)
    a = oracle.bwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"), wy, D=p.D.numpy(),
                   z=p.f32("z"), dt_bias=p.dt_bias.numpy(), dfinal=None)
    b = oracle.bwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"), wy, D=p.D.numpy(),
                   z=p.f32("z"), dt_bias=p.dt_bias.numpy(), dfinal=np.zeros((2, 3, 4)))
    for k in a:
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k


# ---------------------------------------------------------------- mutations
SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")
MUTATIONS = {
    "state_carry_dropped": ("                lam[n] *= at;\n", ""),
    "dB_without_delta": ("if (dBm) dBm[bi] += lam[n] * Dl[t] * xt;", "if (dBm) dBm[bi] += lam[n] * xt;"),
    "dA_without_delta": ("dA[(size_t)d * (size_t)dstate + (size_t)n] += da * at * Dl[t];",
                         "dA[(size_t)d * (size_t)dstate + (size_t)n] += da * at;"),
    "softplus_slope_dropped": ("double dv = softplus ? dDl / (1.0 + exp(-vv[t])) : dDl;", "double dv = dDl;"),
    "skip_in_dx_dropped": ("dx[(size_t)c * (size_t)L + (size_t)t] = du * Dl[t] + dq * Dd;",
                           "dx[(size_t)c * (size_t)L + (size_t)t] = du * Dl[t];"),
    "gate_slope_wrong": ("* (sg + zt * sg * (1.0 - sg));", "* sg;"),
    "dC_from_previous_state": ("if (dCm) dCm[bi] += dq * ht;", "if (dCm) dCm[bi] += dq * hp;"),
    "delta_input_term_dropped": ("            dDl += du * xt;\n", ""),
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
    fp, dp = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    lib.ssm_oracle_bwd.argtypes = [fp] * 8 + [ctypes.c_int] + [dp] * 12 + [ctypes.c_long] * 4
    return lib


def _mutant_bwd(lib, p, h0, wy, wf):
    fp, dp = ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_double)
    ptr = lambda a, t: ctypes.cast(None, t) if a is None else a.ctypes.data_as(t)
    f = lambda a: None if a is None else np.ascontiguousarray(a, np.float32)
    ins = [f(p.f32("x")), f(p.f32("delta")), f(p.A.numpy()), f(p.f32("B")), f(p.f32("C")),
           f(None if p.D is None else p.D.numpy()), f(p.f32("z")), f(None if p.dt_bias is None else p.dt_bias.numpy())]
    out = dict(dx=np.empty(p.x.shape), ddelta=np.empty(p.x.shape), dA=np.empty(p.A.shape), dB=np.empty(p.B.shape),
               dC=np.empty(p.C.shape), dD=np.empty((p.dim,)), dz=np.empty(p.x.shape) if p.z is not None else None,
               ddt_bias=np.empty((p.dim,)), dh0=np.empty((p.batch, p.dim, p.dstate)))
    wy = np.ascontiguousarray(wy, np.float64)
    wf = np.ascontiguousarray(wf, np.float64)
    h0 = None if h0 is None else np.ascontiguousarray(h0, np.float64)
    rc = lib.ssm_oracle_bwd(*[ptr(a, fp) for a in ins], int(p.delta_softplus), ptr(h0, dp), ptr(wy, dp),
                            ptr(wf, dp), *[ptr(out[k], dp) for k in ("dx", "ddelta", "dA", "dB", "dC", "dD", "dz",
                                                                     "ddt_bias", "dh0")],
                            p.batch, p.dim, p.dstate, p.seqlen)
    assert rc == 0
    return out


@pytest.fixture(scope="module")
def tmp():
    with tempfile.TemporaryDirectory() as d:
        yield d


def _worst(got, prm, wy, wf):
    worst = 0.0
    for n in ["x", "delta", "A", "B", "C", "D", "bias", "z", "h0"]:
        fd = _fd(prm, wy, wf, True, n)
        worst = max(worst, float(np.max(np.abs(got[ORACLE_NAME[n]] - fd) / (1e-8 + 1e-6 * np.abs(fd)))))
    return worst


def test_mutation_harness_control():
    p, h0, wy, wf = _case(True, True, True, seed=99)
    assert _worst(_oracle_grads(p, h0, wy, wf), _params(p, h0), wy, wf) < 1.0


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_finite_differences_catch(name, tmp):
    lib = _mutant(name, tmp)
    p, h0, wy, wf = _case(True, True, True, seed=99)
    assert _worst(_oracle_grads(p, h0, wy, wf, lib), _params(p, h0), wy, wf) > 1.0, f"mutation {name} was not caught"
