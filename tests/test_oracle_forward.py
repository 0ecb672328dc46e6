"""Pins of the oracle's full forward selective scan (no GPU).

The forward is checked against a different statement of the same result:
the unrolled closed form
    h_t[n] = sum_{j<=t} exp(A[n] * (S_t - S_j)) * Delta_j * B_j[n] * x_j,
    S_t = Delta_1 + ... + Delta_t,
evaluated with numpy (prefix sums, logaddexp for softplus, expit for the
gate), plus special cases that reduce to library routines (cumsum), the
impulse response, degenerate inputs and the chunked two-pass scan fed with
the recurrence's own pairs.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from selective_state_space_02_gb300 import synth


def _closed_form(p):
    x = p.f32("x").astype(np.float64)
    dl = p.f32("delta").astype(np.float64)
    A = p.A.numpy().astype(np.float64)
    Bm = p.f32("B").astype(np.float64)
    Cm = p.f32("C").astype(np.float64)
    Dv = p.D.numpy().astype(np.float64) if p.D is not None else None
    z = p.f32("z").astype(np.float64) if p.z is not None else None
    bias = p.dt_bias.numpy().astype(np.float64) if p.dt_bias is not None else 0.0
    v = dl + (bias[None, :, None] if p.dt_bias is not None else 0.0)
    Delta = np.logaddexp(0.0, v) if p.delta_softplus else v
    S = np.cumsum(Delta, axis=-1)                         # [b, d, t]
    Bt, Dm, L = x.shape
    N = A.shape[1]
    y = np.zeros_like(x)
    hL = np.zeros((Bt, Dm, N))
    t_idx = np.arange(L)
    mask = t_idx[:, None] >= t_idx[None, :]                # j <= t
    for b in range(Bt):
        for d in range(Dm):
            u = Delta[b, d] * x[b, d]                          # [t]
            diff = S[b, d][:, None] - S[b, d][None, :]         # S_t - S_j
            for n in range(N):
                W = np.where(mask, np.exp(np.where(mask, A[d, n] * diff, 0.0)), 0.0)
                h = W @ (u * Bm[b, n])                          # [t]
                y[b, d] += Cm[b, n] * h
                hL[b, d, n] = h[-1]
            if Dv is not None:
                y[b, d] += Dv[d] * x[b, d]
            if z is not None:
                y[b, d] *= z[b, d] * expit(z[b, d])
    return y, hL


def _run(p, **kw):
    y, fs = oracle.fwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
                       None if p.D is None else p.D.numpy(), p.f32("z"),
                       None if p.dt_bias is None else p.dt_bias.numpy(),
                       p.delta_softplus, **kw)
    return y.reshape(p.batch, p.dim, p.seqlen), fs.reshape(p.batch, p.dim, p.dstate)


@pytest.mark.parametrize("gate,dtype,A_mode,softplus", [
    (False, "f32", "structured", True),
    (True, "f32", "random", True),
    (True, "bf16", "structured", True),
    (False, "f32", "random", False),
])
def test_forward_matches_unrolled_closed_form(gate, dtype, A_mode, softplus):
    p = synth.make_problem(2, 3, 5, 41, dtype=dtype, gate=gate, A_mode=A_mode, seed=7,
                           delta_softplus=softplus)
    if not softplus:
        # keep the step positive without the softplus: delta + bias > 0
        p.delta = p.delta.abs() * 0.05
        p.dt_bias = None
    y, hL = _run(p)
    yc, hc = _closed_form(p)
    np.testing.assert_allclose(y, yc, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(hL, hc, rtol=1e-10, atol=1e-13)


def test_forward_zero_A_is_prefix_sum():
    # A = 0 makes every a_t = 1 and the state a running sum of Delta*B*x
    p = synth.make_problem(1, 4, 3, 64, seed=11, delta_softplus=False, use_dt_bias=False)
    p.A = p.A * 0
    p.delta = p.delta.abs() * 0.1
    y, hL = _run(p)
    x = p.f32("x").astype(np.float64)
    dl = p.f32("delta").astype(np.float64)
    Bm = p.f32("B").astype(np.float64)
    Cm = p.f32("C").astype(np.float64)
    Dv = p.D.numpy().astype(np.float64)
    for d in range(4):
        h = np.cumsum(dl[0, d][None, :] * x[0, d][None, :] * Bm[0], axis=-1)   # [n, t]
        yref = (Cm[0] * h).sum(0) + Dv[d] * x[0, d]
        np.testing.assert_allclose(y[0, d], yref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(hL[0, d], h[:, -1], rtol=1e-12, atol=1e-13)


def test_forward_impulse_response():
    # x nonzero only at step j: h_t[n] = Delta_j B_j[n] x_j exp(A[n] (S_t - S_j))
    p = synth.make_problem(1, 2, 4, 50, seed=12, delta_softplus=False, use_dt_bias=False,
                           use_D=False, A_mode="random")
    p.delta = p.delta.abs() * 0.2
    j = 17
    xx = p.x.clone() * 0
    xx[:, :, j] = p.x[:, :, j]
    p.x = xx
    y, hL = _run(p)
    dl = p.f32("delta").astype(np.float64)
    A = p.A.numpy().astype(np.float64)
    Bm = p.f32("B").astype(np.float64)
    x = p.f32("x").astype(np.float64)
    for d in range(2):
        span = dl[0, d, j + 1:].sum()
        ref = dl[0, d, j] * Bm[0, :, j] * x[0, d, j] * np.exp(A[d] * span)
        np.testing.assert_allclose(hL[0, d], ref, rtol=1e-12)
        assert np.all(y[0, d, :j] == 0.0)


def test_forward_degenerate_cases():
    # B = 0: the state stays zero and y = D * x * silu(z)
    p = synth.make_problem(1, 3, 4, 30, gate=True, seed=13, B_zero=True)
    y, hL = _run(p)
    x = p.f32("x").astype(np.float64)
    z = p.f32("z").astype(np.float64)
    ref = p.D.numpy()[None, :, None] * x * (z * expit(z))
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-15)
    assert np.all(hL == 0.0)
    # C = 0 without D and gate: y = 0 exactly while the state still moves
    p = synth.make_problem(1, 3, 4, 30, seed=14, C_zero=True, use_D=False)
    y, hL = _run(p)
    assert np.all(y == 0.0) and np.any(hL != 0.0)
    # L = 1: h = Delta * B * x
    p = synth.make_problem(2, 3, 4, 1, seed=15, delta_softplus=False, use_dt_bias=False)
    p.delta = p.delta.abs()
    y, hL = _run(p)
    ref = p.f32("delta")[:, :, None, 0] * p.f32("B")[:, None, :, 0] * p.f32("x")[:, :, None, 0]
    np.testing.assert_allclose(hL, ref, rtol=1e-7)


def test_forward_channel_subset_and_threads():
    p = synth.make_problem(2, 5, 4, 37, gate=True, seed=16)
    yall, fall = _run(p)
    sel = [9, 0, 4]
    y, fs = oracle.fwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
                       p.D.numpy(), p.f32("z"), p.dt_bias.numpy(), True, channels=sel, nthreads=3)
    flat = yall.reshape(10, 37)
    np.testing.assert_array_equal(y, flat[sel])
    np.testing.assert_array_equal(fs, fall.reshape(10, 4)[sel])


def test_forward_consistent_with_chunked_pairs():
    # the forward's state equals the chunked two-pass scan of its own pairs
    p = synth.make_problem(1, 2, 3, 40, seed=17)
    _, hL = _run(p)
    for d in range(2):
        for n in range(3):
            a, b = oracle.pairs(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"),
                                p.dt_bias.numpy(), True, 0, d, n)
            h, bd = oracle.scan_chunked(a, b, 8)
            assert h[-1] == pytest.approx(hL[0, d, n], rel=1e-12, abs=1e-15)
            assert bd[-1] == h[-1]


def test_forward_rejects_bad_arguments():
    p = synth.make_problem(1, 2, 3, 8, seed=18)
    with pytest.raises(RuntimeError):
        oracle.fwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
                   channels=[5])
