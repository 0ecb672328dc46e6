"""GPU parity at the numerical extremes the scan page warns about ("Mamba
hardware-aware parallel associative scan", sect. 3.2 and 4.3): decay
products that underflow, and sequences long enough that a chain of
multipliers or an accumulation order could lose precision.

The kernels never multiply the a_t of a chunk into one product: the serial
recurrence h = a h + b absorbs an underflowing a (h becomes b), and every
carry across segments or chunks is exp(A * sum Delta), the log-domain form the
page recommends.  These tests hold the results at those extremes to the same
tolerances as everywhere else (1e-4 (1 + |ref|) for float32 I/O).
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import synth

from test_parity import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_02_gb300 import build
    build.build()
    oracle.build()


@pytest.mark.parametrize("variant", ["twopass", "fused"])
def test_a_million_steps(variant):
    """2^20 steps of slow decay (Delta near 1e-3, the long-sequence recipe):
    the two-pass plan cuts it into hundreds of segments, so the carry scan runs
    many 32-segment rounds."""
    p = synth.make_problem(1, 24, 16, 1 << 20, dtype="f32", gate=False, delta="slow", seed=600)
    yg, fg = run_gpu(p, variant)
    yr, fr = run_oracle(p)
    assert_close(yg.reshape(yr.shape), yr, "f32", f"y[{variant}]")
    assert_close(fg.reshape(fr.shape), fr, "f32", f"final_state[{variant}]")


@pytest.mark.parametrize("variant", ["fused", "twopass", "chunked"])
def test_decay_that_underflows(variant):
    """Delta near 4 and A down to -64: exp(Delta A) reaches 1e-111, far below
    the float32 range, so most multipliers are exactly 0 on the GPU and the
    state forgets at every step; a few slow states (A near -0.05) keep long
    memory beside them."""
    p = synth.make_problem(2, 20, 16, 3000, dtype="f32", gate=True, seed=601, A_mode="random", a_scale=4.0)
    p.delta = p.delta + 4.0
    A = p.A.clone()
    A[:, ::4] = -0.05                                     # slow states among the fast ones
    p.A = A * 4.0
    yg, fg = run_gpu(p, variant)
    yr, fr = run_oracle(p)
    assert np.isfinite(yg).all() and np.isfinite(fg).all()
    assert_close(yg.reshape(yr.shape), yr, "f32", f"y[{variant}]")
    assert_close(fg.reshape(fr.shape), fr, "f32", f"final_state[{variant}]")


def test_backward_over_many_chunks_with_fast_decay():
    """The backward's adjoint is carried across 256 chunks with multipliers
    that underflow; its gradients stay within the backward's tolerance."""
    from test_parity_bwd import _run, _compare, _dy
    p = synth.make_problem(1, 16, 16, 8192, dtype="f32", gate=False, seed=602, A_mode="random")
    p.delta = p.delta + 2.0
    g, ref = _run(p, _dy(p, 11))
    _compare(g, ref, "f32")
