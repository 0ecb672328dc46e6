"""Failure detection of the bounded waits, made to fire without a GPU fault.

Every mbarrier wait in the scan kernels gives up after a cycle limit, sets bit
0 of the device status word and lets its kernel return, so a lost copy shows
up as a status the host reads instead of a hung GPU.  Here a self-test kernel
waits on a barrier that nothing arrives on and no copy targets (so no copy is
in flight when it gives up); the test checks that the status word reports it,
that clearing resets it, and that a scan launched afterwards still runs and
matches the oracle (the context stays usable).
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import _native, synth

ERR_DIMS = -2


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_02_gb300 import build
    build.build()
    return _native.load()


def test_limit_out_of_range_is_refused_on_the_host(lib):
    # validation happens before anything is launched: no GPU needed
    assert lib.ssm_scan_selftest_wait_timeout(0, None) == ERR_DIMS
    assert lib.ssm_scan_selftest_wait_timeout(-5, None) == ERR_DIMS
    assert lib.ssm_scan_selftest_wait_timeout((1 << 31) + 1, None) == ERR_DIMS


@pytest.mark.gpu
def test_bounded_wait_runs_out_and_is_reported(lib):
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.ssm_scan_device_status(stream, 1) >= 0          # start from a clear word
    assert lib.ssm_scan_device_status(stream, 0) == 0
    assert lib.ssm_scan_selftest_wait_timeout(100_000, stream) == 0
    assert lib.ssm_scan_device_status(stream, 1) & 1 == 1       # the wait gave up and said so
    assert lib.ssm_scan_device_status(stream, 0) == 0           # cleared
    # the context is still usable: a scan right after matches the oracle and
    # leaves the word clear
    p = synth.make_problem(2, 40, 16, 300, dtype="f32", gate=True, seed=610)
    dev = lambda t: None if t is None else t.cuda()
    y, fs = ssm.scan_fwd(dev(p.x), dev(p.delta), dev(p.A), dev(p.B), dev(p.C), D=dev(p.D), z=dev(p.z),
                         dt_bias=dev(p.dt_bias), return_final_state=True, variant="fused")
    torch.cuda.synchronize()
    oracle.build()
    yr, fr = oracle.fwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"), p.D.numpy(),
                        p.f32("z"), p.dt_bias.numpy(), True)
    err = np.abs(y.cpu().numpy().reshape(yr.shape) - yr) / (1 + np.abs(yr))
    assert err.max() <= 1e-4
    assert lib.ssm_scan_device_status(stream, 0) == 0
