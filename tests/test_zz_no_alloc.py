"""The allocation-free entry point, ssm_scan_fwd_noalloc, on the GPU.

It exists for callers that cannot call cudaMalloc where they run the scan
(allocation may synchronise the device or fail under memory pressure), so it
keeps its scratch in a fixed array inside the library.  This file checks,
through the C ABI, that two calls in a row give the same results as the
regular device entry point (within the parity tolerances), that a problem too
large for the built-in scratch is refused before anything runs, and that the
call needs no workspace argument.  It is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import _native, synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
SSM_ERR_TOO_LARGE = -11


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_02_gb300 import build
    build.build()
    return _native.load()


def _dev(p):
    g = lambda t: None if t is None else t.cuda()
    return dict(x=g(p.x), delta=g(p.delta), A=g(p.A), B=g(p.B), C=g(p.C), D=g(p.D), z=g(p.z),
                dt_bias=g(p.dt_bias))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _noalloc(lib, p, t):
    y = torch.empty_like(t["x"])
    fs = torch.empty(p.batch, p.dim, p.dstate, dtype=torch.float32, device="cuda")
    code = _native.SSM_BF16 if p.dtype == "bf16" else _native.SSM_F32
    rc = lib.ssm_scan_fwd_noalloc(_ptr(t["x"]), _ptr(t["delta"]), _ptr(t["A"]), _ptr(t["B"]), _ptr(t["C"]),
                                  _ptr(t["D"]), _ptr(t["z"]), _ptr(t["dt_bias"]), int(p.delta_softplus),
                                  _ptr(y), _ptr(fs), p.batch, p.dim, p.dstate, p.seqlen, code,
                                  torch.cuda.current_stream().cuda_stream)
    return rc, y, fs


def _close(got, ref, dtype):
    got = got.float().cpu().numpy().astype(np.float64)
    ref = ref.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= TOL[dtype] * (1.0 + np.abs(ref)))


def test_two_calls_match_the_device_entry_point(lib):
    problems = [
        synth.make_problem(3, 70, 16, 600, dtype="bf16", gate=True, seed=501),
        synth.make_problem(2, 33, 64, 257, dtype="f32", gate=False, seed=502, A_mode="random"),
    ]
    for p in problems:                                  # two calls in a row, different shapes
        t = _dev(p)
        rc, y, fs = _noalloc(lib, p, t)
        assert rc == 0, _native.status_string(rc)
        yr, fr = ssm.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                              dt_bias=t["dt_bias"], delta_softplus=p.delta_softplus,
                              return_final_state=True, variant="fused")
        torch.cuda.synchronize()
        _close(y, yr, p.dtype)
        _close(fs, fr, "f32")


def test_too_large_is_refused_before_launch(lib):
    # 64 states, 2 x 60000 steps need 2 * 60000 * 144 * 4 bytes > 16 MiB
    rc = lib.ssm_scan_fwd_noalloc(None, None, None, None, None, None, None, None, 1, None, None,
                                  2, 8, 64, 60000, _native.SSM_BF16, None)
    assert rc == SSM_ERR_TOO_LARGE
    assert "scratch" in _native.status_string(rc)
