"""The allocation-free entry point, ssm_scan_fwd_noalloc, on the GPU.

It exists for callers that cannot call cudaMalloc where they run the scan
(allocation may synchronise the device or fail under memory pressure), so it
keeps its scratch in a fixed 16 MiB array inside the library.  This file
checks, through the C ABI:
  * two calls in a row (different shapes) against the fp64 oracle and against
    the regular device entry point, within the parity tolerances;
  * the largest problem whose scratch fits the array exactly, which runs and
    matches the oracle, and the same problem one step longer, which is refused
    before anything runs;
  * a problem far too large, refused with its own status.
It is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import _native, synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
SSM_ERR_TOO_LARGE = -11
SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_02_gb300 import build
    build.build()
    oracle.build()
    return _native.load()


def _dev(p):
    g = lambda t: None if t is None else t.cuda()
    return dict(x=g(p.x), delta=g(p.delta), A=g(p.A), B=g(p.B), C=g(p.C), D=g(p.D), z=g(p.z),
                dt_bias=g(p.dt_bias))


def _ptr(t):
    return None if t is None else t.data_ptr()


def _noalloc(lib, p, t):
    y = torch.full_like(t["x"], float("nan"))
    fs = torch.full((p.batch, p.dim, p.dstate), float("nan"), dtype=torch.float32, device="cuda")
    code = _native.SSM_BF16 if p.dtype == "bf16" else _native.SSM_F32
    rc = lib.ssm_scan_fwd_noalloc(_ptr(t["x"]), _ptr(t["delta"]), _ptr(t["A"]), _ptr(t["B"]), _ptr(t["C"]),
                                  _ptr(t["D"]), _ptr(t["z"]), _ptr(t["dt_bias"]), int(p.delta_softplus),
                                  _ptr(y), _ptr(fs), p.batch, p.dim, p.dstate, p.seqlen, code,
                                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc, y, fs


def _close(got, ref, dtype, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bound = TOL[dtype] * (1.0 + np.abs(ref))
    assert np.all(err <= bound), f"{what}: {(err > bound).sum()} of {err.size} outside tolerance"


def _oracle(p):
    return oracle.fwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
                      None if p.D is None else p.D.numpy(), p.f32("z"),
                      None if p.dt_bias is None else p.dt_bias.numpy(), p.delta_softplus)


def _check_against_oracle(p, y, fs):
    yr, fr = _oracle(p)
    nch = p.batch * p.dim
    _close(y.float().cpu().numpy().reshape(nch, p.seqlen), yr, p.dtype, "y vs oracle")
    _close(fs.cpu().numpy().reshape(nch, p.dstate), fr, "f32", "final_state vs oracle")


def test_two_calls_match_oracle_and_device_entry_point(lib):
    problems = [
        synth.make_problem(3, 70, 16, 600, dtype="bf16", gate=True, seed=501),
        synth.make_problem(2, 33, 64, 257, dtype="f32", gate=False, seed=502, A_mode="random"),
    ]
    for p in problems:                                  # two calls in a row, different shapes
        t = _dev(p)
        rc, y, fs = _noalloc(lib, p, t)
        assert rc == 0, _native.status_string(rc)
        _check_against_oracle(p, y, fs)
        yd, fd = ssm.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                              dt_bias=t["dt_bias"], delta_softplus=p.delta_softplus,
                              return_final_state=True, variant="fused")
        torch.cuda.synchronize()
        _close(y.float().cpu().numpy(), yd.float().cpu().numpy(), p.dtype, "y vs device entry point")
        _close(fs.cpu().numpy(), fd.cpu().numpy(), "f32", "final_state vs device entry point")


def _largest_fitting_seqlen(batch, dim, dstate, dtype):
    """Largest L whose fused scratch fits the array (binary search over the
    library's own size query)."""
    ws = lambda L: ssm.workspace_size(batch, dim, dstate, L, dtype, "fused")
    lo, hi = 1, 1 << 24
    assert ws(lo) <= SCRATCH_BYTES < ws(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if ws(mid) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo, ws(lo)


def test_limit_edge(lib):
    # eight states, two sequences: the scratch reaches exactly 16 MiB
    batch, dim, dstate = 2, 6, 8
    L, used = _largest_fitting_seqlen(batch, dim, dstate, torch.float32)
    assert used == SCRATCH_BYTES, (L, used)
    p = synth.make_problem(batch, dim, dstate, L, dtype="f32", gate=True, seed=503, A_mode="random")
    t = _dev(p)
    rc, y, fs = _noalloc(lib, p, t)
    assert rc == 0, _native.status_string(rc)
    _check_against_oracle(p, y, fs)
    # one step longer no longer fits: refused, nothing written
    q = synth.make_problem(batch, dim, dstate, L + 1, dtype="f32", gate=True, seed=504)
    tq = _dev(q)
    rc, y, fs = _noalloc(lib, q, tq)
    assert rc == SSM_ERR_TOO_LARGE
    assert torch.isnan(y).all() and torch.isnan(fs).all()


def test_too_large_is_refused_before_launch(lib):
    # 64 states, 2 x 60000 steps need 2 * 60000 * 144 * 4 bytes > 16 MiB; no
    # pointer is ever dereferenced
    rc = lib.ssm_scan_fwd_noalloc(None, None, None, None, None, None, None, None, 1, None, None,
                                  2, 8, 64, 60000, _native.SSM_BF16, None)
    assert rc == SSM_ERR_TOO_LARGE
    assert "scratch" in _native.status_string(rc)
    # sizes whose product would wrap a 64-bit byte count are refused as well
    rc = lib.ssm_scan_fwd_noalloc(None, None, None, None, None, None, None, None, 1, None, None,
                                  1 << 20, 1, 64, 1 << 40, _native.SSM_BF16, None)
    assert rc == SSM_ERR_TOO_LARGE
