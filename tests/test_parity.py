"""GPU parity: the CUDA library against the fp64 oracle, element by element.

Tolerances (float32 arithmetic, fp64 reference):
  float32 I/O: |y - y_ref| <= 1e-4 * (1 + |y_ref|)
  bf16 I/O   : |y - y_ref| <= 2e-2 * (1 + |y_ref|)
final_state (float32 in both cases) is held to the float32 bound.  Because the
skip term D*x dominates |y|, scan-only runs (no D, no gate) add a relative-RMS
check of y: <= 1e-3 (float32) and <= 3e-2 (bf16).
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}
RMS_TOL = {"f32": 1e-3, "bf16": 3e-2}
VARIANTS = ["fused", "chunked", "twopass"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_02_gb300 import build
    build.build()
    oracle.build()


def to_dev(p):
    dev = "cuda"
    g = lambda t: None if t is None else t.to(dev)
    return dict(x=g(p.x), delta=g(p.delta), A=g(p.A), B=g(p.B), C=g(p.C), D=g(p.D), z=g(p.z),
                dt_bias=g(p.dt_bias))


def run_gpu(p, variant="auto", final_state=True):
    t = to_dev(p)
    out = ssm.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                       dt_bias=t["dt_bias"], delta_softplus=p.delta_softplus,
                       return_final_state=final_state, variant=variant)
    torch.cuda.synchronize()
    if final_state:
        y, fs = out
        return y.float().cpu().numpy(), fs.cpu().numpy()
    return out.float().cpu().numpy(), None


def run_oracle(p, channels=None):
    y, fs = oracle.fwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"),
                       None if p.D is None else p.D.numpy(), p.f32("z"),
                       None if p.dt_bias is None else p.dt_bias.numpy(), p.delta_softplus,
                       channels=channels)
    return y, fs


def assert_close(got, ref, dtype, what):
    tol = TOL[dtype]
    err = np.abs(got.astype(np.float64) - ref)
    bound = tol * (1.0 + np.abs(ref))
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r}")


def check_problem(p, variant, channels=None):
    yg, fg = run_gpu(p, variant)
    nch = p.batch * p.dim
    yr, fr = run_oracle(p, channels)
    yg = yg.reshape(nch, p.seqlen)
    fg = fg.reshape(nch, p.dstate)
    if channels is not None:
        yg = yg[channels]
        fg = fg[channels]
    assert_close(yg, yr, p.dtype, f"y[{variant}]")
    assert_close(fg, fr, "f32", f"final_state[{variant}]")
    return yg, yr


# ---------------------------------------------------------------- small cases
SMALL = [
    # batch, dim, dstate, L, dtype, gate
    (1, 64, 16, 256, "f32", False),     # the tiny workload's shape
    (2, 37, 16, 333, "f32", True),      # ragged channels and length (scalar path)
    (3, 50, 16, 1000, "bf16", True),    # ragged length, 16-byte rows (1000*2 % 16 == 0)
    (1, 20, 64, 300, "bf16", True),     # wide state, ragged tile
    (2, 9, 5, 130, "f32", False),       # odd dstate
    (1, 3, 1, 77, "bf16", False),       # dstate = 1
    (1, 33, 32, 2100, "f32", True),     # several chunks of the chunked variant
    (1, 5, 8, 4097, "bf16", True),      # one step past a power of two
]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s[:4])) + f"-{s[4]}-g{int(s[5])}")
def test_small_parity(shape, variant):
    b, d, n, L, dt, gate = shape
    p = synth.make_problem(b, d, n, L, dtype=dt, gate=gate, seed=1000 + b * 7 + d + n + L,
                           A_mode="random")
    check_problem(p, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_workload_all_elements(variant):
    p = synth.workload("tiny_f32")
    check_problem(p, variant)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scan_only_rms(variant, dtype):
    # no skip, no gate: y is the scan contraction alone
    p = synth.make_problem(2, 48, 16, 700, dtype=dtype, gate=False, use_D=False, seed=77)
    yg, yr = check_problem(p, variant)
    rel = np.sqrt(np.mean((yg - yr) ** 2)) / np.sqrt(np.mean(yr ** 2))
    assert rel <= RMS_TOL[dtype], rel


@pytest.mark.parametrize("variant", VARIANTS)
def test_flags_off(variant):
    # softplus off (delta + bias must stay positive), no dt_bias, no D
    p = synth.make_problem(1, 24, 16, 200, dtype="f32", gate=True, use_D=False, use_dt_bias=False,
                           delta_softplus=False, seed=78)
    p.delta = p.delta.abs() * 0.05
    check_problem(p, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_slow_decay_long(variant):
    # a ~ 1 - 1e-3 over 20k steps: float32 error accumulation along L
    p = synth.make_problem(1, 16, 16, 20000, dtype="f32", delta="slow", seed=79)
    check_problem(p, variant)


def test_misaligned_views_take_scalar_path():
    # f32 rows starting 4 bytes past a 16-byte boundary
    p = synth.make_problem(1, 8, 16, 96, dtype="f32", gate=True, seed=80)
    t = to_dev(p)
    def shift(a):
        buf = torch.empty(a.numel() + 1, dtype=a.dtype, device="cuda")
        v = buf[1:].view(a.shape)
        v.copy_(a)
        return v
    xs, ds, zs, Bs, Cs = (shift(t[k]) for k in ("x", "delta", "z", "B", "C"))
    assert xs.data_ptr() % 16 != 0
    for variant in VARIANTS:
        y, fs = ssm.scan_fwd(xs, ds, t["A"], Bs, Cs, D=t["D"], z=zs, dt_bias=t["dt_bias"],
                             return_final_state=True, variant=variant)
        yr, fr = run_oracle(p)
        assert_close(y.float().cpu().numpy().reshape(8, 96), yr, "f32", f"misaligned y[{variant}]")
        assert_close(fs.cpu().numpy().reshape(8, 16), fr, "f32", f"misaligned fs[{variant}]")


@pytest.mark.parametrize("variant", VARIANTS)
def test_empty_and_degenerate(variant):
    # seqlen 0: y empty, final state zero
    p = synth.make_problem(2, 3, 4, 1, seed=81)
    t = to_dev(p)
    x0 = t["x"][:, :, :0].contiguous()
    B0 = t["B"][:, :, :0].contiguous()
    y, fs = ssm.scan_fwd(x0, x0.clone(), t["A"], B0, B0.clone(), return_final_state=True, variant=variant)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.all(fs == 0)
    # batch 0
    xe = torch.empty(0, 3, 5, device="cuda")
    ye = ssm.scan_fwd(xe, xe.clone(), t["A"], torch.empty(0, 4, 5, device="cuda"),
                      torch.empty(0, 4, 5, device="cuda"), variant=variant)
    assert ye.shape == (0, 3, 5)
    # L = 1
    p = synth.make_problem(2, 5, 16, 1, dtype="bf16", gate=True, seed=82)
    check_problem(p, variant)
    # B = 0: y is the gated skip exactly (float32 rounding only)
    p = synth.make_problem(1, 16, 16, 64, dtype="f32", gate=True, seed=83, B_zero=True)
    check_problem(p, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_deterministic(variant):
    p = synth.make_problem(2, 40, 16, 900, dtype="bf16", gate=True, seed=84)
    t = to_dev(p)
    outs = []
    for _ in range(3):
        y, fs = ssm.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                             dt_bias=t["dt_bias"], return_final_state=True, variant=variant)
        outs.append((y.clone(), fs.clone()))
    torch.cuda.synchronize()
    for y, fs in outs[1:]:
        assert torch.equal(y, outs[0][0]) and torch.equal(fs, outs[0][1])


def test_variants_agree_closely():
    p = synth.make_problem(2, 64, 16, 1500, dtype="f32", gate=True, seed=85)
    ys = {v: run_gpu(p, v)[0] for v in VARIANTS}
    for v in VARIANTS[1:]:
        np.testing.assert_allclose(ys[v], ys["fused"], rtol=1e-4, atol=1e-4)


def test_host_entry_point_matches_device():
    p = synth.make_problem(2, 30, 16, 500, dtype="bf16", gate=True, seed=86)
    yd, _ = run_gpu(p, final_state=False)
    pin = lambda a: None if a is None else a.pin_memory()
    fs = torch.empty(2, 30, 16).pin_memory()
    y = ssm.scan_fwd_host(pin(p.x), pin(p.delta), pin(p.A), pin(p.B), pin(p.C), D=pin(p.D), z=pin(p.z),
                          dt_bias=pin(p.dt_bias), final_state=fs)
    assert np.array_equal(y.float().numpy(), yd)
    yr, fr = run_oracle(p)
    assert_close(fs.numpy().reshape(60, 16), fr, "f32", "host final_state")


@pytest.mark.parametrize("batch,dim,L,dtype,gate,pinned_y", [
    (2, 1024, 4096, "bf16", True, True),     # three aligned time chunks
    (2, 1024, 4096, "bf16", True, False),    # the same into a pageable y
    (2, 1024, 4100, "bf16", True, True),     # ragged last chunk: rows not 16-byte aligned, element-load path
    (1, 256, 40000, "f32", False, True),     # three chunks, each scanned by the two-pass variant
    (1, 256, 40000, "f32", False, False),
    (2, 30, 500, "bf16", True, True),        # one chunk
])
def test_host_entry_point_time_chunks(batch, dim, L, dtype, gate, pinned_y):
    """Problems of 16 MiB or more go through the host entry point in time
    chunks, each starting from the state the previous one ended in, into a
    page-locked or a pageable y.  The result matches the oracle on sampled
    channels and the single-call device path everywhere within the
    tolerance."""
    p = synth.make_problem(batch, dim, 16, L, dtype=dtype, gate=gate, seed=87 + L)
    pin = lambda a: None if a is None else a.pin_memory()
    fs = torch.empty(batch, dim, 16).pin_memory()
    y0 = torch.full_like(p.x, float("nan"))
    y0 = y0.pin_memory() if pinned_y else y0
    assert y0.is_pinned() == pinned_y
    y = ssm.scan_fwd_host(pin(p.x), pin(p.delta), pin(p.A), pin(p.B), pin(p.C), D=pin(p.D), z=pin(p.z),
                          dt_bias=pin(p.dt_bias), delta_softplus=p.delta_softplus, y=y0, final_state=fs)
    assert y is y0
    nch = batch * dim
    yh = y.float().numpy().reshape(nch, L)
    yd, fd = run_gpu(p)
    assert_close(yh, yd.reshape(nch, L).astype(np.float64), dtype, "host y vs device y")
    assert_close(fs.numpy().reshape(nch, 16), fd.reshape(nch, 16).astype(np.float64), "f32",
                 "host final_state vs device final_state")
    ch = _sample_channels(p, 6, seed=88)
    yr, fr = run_oracle(p, ch)
    assert_close(yh[ch], yr, dtype, "host y vs oracle")
    assert_close(fs.numpy().reshape(nch, 16)[ch], fr, "f32", "host final_state vs oracle")


@pytest.mark.parametrize("variant", ["fused", "chunked", "twopass"])
def test_host_entry_point_explicit_variants(variant):
    """Every variant through the time-chunked host path (three chunks), with
    pageable inputs and output and the optional operands absent."""
    p = synth.make_problem(2, 1024, 16, 4096, dtype="bf16", gate=False, use_D=False, use_dt_bias=False, seed=95)
    y = ssm.scan_fwd_host(p.x, p.delta, p.A, p.B, p.C, delta_softplus=p.delta_softplus, variant=variant)
    assert not y.is_pinned()
    yd, _ = run_gpu(p, variant=variant, final_state=False)
    assert_close(y.float().numpy(), yd.astype(np.float64), "bf16", f"host y vs device y [{variant}]")
    ch = _sample_channels(p, 4, seed=96)
    yr, _ = run_oracle(p, ch)
    assert_close(y.float().numpy().reshape(-1, p.seqlen)[ch], yr, "bf16", f"host y vs oracle [{variant}]")


# ----------------------------------------------------- full-size workloads
def _sample_channels(p, k, seed):
    nch = p.batch * p.dim
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(nch, size=min(k, nch), replace=False).tolist())
    pick |= {0, nch - 1, p.dim - 1, min(p.dim, nch - 1)}
    return sorted(pick)


WORKLOAD_NAMES = ["tiny_f32", "mid_bf16", "large_batch_bf16", "long_seq_f32", "wide_state_bf16"]


def _full_compare(p, variant="auto", final_state=None):
    """Every element of y (and of the final state) against the oracle."""
    fs_flag = p.final_state if final_state is None else final_state
    yg, fg = run_gpu(p, variant, final_state=fs_flag)
    nch = p.batch * p.dim
    yr, fr = run_oracle(p)
    assert_close(yg.reshape(nch, p.seqlen), yr, p.dtype, f"y[{variant}]")
    if fs_flag:
        assert_close(fg.reshape(nch, p.dstate), fr, "f32", f"final_state[{variant}]")
    return yg.reshape(nch, p.seqlen), yr, fr


@pytest.mark.parametrize("name", WORKLOAD_NAMES)
def test_full_workload_all_elements(name):
    """The benchmark workloads at full size, in the launch configuration the
    benchmark times (AUTO variant, the workload's own final-state flag): every
    element of y against the oracle.  Workloads that do not return the final
    state run once more with it, and every element of it is checked too."""
    p = synth.workload(name)
    _, _, fr = _full_compare(p)
    if not p.final_state:
        fg = run_gpu(p, "auto", final_state=True)[1]
        assert_close(fg.reshape(p.batch * p.dim, p.dstate), fr, "f32", "final_state[auto]")


@pytest.mark.parametrize("name", ["tiny_f32", "mid_bf16", "large_batch_bf16"])
def test_full_workload_scan_only(name):
    """The first three workloads' shapes with the skip and the gate removed, so
    that y is the state contraction alone (at full size D*x*silu(z) dominates
    |y| and the elementwise bound alone could hide a broken scan): every
    element within the elementwise bound, and the relative RMS error of y
    within 1e-3 (float32) or 3e-2 (bf16)."""
    p = synth.workload(name, gate=False, use_D=False)
    yg, yr, _ = _full_compare(p, final_state=True)
    rel = np.sqrt(np.mean((yg - yr) ** 2)) / np.sqrt(np.mean(yr ** 2))
    assert rel <= RMS_TOL[p.dtype], rel
