"""GPU parity of the backward (ssm_scan_bwd) against the fp64 oracle's
backward, element by element, on seeded problems with ragged chunk tails and
partial channel blocks.

Tolerance.  The GPU runs the forward's float32 arithmetic (ex2.approx, the
fast softplus) twice per chunk and sums dA, dB, dC, dD and ddt_bias with float32
atomic additions in no fixed order; every gradient is a sum of many terms of
both signs, so an element near zero carries the rounding of its largest
terms.  Each gradient g of the oracle's g_ref is therefore held to
    |g - g_ref| <= rtol * |g_ref| + atol * max|g_ref|
with rtol = 1e-3, atol = 1e-4 for float32 I/O, and for bf16 I/O (dx, ddelta
and dz are stored in bf16, relative rounding 2^-9) rtol = 2e-2, atol = 5e-3.
For float32 I/O every element that is not small against its array
(|g_ref| >= 1e-2 * max|g_ref|) is also held to a purely relative bound,
|g - g_ref| <= 1e-3 * |g_ref|, so that the absolute term cannot cover a wrong
element of moderate size.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import synth

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-3, 1e-4), "bf16": (2e-2, 5e-3)}
REL_F32 = 1e-3          # per-element relative bound, float32 I/O
REL_FLOOR = 1e-2        # ... on elements with |g_ref| >= REL_FLOOR * max|g_ref|


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_02_gb300 import build
    build.build()
    oracle.build()


def _dy(p, seed):
    g = torch.from_numpy(np.random.default_rng(seed).standard_normal((p.batch, p.dim, p.seqlen)).astype(np.float32))
    return g.to(p.torch_dtype)


def _check(name, got, ref, dtype):
    rtol, atol = TOL[dtype]
    got = got.float().cpu().numpy().astype(np.float64) if torch.is_tensor(got) else got
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    err = np.abs(got - ref)
    bound = rtol * np.abs(ref) + atol * scale
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{name}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} (max|ref| {scale:.3g})")
    if dtype == "f32" and ref.size:
        big = np.abs(ref) >= REL_FLOOR * scale
        rel = np.where(big, err / np.maximum(np.abs(ref), 1e-300), 0.0)
        if rel.max() > REL_F32:
            i = np.unravel_index(np.argmax(rel), rel.shape)
            raise AssertionError(f"{name}: {(rel > REL_F32).sum()} of {big.sum()} elements above "
                                 f"{REL_FLOOR:g} * max|ref| outside the relative bound {REL_F32:g}; worst at "
                                 f"{i}: got {got[i]!r} ref {ref[i]!r}")


def _run(p, dy, h0=None, dfinal=None):
    dev = lambda t: None if t is None else t.cuda()
    g = ssm.scan_bwd(dev(p.x), dev(p.delta), dev(p.A), dev(p.B), dev(p.C), dev(dy), D=dev(p.D), z=dev(p.z),
                     dt_bias=dev(p.dt_bias), delta_softplus=p.delta_softplus, initial_state=dev(h0),
                     dfinal_state=dev(dfinal))
    torch.cuda.synchronize()
    ref = oracle.bwd(p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"), dy.float().numpy(),
                     D=None if p.D is None else p.D.numpy(), z=p.f32("z"),
                     dt_bias=None if p.dt_bias is None else p.dt_bias.numpy(), delta_softplus=p.delta_softplus,
                     h0=None if h0 is None else h0.numpy(), dfinal=None if dfinal is None else dfinal.numpy())
    return g, ref


PAIRS = [("dx", "dx"), ("ddelta", "ddelta"), ("dz", "dz"), ("dA", "dA"), ("dB", "dB"), ("dC", "dC"),
         ("dD", "dD"), ("ddt_bias", "ddt_bias"), ("dinitial_state", "dh0")]


def _compare(g, ref, dtype):
    for gk, rk in PAIRS:
        if g.get(gk) is None or ref.get(rk) is None:
            continue
        io = dtype if gk in ("dx", "ddelta", "dz") else ("f32" if dtype == "f32" else "bf16")
        _check(gk, g[gk], ref[rk], io)


@pytest.mark.parametrize("shape,dtype,gate", [
    ((2, 19, 16, 77), "f32", True),       # N = 16: 8 channels per CTA, ragged last chunk and block
    ((1, 9, 5, 64), "f32", False),        # padded states, two whole chunks
    ((2, 7, 64, 45), "bf16", True),       # N = 64: two states per lane
    ((3, 20, 32, 33), "bf16", False),     # N = 32, one step past a chunk
    ((1, 40, 8, 129), "f32", True),       # N = 8: 16 channels per CTA
    # one consumer warp per SM sub-partition or more: the chunk-start states come from one
    # whole-sequence forward pass that stores them, not from the totals pass and carry scan
    ((1, 4880, 16, 100), "f32", True),    # TMA rows, ragged last chunk
    ((2, 2440, 13, 70), "bf16", False),   # rows not 16-byte aligned (element loads), padded states
    ((1, 5120, 64, 40), "bf16", True),    # 64 states: 16-step tiles, a state every other tile
    ((1, 2440, 16, 96), "f32", True),     # the pass at 2 states a lane; walk split into segments
    # more CTAs than one wave of 3 per SM: the walk at 4 CTAs per SM
    ((2, 4000, 16, 40), "f32", True),
    ((2, 4000, 16, 75), "bf16", False),
])
def test_backward_matches_oracle(shape, dtype, gate):
    p = synth.make_problem(*shape, dtype=dtype, gate=gate, seed=400 + shape[2] + shape[3], A_mode="random")
    g, ref = _run(p, _dy(p, 7))
    _compare(g, ref, dtype)


def test_backward_with_start_state_and_final_state_gradient():
    p = synth.make_problem(2, 24, 16, 100, dtype="f32", gate=True, seed=420, A_mode="random")
    h0 = synth.make_state(2, 24, 16, seed=421)
    dfinal = synth.make_state(2, 24, 16, seed=422)
    g, ref = _run(p, _dy(p, 8), h0=h0, dfinal=dfinal)
    _compare(g, ref, "f32")


def test_backward_whole_pass_states_with_start_state():
    """Chunk-start states from the whole-sequence pass, seeded with a start state."""
    p = synth.make_problem(1, 4880, 16, 72, dtype="f32", gate=True, seed=429, A_mode="random")
    h0 = synth.make_state(1, 4880, 16, seed=430)
    dfinal = synth.make_state(1, 4880, 16, seed=431)
    g, ref = _run(p, _dy(p, 11), h0=h0, dfinal=dfinal)
    _compare(g, ref, "f32")


def test_backward_without_softplus():
    p = synth.make_problem(1, 16, 16, 70, dtype="f32", gate=False, seed=423, delta_softplus=False, delta="slow",
                           use_dt_bias=False, use_D=False)
    g, ref = _run(p, _dy(p, 9))
    _compare(g, ref, "f32")


def test_only_the_final_state_gradient():
    """dy = 0: only dL/dfinal_state drives the adjoint."""
    p = synth.make_problem(2, 8, 16, 50, dtype="f32", gate=False, seed=424, A_mode="random")
    dfinal = synth.make_state(2, 8, 16, seed=425)
    g, ref = _run(p, torch.zeros(2, 8, 50), dfinal=dfinal)
    _compare(g, ref, "f32")


def test_empty_sequence():
    p = synth.make_problem(2, 8, 16, 0, dtype="f32", seed=426)
    dfinal = synth.make_state(2, 8, 16, seed=427).cuda()
    dev = lambda t: None if t is None else t.cuda()
    g = ssm.scan_bwd(dev(p.x), dev(p.delta), dev(p.A), dev(p.B), dev(p.C), dev(p.x), D=dev(p.D),
                     dt_bias=dev(p.dt_bias), dfinal_state=dfinal)
    torch.cuda.synchronize()
    assert torch.equal(g["dinitial_state"], dfinal)
    assert float(g["dA"].abs().max()) == 0.0 and float(g["dD"].abs().max()) == 0.0


@pytest.mark.parametrize("shape", [(4, 1536, 16, 2048), (8, 2048, 16, 4096)], ids=["mid", "large"])
def test_large_workload_sampled(shape):
    """The mid-size (4 x 1536 x 16, 2048 steps) and large-batch (8 x 2048 x 16,
    4096 steps) bf16 shapes, in the launch configurations they get at those
    sizes (the walk at 3 and at 4 CTAs per SM): the per-channel gradients (dx,
    ddelta, dz) of sampled channels against the oracle run on those channels
    alone.  (dA, dB, dC, dD and ddt_bias are sums over all channels or
    batches; the smaller cases above check them.)"""
    p = synth.make_problem(*shape, dtype="bf16", gate=True, seed=428)
    dy = _dy(p, 10)
    dev = lambda t: None if t is None else t.cuda()
    g = ssm.scan_bwd(dev(p.x), dev(p.delta), dev(p.A), dev(p.B), dev(p.C), dev(dy), D=dev(p.D), z=dev(p.z),
                     dt_bias=dev(p.dt_bias))
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    for b, d in [(int(rng.integers(p.batch)), int(rng.integers(p.dim))) for _ in range(6)]:
        sl = lambda t: None if t is None else t[b:b + 1, d:d + 1].contiguous()
        ref = oracle.bwd(sl(p.x).float().numpy(), sl(p.delta).float().numpy(), p.A[d:d + 1].numpy(),
                         p.B[b:b + 1].float().numpy(), p.C[b:b + 1].float().numpy(), sl(dy).float().numpy(),
                         D=p.D[d:d + 1].numpy(), z=sl(p.z).float().numpy(), dt_bias=p.dt_bias[d:d + 1].numpy())
        for gk in ("dx", "ddelta", "dz"):
            _check(f"{gk}[{b},{d}]", g[gk][b, d].float().cpu().numpy(), ref[gk][0, 0], "bf16")
