"""GPU parity of the training pair: the forward that stores the state at the
start of every 32-step chunk (ssm_scan_fwd_ckpt) and the backward that starts
from those checkpoints (ssm_scan_bwd_ckpt).

  * The checkpoints against the fp64 oracle's states at the chunk starts: the
    oracle's serial forward run chunk by chunk, each chunk from the state the
    previous one ended in (entry k is h before step 32 k).  Float32 bound
    |h - h_ref| <= 1e-4 (1 + |h_ref|), the forward's final-state tolerance.
  * y and final_state of the checkpointing forward equal those of the plain
    forward of the same variant bit for bit (the same kernels, with the extra
    stores), and match the oracle.
  * The gradients of the backward from the checkpoints against the oracle's
    backward, with the tolerances of test_parity_bwd.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import synth

from test_parity import assert_close
from test_parity_bwd import _compare, _dy

pytestmark = pytest.mark.gpu

CK = 32


@pytest.fixture(scope="module", autouse=True)
def _built():
    from selective_state_space_02_gb300 import build
    build.build()
    oracle.build()


def _args(p):
    return (p.f32("x"), p.f32("delta"), p.A.numpy(), p.f32("B"), p.f32("C"))


def _kw(p):
    return dict(D=None if p.D is None else p.D.numpy(), z=p.f32("z"),
                dt_bias=None if p.dt_bias is None else p.dt_bias.numpy(), delta_softplus=p.delta_softplus)


def _oracle_chunk_states(p, h0):
    """The oracle's state before step 32 k, k = 0 .. ceil(L / 32) - 1."""
    x, dl, A, B, C = _args(p)
    kw = _kw(p)
    z = kw.pop("z")
    h = np.zeros((p.batch, p.dim, p.dstate)) if h0 is None else h0.double().numpy()
    out = []
    for t0 in range(0, p.seqlen, CK):
        sl = slice(t0, min(t0 + CK, p.seqlen))
        out.append(h.reshape(p.batch * p.dim, p.dstate).copy())
        _, fs = oracle.fwd(x[:, :, sl], dl[:, :, sl], A, B[:, :, sl], C[:, :, sl],
                           z=None if z is None else z[:, :, sl], h0=h, **kw)
        h = fs.reshape(p.batch, p.dim, p.dstate)
    return np.stack(out) if out else np.zeros((0, p.batch * p.dim, p.dstate))


def _dev(p):
    g = lambda t: None if t is None else t.cuda()
    return dict(x=g(p.x), delta=g(p.delta), A=g(p.A), B=g(p.B), C=g(p.C), D=g(p.D), z=g(p.z),
                dt_bias=g(p.dt_bias))


def _fwd(t, p, variant, h0=None, ckpt=True):
    return ssm.scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"], dt_bias=t["dt_bias"],
                        delta_softplus=p.delta_softplus, return_final_state=True, variant=variant,
                        initial_state=h0, return_ckpt=ckpt)


CASES = [
    # batch, dim, dstate, L, dtype, gate, variant
    (2, 40, 16, 300, "f32", True, "fused"),       # ragged last chunk, partial channel block
    (2, 40, 16, 300, "f32", True, "twopass"),     # segment starts between the chunk starts
    (1, 37, 16, 333, "f32", False, "fused"),      # rows not 16-byte aligned: element loads
    (3, 50, 16, 1000, "bf16", True, "twopass"),
    (1, 20, 64, 300, "bf16", True, "fused"),      # 64 states: 16-step tiles, a checkpoint every other tile
    (2, 9, 5, 130, "f32", False, "auto"),         # AUTO would run CHUNKED here: TWOPASS instead
    (1, 4880, 16, 100, "f32", True, "auto"),      # AUTO fused at this size
    (1, 37, 16, 333, "f32", False, "twopass"),    # element loads, segments
    (1, 20, 32, 300, "bf16", True, "fused"),      # 32 states
]


def _ids(c):
    return "x".join(map(str, c[:4])) + f"-{c[4]}-g{int(c[5])}-{c[6]}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_checkpoints_match_oracle(case):
    b, d, n, L, dt, gate, variant = case
    p = synth.make_problem(b, d, n, L, dtype=dt, gate=gate, seed=800 + d + L, A_mode="random")
    t = _dev(p)
    y, fs, ck = _fwd(t, p, variant)
    yp, fsp = _fwd(t, p, "twopass" if variant == "auto" and ssm.select_variant(b, d, n, L, p.torch_dtype) ==
                   "chunked" else variant, ckpt=False)
    torch.cuda.synchronize()
    assert torch.equal(y, yp) and torch.equal(fs, fsp), "the checkpointing forward changed y or the final state"
    yr, fr = oracle.fwd(*_args(p), **_kw(p))
    nch = b * d
    assert_close(y.float().cpu().numpy().reshape(nch, L), yr, dt, "y")
    assert_close(fs.cpu().numpy().reshape(nch, n), fr, "f32", "final_state")
    ref = _oracle_chunk_states(p, None)
    assert ck.shape == ((L + CK - 1) // CK, b, d, n)
    assert_close(ck.cpu().numpy().reshape(ref.shape), ref, "f32", "checkpoints")


@pytest.mark.parametrize("case", [CASES[0], CASES[3], CASES[4], CASES[5], CASES[7], CASES[8]], ids=_ids)
def test_backward_from_checkpoints(case):
    b, d, n, L, dt, gate, variant = case
    p = synth.make_problem(b, d, n, L, dtype=dt, gate=gate, seed=820 + d + L, A_mode="random")
    t = _dev(p)
    dy = _dy(p, 21)
    _, _, ck = _fwd(t, p, variant)
    g = ssm.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], dy.cuda(), D=t["D"], z=t["z"],
                     dt_bias=t["dt_bias"], delta_softplus=p.delta_softplus, ckpt=ck)
    torch.cuda.synchronize()
    ref = oracle.bwd(*_args(p), dy.float().numpy(), **_kw(p))
    _compare(g, ref, dt)


@pytest.mark.parametrize("variant", ["fused", "twopass"])
def test_start_state_through_checkpoints(variant):
    """A start state and a final-state gradient: the forward's checkpoints
    carry the start state (entry 0 is h0), the backward from them gives the
    start state's gradient."""
    p = synth.make_problem(2, 24, 16, 100, dtype="f32", gate=True, seed=830, A_mode="random")
    h0 = synth.make_state(2, 24, 16, seed=831)
    dfinal = synth.make_state(2, 24, 16, seed=832)
    t = _dev(p)
    y, fs, ck = _fwd(t, p, variant, h0=h0.cuda())
    torch.cuda.synchronize()
    assert torch.equal(ck[0].cpu(), h0)
    ref = _oracle_chunk_states(p, h0)
    assert_close(ck.cpu().numpy().reshape(ref.shape), ref, "f32", "checkpoints from h0")
    dy = _dy(p, 22)
    g = ssm.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], dy.cuda(), D=t["D"], z=t["z"],
                     dt_bias=t["dt_bias"], delta_softplus=p.delta_softplus, dfinal_state=dfinal.cuda(), ckpt=ck)
    torch.cuda.synchronize()
    r = oracle.bwd(*_args(p), dy.float().numpy(), h0=h0.numpy(), dfinal=dfinal.numpy(), **_kw(p))
    _compare(g, r, "f32")


@pytest.mark.parametrize("L", [1, 31, 32, 33, 64])
@pytest.mark.parametrize("variant", ["fused", "twopass"])
def test_chunk_edges(L, variant):
    """Sequences of one step, one step short of a chunk, exactly one chunk,
    one step past it, two chunks: the checkpoint count and values, and the
    backward from them."""
    p = synth.make_problem(2, 24, 16, L, dtype="f32", gate=True, seed=850 + L, A_mode="random")
    t = _dev(p)
    y, fs, ck = _fwd(t, p, variant)
    torch.cuda.synchronize()
    ref = _oracle_chunk_states(p, None)
    assert ck.shape == ((L + CK - 1) // CK, 2, 24, 16)
    assert_close(ck.cpu().numpy().reshape(ref.shape), ref, "f32", "checkpoints")
    dy = _dy(p, 25)
    g = ssm.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], dy.cuda(), D=t["D"], z=t["z"],
                     dt_bias=t["dt_bias"], delta_softplus=p.delta_softplus, ckpt=ck)
    torch.cuda.synchronize()
    _compare(g, oracle.bwd(*_args(p), dy.float().numpy(), **_kw(p)), "f32")


def test_refusals():
    p = synth.make_problem(1, 16, 16, 64, dtype="f32", seed=840)
    t = _dev(p)
    with pytest.raises(ssm.ScanError):      # CHUNKED does not store checkpoints
        _fwd(t, p, "chunked")
    _, _, ck = _fwd(t, p, "fused")
    dy = _dy(p, 23).cuda()
    with pytest.raises(ValueError):         # the start state enters through the checkpoints
        ssm.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], dy, D=t["D"], dt_bias=t["dt_bias"],
                     initial_state=torch.zeros(1, 16, 16, device="cuda"), ckpt=ck)
    with pytest.raises(ValueError):         # checkpoints of another length
        ssm.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], dy, D=t["D"], dt_bias=t["dt_bias"],
                     ckpt=ck[:1].contiguous())


def test_mid_workload_training_pair():
    """The mid-size shape (4 x 1536 x 16, 2048 steps, bf16, gate on): every
    checkpoint against the oracle, and the per-channel gradients of sampled
    channels from the backward over the checkpoints against the oracle run on
    those channels alone."""
    p = synth.workload("mid_bf16")
    t = _dev(p)
    y, fs, ck = _fwd(t, p, "auto")
    dy = _dy(p, 24)
    g = ssm.scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], dy.cuda(), D=t["D"], z=t["z"],
                     dt_bias=t["dt_bias"], delta_softplus=p.delta_softplus, ckpt=ck)
    torch.cuda.synchronize()
    ref = _oracle_chunk_states(p, None)
    assert_close(ck.cpu().numpy().reshape(ref.shape), ref, "f32", "checkpoints")
    rng = np.random.default_rng(1)
    from test_parity_bwd import _check
    for b, d in [(int(rng.integers(p.batch)), int(rng.integers(p.dim))) for _ in range(4)]:
        sl = lambda a: None if a is None else a[b:b + 1, d:d + 1].contiguous()
        r = oracle.bwd(sl(p.x).float().numpy(), sl(p.delta).float().numpy(), p.A[d:d + 1].numpy(),
                       p.B[b:b + 1].float().numpy(), p.C[b:b + 1].float().numpy(), sl(dy).float().numpy(),
                       D=p.D[d:d + 1].numpy(), z=sl(p.z).float().numpy(), dt_bias=p.dt_bias[d:d + 1].numpy())
        for gk in ("dx", "ddelta", "dz"):
            _check(f"{gk}[{b},{d}]", g[gk][b, d].float().cpu().numpy(), r[gk][0, 0], "bf16")
