"""Seeded synthetic inputs for the forward selective scan.

This module only draws random numbers and rounds them to the I/O dtype; it
holds none of the scan's arithmetic.  Both the CUDA path (through the public
binding) and the CPU oracle consume what it returns, so they always see
bit-identical inputs.

Distributions follow the workload descriptions: x, z, B, C, D ~ N(0, 1);
A[d, n] = -(n + 1) * a_scale; delta ~ N(0, sigma^2); dt_bias per channel is
the inverse softplus of a target step dt_d, so that softplus(delta + dt_bias)
is centred on dt_d.  For the log-uniform recipe dt_d ~ logU[1e-3, 1e-1] per
channel (the usual Mamba step initialisation); for the slow-decay recipe
dt_d = 1e-3 for every channel and sigma = 0.1.

Draw order (numpy PCG64, one generator per workload seed):
x, delta, z (if gated), B, C, D, dt.
bf16 workloads are drawn in float32 and rounded to bf16 (round to nearest
even); the oracle receives the exact float32 widening of those bf16 values.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

# Named workloads (shapes and recipes of the five benchmark cases).
WORKLOADS = {
    # tiny fp32 scan, final state returned, no gate
    "tiny_f32": dict(batch=1, dim=64, dstate=16, seqlen=256, dtype="f32", gate=False,
                     final_state=True, a_scale=1.0, delta="logu", seed=20261202),
    # mid-size bf16 scan with fp32 state, silu gate on
    "mid_bf16": dict(batch=4, dim=1536, dstate=16, seqlen=2048, dtype="bf16", gate=True,
                     final_state=False, a_scale=1.0, delta="logu", seed=20261203),
    # large-batch bf16 scan, gate on, final state returned
    "large_batch_bf16": dict(batch=8, dim=2048, dstate=16, seqlen=4096, dtype="bf16", gate=True,
                             final_state=True, a_scale=1.0, delta="logu", seed=20261204),
    # long-sequence low-parallelism fp32 scan, slow decay, no gate
    "long_seq_f32": dict(batch=1, dim=768, dstate=16, seqlen=131072, dtype="f32", gate=False,
                         final_state=False, a_scale=1.0, delta="slow", seed=20261205),
    # wide-state bf16 scan, N = 64, gate on
    "wide_state_bf16": dict(batch=2, dim=5120, dstate=64, seqlen=8192, dtype="bf16", gate=True,
                            final_state=False, a_scale=0.25, delta="logu", seed=20261206),
}

# Named decode-step workloads: one token for every sequence of a serving
# batch, the state [batch, dim, dstate] resident on the device.
STEP_WORKLOADS = {
    # 256 sequences x 2048 channels x 16 states, bf16 I/O, gate on
    "decode_bf16": dict(batch=256, dim=2048, dstate=16, seqlen=1, dtype="bf16", gate=True,
                        final_state=True, a_scale=1.0, delta="logu", seed=20261210),
}


@dataclasses.dataclass
class Problem:
    """One seeded problem.  ``io`` tensors are CPU torch tensors in the I/O
    dtype (what the library receives); ``f32`` arrays are their exact float32
    values (what the oracle receives)."""
    batch: int
    dim: int
    dstate: int
    seqlen: int
    dtype: str                     # "f32" or "bf16"
    gate: bool
    final_state: bool
    delta_softplus: bool
    x: torch.Tensor
    delta: torch.Tensor
    z: Optional[torch.Tensor]
    B: torch.Tensor
    C: torch.Tensor
    A: torch.Tensor                # float32 [dim, dstate]
    D: Optional[torch.Tensor]      # float32 [dim]
    dt_bias: Optional[torch.Tensor]  # float32 [dim]

    def f32(self, name):
        t = getattr(self, name)
        if t is None:
            return None
        return t.float().numpy()

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def elems(self) -> int:
        return self.batch * self.dim * self.seqlen


def _inv_softplus(dt: np.ndarray) -> np.ndarray:
    # inverse of log(1 + e^v): v = dt + log(1 - e^-dt); only used to build inputs
    return dt + np.log(-np.expm1(-dt))


def make_problem(batch: int, dim: int, dstate: int, seqlen: int, dtype: str = "f32",
                 gate: bool = False, final_state: bool = True, a_scale: float = 1.0,
                 delta: str = "logu", seed: int = 0, use_D: bool = True,
                 use_dt_bias: bool = True, delta_softplus: bool = True,
                 A_mode: str = "structured", B_zero: bool = False, C_zero: bool = False,
                 x_scale: float = 1.0) -> Problem:
    """Draw one problem.  ``A_mode`` "structured" gives A[d,n] = -(n+1)*a_scale;
    "random" gives A[d,n] = -exp(U[log 0.05, log 16]) (no shared structure)."""
    if dtype not in ("f32", "bf16"):
        raise ValueError(dtype)
    rng = np.random.Generator(np.random.PCG64(seed))
    shp = (batch, dim, seqlen)
    bshp = (batch, dstate, seqlen)
    x = rng.standard_normal(shp, dtype=np.float32) * np.float32(x_scale)
    if delta == "slow":
        dl = rng.standard_normal(shp, dtype=np.float32) * np.float32(0.1)
    else:
        dl = rng.standard_normal(shp, dtype=np.float32)
    z = rng.standard_normal(shp, dtype=np.float32) if gate else None
    Bm = rng.standard_normal(bshp, dtype=np.float32)
    Cm = rng.standard_normal(bshp, dtype=np.float32)
    Dv = rng.standard_normal((dim,), dtype=np.float32)
    if delta == "slow":
        dt = np.full((dim,), 1e-3, np.float64)
    else:
        dt = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=(dim,)))
    dt_bias = _inv_softplus(dt).astype(np.float32)
    if A_mode == "structured":
        A = -(np.arange(1, dstate + 1, dtype=np.float32)[None, :] * np.float32(a_scale))
        A = np.ascontiguousarray(np.broadcast_to(A, (dim, dstate)), dtype=np.float32)
    elif A_mode == "random":
        A = -np.exp(rng.uniform(math.log(0.05), math.log(16.0), size=(dim, dstate))).astype(np.float32)
    else:
        raise ValueError(A_mode)
    if B_zero:
        Bm[...] = 0
    if C_zero:
        Cm[...] = 0
    td = torch.bfloat16 if dtype == "bf16" else torch.float32

    def io(a):
        if a is None:
            return None
        return torch.from_numpy(np.ascontiguousarray(a)).to(td).contiguous()

    return Problem(batch=batch, dim=dim, dstate=dstate, seqlen=seqlen, dtype=dtype, gate=gate,
                   final_state=final_state, delta_softplus=delta_softplus,
                   x=io(x), delta=io(dl), z=io(z), B=io(Bm), C=io(Cm),
                   A=torch.from_numpy(A), D=torch.from_numpy(Dv) if use_D else None,
                   dt_bias=torch.from_numpy(dt_bias) if use_dt_bias else None)


def workload(name: str, **overrides) -> Problem:
    """The named benchmark workload (see ``WORKLOADS``)."""
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    return make_problem(**cfg)


def min_bytes(p: Problem) -> int:
    """Bytes that must cross HBM at least once: x, delta, (z), y in the I/O
    dtype; B, C in the I/O dtype; A, D, dt_bias in float32; the final state in
    float32 when it is returned."""
    e = 2 if p.dtype == "bf16" else 4
    n = p.batch * p.dim * p.seqlen * e * (3 + (1 if p.z is not None else 0))
    n += 2 * p.batch * p.dstate * p.seqlen * e
    n += p.dim * p.dstate * 4
    n += p.dim * 4 * ((1 if p.D is not None else 0) + (1 if p.dt_bias is not None else 0))
    if p.final_state:
        n += p.batch * p.dim * p.dstate * 4
    return n


def make_state(batch: int, dim: int, dstate: int, seed: int = 0, scale: float = 1.0) -> torch.Tensor:
    """A start state [batch, dim, dstate] float32 drawn N(0, scale^2): the
    boundary state a resumed segment or a decode session begins from."""
    rng = np.random.Generator(np.random.PCG64(seed))
    s = rng.standard_normal((batch, dim, dstate), dtype=np.float32) * np.float32(scale)
    return torch.from_numpy(np.ascontiguousarray(s))


def step_inputs(p: Problem, t: int) -> dict:
    """The inputs of token t of problem p for a single decode step: x, delta
    and z as [batch, dim], B and C as [batch, dstate] (contiguous copies in the
    I/O dtype), plus the per-channel parameters."""
    col = lambda a: None if a is None else a[:, :, t].contiguous()
    return dict(x=col(p.x), delta=col(p.delta), z=col(p.z), B=col(p.B), C=col(p.C),
                A=p.A, D=p.D, dt_bias=p.dt_bias)


def step_min_bytes(p: Problem) -> int:
    """Bytes one decode step must move at least: the float32 state read and
    written once, x, delta, (z) and y in the I/O dtype, B and C of the token,
    A, D and dt_bias."""
    e = 2 if p.dtype == "bf16" else 4
    n = 2 * p.batch * p.dim * p.dstate * 4
    n += p.batch * p.dim * e * (3 + (1 if p.z is not None else 0))
    n += 2 * p.batch * p.dstate * e
    n += p.dim * p.dstate * 4
    n += p.dim * 4 * ((1 if p.D is not None else 0) + (1 if p.dt_bias is not None else 0))
    return n


def make_conv(dim: int, width: int = 4, seed: int = 0):
    """Depthwise causal convolution parameters: weight [dim, width] and bias
    [dim], float32, drawn U(-1/sqrt(width), 1/sqrt(width)) (the usual fan-in
    scale for a depthwise filter of `width` taps)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    s = 1.0 / math.sqrt(width)
    w = rng.uniform(-s, s, size=(dim, width)).astype(np.float32)
    b = rng.uniform(-s, s, size=(dim,)).astype(np.float32)
    return torch.from_numpy(w), torch.from_numpy(b)


def make_conv_state(batch: int, dim: int, width: int = 4, dtype: str = "f32", seed: int = 0) -> torch.Tensor:
    """The width-1 inputs that preceded a segment, [batch, dim, width-1], in the I/O dtype."""
    rng = np.random.Generator(np.random.PCG64(seed))
    s = rng.standard_normal((batch, dim, width - 1), dtype=np.float32)
    t = torch.from_numpy(np.ascontiguousarray(s))
    return t.to(torch.bfloat16) if dtype == "bf16" else t
