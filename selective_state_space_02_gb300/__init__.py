"""GB300-native forward selective scan (Mamba-style SSM), sm_103a.

Thin PyTorch binding over libssmscan.so (include/ssm_scan.h): it checks
dtypes, devices and contiguity, allocates outputs with torch, and passes raw
pointers and the current CUDA stream.  Every step of the scan runs in the
library's kernels; there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _native
from ._native import ScanError, VARIANTS, SSM_BF16, SSM_F32

__all__ = ["scan_fwd", "scan_fwd_conv", "conv_scan_workspace_size", "scan_fwd_host", "scan_step", "scan_bwd", "conv1d", "select_variant", "workspace_size", "ScanError",
           "VARIANTS", "host_buffer_size"]


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return SSM_F32
    if t == torch.bfloat16:
        return SSM_BF16
    raise TypeError(f"unsupported I/O dtype {t}; use float32 or bfloat16")


def _variant_code(variant) -> int:
    if isinstance(variant, str):
        return VARIANTS[variant]
    return int(variant)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t: torch.Tensor) -> int:
    """The handle of the current CUDA stream on t's device (the cheap lookup
    where this PyTorch has it: a decode step pays it once per layer and token)."""
    if _raw_stream is not None:
        return _raw_stream(t.get_device())
    return torch.cuda.current_stream(t.device).cuda_stream


def select_variant(batch: int, dim: int, dstate: int, seqlen: int, dtype=torch.float32) -> str:
    v = _native.load().ssm_scan_select_variant(batch, dim, dstate, seqlen, _dtype_code(dtype))
    if v < 0:
        _native.check(v)
    return _native.VARIANT_NAMES[v]


def workspace_size(batch: int, dim: int, dstate: int, seqlen: int, dtype=torch.float32,
                   variant="auto") -> int:
    n = _native.load().ssm_scan_fwd_workspace_size(batch, dim, dstate, seqlen, _dtype_code(dtype),
                                                   _variant_code(variant))
    if n == (1 << 64) - 1:
        raise ScanError(-2, "invalid sizes")
    return n


def host_buffer_size(batch, dim, dstate, seqlen, dtype, has_D, has_z, has_dt_bias,
                     has_final_state, variant="auto") -> int:
    n = _native.load().ssm_scan_fwd_host_buffer_size(batch, dim, dstate, seqlen, _dtype_code(dtype),
                                                     int(has_D), int(has_z), int(has_dt_bias),
                                                     int(has_final_state), _variant_code(variant))
    if n == (1 << 64) - 1:
        raise ScanError(-2, "invalid sizes")
    return n


def _check_inputs(x, delta, A, B, C, D, z, dt_bias, device_type):
    io = x.dtype
    _dtype_code(io)
    ios = (("x", x), ("delta", delta), ("B", B), ("C", C), ("z", z))
    f32s = (("A", A), ("D", D), ("dt_bias", dt_bias))
    for name, t in ios:
        if t is not None and t.dtype != io:
            raise TypeError(f"{name} has dtype {t.dtype}, expected {io}")
    for name, t in f32s:
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    for name, t in ios + f32s:
        if t is None:
            continue
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device.type != device_type:
            raise ValueError(f"{name} must be on {device_type}")
    if x.dim() != 3:
        raise ValueError("x must be [batch, dim, seqlen]")
    batch, dim, L = x.shape
    N = A.shape[1]
    if delta.shape != x.shape or (z is not None and z.shape != x.shape):
        raise ValueError("delta and z must have the shape of x")
    if A.shape != (dim, N) or B.shape != (batch, N, L) or C.shape != (batch, N, L):
        raise ValueError("A must be [dim, dstate]; B and C [batch, dstate, seqlen]")
    for name, t in (("D", D), ("dt_bias", dt_bias)):
        if t is not None and t.shape != (dim,):
            raise ValueError(f"{name} must be [dim]")
    return batch, dim, N, L


def scan_fwd(x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
             C: torch.Tensor, D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
             dt_bias: Optional[torch.Tensor] = None, delta_softplus: bool = True,
             return_final_state: bool = False, variant="auto", y: Optional[torch.Tensor] = None,
             final_state: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
             initial_state: Optional[torch.Tensor] = None, return_ckpt: bool = False):
    """Forward selective scan on CUDA tensors, launched on the current stream.

    x, delta, z: [batch, dim, L]; B, C: [batch, dstate, L] (float32 or
    bfloat16, all the same); A: [dim, dstate], D, dt_bias: [dim] (float32).
    Returns y (same dtype as x), or (y, final_state [batch, dim, dstate]
    float32) when ``return_final_state``.  ``y``, ``final_state`` and
    ``workspace`` may be given to avoid allocations.  ``initial_state``
    [batch, dim, dstate] float32 starts the recurrence from that state (a
    resumed segment); ``final_state`` may be the same tensor to advance it in
    place.  With ``return_ckpt`` the forward also stores the state at the
    start of every 32-step chunk (ssm_scan_fwd_ckpt), returned last as a
    float32 [ceil(L / 32), batch, dim, dstate] tensor for ``scan_bwd(...,
    ckpt=...)``.
    """
    batch, dim, N, L = _check_inputs(x, delta, A, B, C, D, z, dt_bias, "cuda")
    if initial_state is not None:
        if initial_state.dtype != torch.float32:
            raise TypeError("initial_state must be float32")
        if not initial_state.is_contiguous() or initial_state.device.type != "cuda":
            raise ValueError("initial_state must be a contiguous CUDA tensor")
        if initial_state.shape != (batch, dim, N):
            raise ValueError("initial_state must be [batch, dim, dstate]")
    lib = _native.load()
    code = _dtype_code(x.dtype)
    v = _variant_code(variant)
    if y is None:
        y = torch.empty_like(x)
    if return_final_state and final_state is None:
        final_state = torch.empty((batch, dim, N), dtype=torch.float32, device=x.device)
    ws_bytes = (lib.ssm_scan_fwd_ckpt_workspace_size if return_ckpt else lib.ssm_scan_fwd_workspace_size)(
        batch, dim, N, L, code, v)
    if ws_bytes == (1 << 64) - 1:
        raise ScanError(-2, "invalid sizes or a variant without checkpoints")
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    stream = _stream(x)
    fs = _ptr(final_state) if return_final_state else None
    ws = _ptr(workspace) if ws_bytes else None
    if return_ckpt:
        ckpt = torch.empty(((L + 31) // 32, batch, dim, N), dtype=torch.float32, device=x.device)
        rc = lib.ssm_scan_fwd_ckpt(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                   _ptr(dt_bias), int(bool(delta_softplus)), _ptr(initial_state), _ptr(y), fs,
                                   _ptr(ckpt), batch, dim, N, L, code, ws, ws_bytes, stream, v)
        _native.check(rc)
        return (y, final_state, ckpt) if return_final_state else (y, ckpt)
    if initial_state is None:
        rc = lib.ssm_scan_fwd_variant(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                      _ptr(dt_bias), int(bool(delta_softplus)), _ptr(y), fs,
                                      batch, dim, N, L, code, ws, ws_bytes, stream, v)
    else:
        rc = lib.ssm_scan_fwd_from_state(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                                         _ptr(dt_bias), int(bool(delta_softplus)), _ptr(initial_state),
                                         _ptr(y), fs, batch, dim, N, L, code, ws, ws_bytes, stream, v)
    _native.check(rc)
    if return_final_state:
        return y, final_state
    return y


CONV_MODES = {"auto": -1, "separate": 0, "fused": 1}


def conv_scan_workspace_size(batch: int, dim: int, dstate: int, seqlen: int, conv_width: int,
                             dtype=torch.float32, mode="auto") -> int:
    n = _native.load().ssm_scan_fwd_conv_workspace_size(batch, dim, dstate, seqlen, conv_width, _dtype_code(dtype),
                                                        CONV_MODES[mode])
    if n == (1 << 64) - 1:
        raise ScanError(-2, "invalid sizes or mode")
    return n


def scan_fwd_conv(x: torch.Tensor, conv_weight: torch.Tensor, delta: torch.Tensor, A: torch.Tensor,
                  B: torch.Tensor, C: torch.Tensor, conv_bias: Optional[torch.Tensor] = None,
                  conv_state: Optional[torch.Tensor] = None, D: Optional[torch.Tensor] = None,
                  z: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
                  delta_softplus: bool = True, return_final_state: bool = False, mode="auto",
                  y: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None):
    """Causal depthwise convolution + SiLU of x (include/ssm_conv.h) feeding
    the forward selective scan, in one call on CUDA tensors.  x is the raw
    input [batch, dim, L]; conv_weight [dim, width] and conv_bias [dim]
    float32; conv_state [batch, dim, width-1] in x's dtype (the inputs that
    preceded the sequence).  ``mode`` "fused" runs the convolution inside the
    scan kernel (width <= 4), "separate" writes its output to the workspace
    first, "auto" picks.  Other arguments and the result as in scan_fwd."""
    batch, dim, N, L = _check_inputs(x, delta, A, B, C, D, z, dt_bias, "cuda")
    if conv_weight.dtype != torch.float32 or conv_weight.dim() != 2 or conv_weight.shape[0] != dim:
        raise ValueError("conv_weight must be float32 [dim, width]")
    width = conv_weight.shape[1]
    if conv_bias is not None and (conv_bias.dtype != torch.float32 or conv_bias.shape != (dim,)):
        raise ValueError("conv_bias must be float32 [dim]")
    if conv_state is not None and (conv_state.dtype != x.dtype or conv_state.shape != (batch, dim, width - 1)):
        raise ValueError("conv_state must be [batch, dim, width-1] in x's dtype")
    for name, t in (("conv_weight", conv_weight), ("conv_bias", conv_bias), ("conv_state", conv_state)):
        if t is not None and (not t.is_contiguous() or t.device.type != "cuda"):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    lib = _native.load()
    code = _dtype_code(x.dtype)
    m = CONV_MODES[mode]
    if y is None:
        y = torch.empty_like(x)
    if return_final_state and final_state is None:
        final_state = torch.empty((batch, dim, N), dtype=torch.float32, device=x.device)
    ws_bytes = lib.ssm_scan_fwd_conv_workspace_size(batch, dim, N, L, width, code, m)
    if ws_bytes == (1 << 64) - 1:
        raise ScanError(-8, "this convolution width cannot run fused")
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    stream = _stream(x)
    rc = lib.ssm_scan_fwd_conv(_ptr(x), _ptr(conv_weight), _ptr(conv_bias), _ptr(conv_state), width,
                               _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
                               int(bool(delta_softplus)), _ptr(y),
                               _ptr(final_state) if return_final_state else None,
                               batch, dim, N, L, code, _ptr(workspace) if ws_bytes else None, ws_bytes, stream, m)
    _native.check(rc)
    if return_final_state:
        return y, final_state
    return y


def scan_fwd_host(x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor,
                  C: torch.Tensor, D=None, z=None, dt_bias=None, delta_softplus: bool = True,
                  y: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
                  device_buffer: Optional[torch.Tensor] = None, variant="auto", stream=None):
    """End-to-end call on CPU tensors (pinned memory recommended): copies the
    inputs to the GPU, runs the scan and copies y (and final_state, if a
    tensor is given) back before returning.  ``device_buffer`` is a CUDA
    uint8 tensor of at least ``host_buffer_size(...)`` bytes."""
    batch, dim, N, L = _check_inputs(x, delta, A, B, C, D, z, dt_bias, "cpu")
    lib = _native.load()
    code = _dtype_code(x.dtype)
    v = _variant_code(variant)
    if y is None:
        y = torch.empty_like(x)
    need = lib.ssm_scan_fwd_host_buffer_size(batch, dim, N, L, code, int(D is not None),
                                             int(z is not None), int(dt_bias is not None),
                                             int(final_state is not None), v)
    if device_buffer is None or device_buffer.numel() < need:
        device_buffer = torch.empty(need, dtype=torch.uint8, device="cuda")
    if stream is None:
        stream = torch.cuda.current_stream()
    rc = lib.ssm_scan_fwd_host(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                               _ptr(dt_bias), int(bool(delta_softplus)), _ptr(y), _ptr(final_state),
                               batch, dim, N, L, code, _ptr(device_buffer), need, stream.cuda_stream, v)
    _native.check(rc)
    return y


def scan_step(state: torch.Tensor, x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor,
              B: torch.Tensor, C: torch.Tensor, D: Optional[torch.Tensor] = None,
              z: Optional[torch.Tensor] = None, dt_bias: Optional[torch.Tensor] = None,
              delta_softplus: bool = True, y: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode step on CUDA tensors (include/ssm_step.h): advances
    ``state`` [batch, dim, dstate] float32 in place by one token and returns
    y [batch, dim].  x, delta, z: [batch, dim]; B, C: [batch, dstate] (float32
    or bfloat16, all the same); A: [dim, dstate], D, dt_bias: [dim] float32."""
    # (the checks use the tensors' cheapest attributes: a decode loop calls
    # this once per layer and token, and the kernel takes about 15 us)
    io = x.dtype
    code = _dtype_code(io)
    for name, t in (("delta", delta), ("B", B), ("C", C), ("z", z)):
        if t is not None and t.dtype != io:
            raise TypeError(f"{name} has dtype {t.dtype}, expected {io}")
    for name, t in (("state", state), ("A", A), ("D", D), ("dt_bias", dt_bias)):
        if t is not None and t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    for name, t in (("state", state), ("x", x), ("delta", delta), ("A", A), ("B", B), ("C", C),
                    ("D", D), ("z", z), ("dt_bias", dt_bias)):
        if t is not None and not (t.is_cuda and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if x.dim() != 2:
        raise ValueError("x must be [batch, dim]")
    batch, dim = x.shape
    N = A.shape[1]
    if state.shape != (batch, dim, N) or delta.shape != x.shape or (z is not None and z.shape != x.shape):
        raise ValueError("state must be [batch, dim, dstate]; delta and z [batch, dim]")
    if A.shape != (dim, N) or B.shape != (batch, N) or C.shape != (batch, N):
        raise ValueError("A must be [dim, dstate]; B and C [batch, dstate]")
    if y is None:
        y = torch.empty_like(x)
    lib = _native._lib or _native.load()
    rc = lib.ssm_scan_step(_ptr(state), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                           _ptr(z), _ptr(dt_bias), int(bool(delta_softplus)), _ptr(y), batch, dim,
                           N, code, _stream(x))
    _native.check(rc)
    return y


def scan_bwd(x: torch.Tensor, delta: torch.Tensor, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor,
             dy: torch.Tensor, D: Optional[torch.Tensor] = None, z: Optional[torch.Tensor] = None,
             dt_bias: Optional[torch.Tensor] = None, delta_softplus: bool = True,
             initial_state: Optional[torch.Tensor] = None, dfinal_state: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, ckpt: Optional[torch.Tensor] = None) -> dict:
    """Gradients of the forward (include/ssm_bwd.h) on CUDA tensors, for a
    loss with dL/dy = dy (dtype of x) and dL/dfinal_state = dfinal_state
    (float32, optional).  Returns a dict: dx, ddelta, dz (dtype of x; dz only
    with z), dA, dB, dC, dD (only with D), ddt_bias (only with dt_bias) and
    dinitial_state (float32).  ``ckpt``: the checkpoints of ``scan_fwd(...,
    return_ckpt=True)`` over the same inputs (ssm_scan_bwd_ckpt); the start
    state then enters through them, so ``initial_state`` must be None."""
    batch, dim, N, L = _check_inputs(x, delta, A, B, C, D, z, dt_bias, "cuda")
    if dy.dtype != x.dtype or dy.shape != x.shape or not dy.is_contiguous():
        raise ValueError("dy must be a contiguous tensor like x")
    for name, t in (("initial_state", initial_state), ("dfinal_state", dfinal_state)):
        if t is not None and (t.dtype != torch.float32 or t.shape != (batch, dim, N) or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float32 [batch, dim, dstate] tensor")
    if ckpt is not None:
        if initial_state is not None:
            raise ValueError("with ckpt the start state enters through the checkpoints: initial_state must be None")
        if (ckpt.dtype != torch.float32 or ckpt.shape != ((L + 31) // 32, batch, dim, N)
                or not ckpt.is_contiguous() or ckpt.device != x.device):
            raise ValueError("ckpt must be the contiguous float32 [ceil(L / 32), batch, dim, dstate] "
                             "checkpoints of scan_fwd(..., return_ckpt=True)")
    lib = _native.load()
    code = _dtype_code(x.dtype)
    f32 = dict(dtype=torch.float32, device=x.device)
    g = dict(dx=torch.empty_like(x), ddelta=torch.empty_like(x), dz=torch.empty_like(x) if z is not None else None,
             dA=torch.empty((dim, N), **f32), dB=torch.empty((batch, N, L), **f32),
             dC=torch.empty((batch, N, L), **f32), dD=torch.empty((dim,), **f32) if D is not None else None,
             ddt_bias=torch.empty((dim,), **f32) if dt_bias is not None else None,
             dinitial_state=torch.empty((batch, dim, N), **f32))
    ws_bytes = (lib.ssm_scan_bwd_ckpt_workspace_size if ckpt is not None else lib.ssm_scan_bwd_workspace_size)(
        batch, dim, N, L, code)
    if ws_bytes == (1 << 64) - 1:
        raise ScanError(-2, "invalid sizes")
    if ws_bytes and (workspace is None or workspace.numel() * workspace.element_size() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    entry = lib.ssm_scan_bwd_ckpt if ckpt is not None else lib.ssm_scan_bwd
    rc = entry(_ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias),
               int(bool(delta_softplus)), _ptr(ckpt if ckpt is not None else initial_state), _ptr(dy),
               _ptr(dfinal_state), _ptr(g["dx"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
               _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["ddt_bias"]), _ptr(g["dinitial_state"]),
               batch, dim, N, L, code, _ptr(workspace) if ws_bytes else None, ws_bytes,
               _stream(x))
    _native.check(rc)
    return g


def conv1d(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor] = None,
           state_in: Optional[torch.Tensor] = None, silu: bool = True, y: Optional[torch.Tensor] = None,
           state_out: Optional[torch.Tensor] = None, return_state: bool = False):
    """Causal depthwise convolution (+ SiLU) on CUDA tensors
    (include/ssm_conv.h).  x: [batch, dim, L] float32 or bfloat16; weight:
    [dim, width] and bias: [dim] float32; state_in / state_out: [batch, dim,
    width-1] in the dtype of x.  Returns y, or (y, state_out) when
    ``return_state``."""
    code = _dtype_code(x.dtype)
    if x.dim() != 3:
        raise ValueError("x must be [batch, dim, seqlen]")
    batch, dim, L = x.shape
    if weight.dtype != torch.float32 or weight.dim() != 2 or weight.shape[0] != dim:
        raise ValueError("weight must be float32 [dim, width]")
    width = weight.shape[1]
    if bias is not None and (bias.dtype != torch.float32 or bias.shape != (dim,)):
        raise ValueError("bias must be float32 [dim]")
    for name, t in (("state_in", state_in), ("state_out", state_out)):
        if t is not None and (t.dtype != x.dtype or t.shape != (batch, dim, width - 1)):
            raise ValueError(f"{name} must be [batch, dim, width-1] in the dtype of x")
    for name, t in (("x", x), ("weight", weight), ("bias", bias), ("state_in", state_in), ("state_out", state_out)):
        if t is not None and (not t.is_contiguous() or t.device.type != "cuda"):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if y is None:
        y = torch.empty_like(x)
    if return_state and state_out is None:
        state_out = torch.empty((batch, dim, width - 1), dtype=x.dtype, device=x.device)
    rc = _native.load().ssm_conv1d_fwd(_ptr(x), _ptr(weight), _ptr(bias), _ptr(state_in), _ptr(y),
                                       _ptr(state_out), int(bool(silu)), batch, dim, L, width, code,
                                       _stream(x))
    _native.check(rc)
    return (y, state_out) if return_state else y
