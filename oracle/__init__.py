"""Serial fp64 CPU oracle for the forward selective scan.

TEST INFRASTRUCTURE ONLY: tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library under
``selective_state_space_02_gb300`` never does.  The oracle shares no code with
the CUDA path.  It is plain C (``ssm_oracle.c``) compiled with gcc and loaded
through ctypes; every function follows one passage of the source pages, cited
in the C file:

  [P1] "Mamba hardware-aware parallel associative scan" (pwwt.cn/news/6375169)
  [P3] "Mamba (part 2): parallel scan and hardware-aware optimisation"
       (scwacadex.pages.dev, blog8_mamba_parallel_scan)

Pins (checked by ``tests/test_oracle_*.py`` without a GPU): associativity and
identity of the composition, brute-force unrolled sums, the geometric-series
closed form, the prefix-sum special case, the impulse response, agreement of
the serial / Hillis-Steele / Blelloch / chunked orderings, and the numbers
the pages print for decay underflow.  Parity of the full forward against
printed outputs is not possible (the pages print none); it is pinned by those
identities instead.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB = os.path.join(_HERE, "libssm_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_lp = ctypes.POINTER(ctypes.c_long)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain IEEE double: no fast-math and no
    floating-point contraction, so rounding is the same on every host)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.ssm_oracle_compose.argtypes = [ctypes.c_double] * 4 + [_dp, _dp]
            lib.ssm_oracle_compose.restype = None
            for name in ("ssm_oracle_scan_serial",):
                getattr(lib, name).argtypes = [_dp, _dp, ctypes.c_long, _dp, _dp]
                getattr(lib, name).restype = None
            for name in ("ssm_oracle_scan_hillis_steele", "ssm_oracle_scan_blelloch"):
                getattr(lib, name).argtypes = [_dp, _dp, ctypes.c_long, _dp, _dp]
                getattr(lib, name).restype = ctypes.c_int
            lib.ssm_oracle_scan_chunked.argtypes = [_dp, _dp, ctypes.c_long, ctypes.c_long,
                                                    ctypes.c_double, _dp, _dp]
            lib.ssm_oracle_scan_chunked.restype = ctypes.c_int
            lib.ssm_oracle_softplus.argtypes = [ctypes.c_double]
            lib.ssm_oracle_softplus.restype = ctypes.c_double
            lib.ssm_oracle_silu.argtypes = [ctypes.c_double]
            lib.ssm_oracle_silu.restype = ctypes.c_double
            lib.ssm_oracle_fwd.argtypes = [_fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, ctypes.c_int,
                                           _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                           ctypes.c_long, _lp, ctypes.c_long, ctypes.c_int]
            lib.ssm_oracle_fwd.restype = ctypes.c_int
            lib.ssm_oracle_fwd_from.argtypes = [_fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, ctypes.c_int, _dp,
                                                _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                                ctypes.c_long, _lp, ctypes.c_long, ctypes.c_int]
            lib.ssm_oracle_fwd_from.restype = ctypes.c_int
            lib.ssm_oracle_step.argtypes = [_dp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, ctypes.c_int, _dp,
                                            ctypes.c_long, ctypes.c_long, ctypes.c_long]
            lib.ssm_oracle_step.restype = ctypes.c_int
            lib.ssm_oracle_bwd.argtypes = [_fp] * 8 + [ctypes.c_int] + [_dp] * 12 + [ctypes.c_long] * 4
            lib.ssm_oracle_bwd.restype = ctypes.c_int
            lib.ssm_oracle_conv1d.argtypes = [_fp, _fp, _fp, _fp, ctypes.c_int, _dp, _dp] + [ctypes.c_long] * 4
            lib.ssm_oracle_conv1d.restype = ctypes.c_int
            lib.ssm_oracle_pairs.argtypes = [_fp, _fp, _fp, _fp, _fp, ctypes.c_int,
                                             ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                             ctypes.c_long, ctypes.c_long, ctypes.c_long, _dp, _dp]
            lib.ssm_oracle_pairs.restype = ctypes.c_int
            lib.ssm_oracle_max_threads.argtypes = []
            lib.ssm_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _ptr(a, typ):
    if a is None:
        return ctypes.cast(None, typ)
    return a.ctypes.data_as(typ)


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def compose(a2, b2, a1, b1):
    """(a2,b2) o (a1,b1): apply step 1, then step 2."""
    lib = _load()
    a = ctypes.c_double()
    b = ctypes.c_double()
    lib.ssm_oracle_compose(a2, b2, a1, b1, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def _scan(fn, a, b):
    a = _f64(a)
    b = _f64(b)
    L = a.shape[0]
    A = np.empty(L, np.float64)
    B = np.empty(L, np.float64)
    rc = fn(_ptr(a, _dp), _ptr(b, _dp), L, _ptr(A, _dp), _ptr(B, _dp))
    if rc not in (None, 0):
        raise RuntimeError(f"oracle scan failed: {rc}")
    return A, B


def scan_serial(a, b):
    return _scan(_load().ssm_oracle_scan_serial, a, b)


def scan_hillis_steele(a, b):
    return _scan(_load().ssm_oracle_scan_hillis_steele, a, b)


def scan_blelloch(a, b):
    return _scan(_load().ssm_oracle_scan_blelloch, a, b)


def scan_chunked(a, b, chunk, h0=0.0):
    """Two-pass chunked scan: returns (h[t] for every t, state at each chunk end)."""
    a = _f64(a)
    b = _f64(b)
    L = a.shape[0]
    K = (L + chunk - 1) // chunk
    h = np.empty(L, np.float64)
    bd = np.empty(max(K, 1), np.float64)
    rc = _load().ssm_oracle_scan_chunked(_ptr(a, _dp), _ptr(b, _dp), L, chunk, float(h0),
                                         _ptr(h, _dp), _ptr(bd, _dp))
    if rc != 0:
        raise RuntimeError(f"oracle chunked scan failed: {rc}")
    return h, bd[:K]


def softplus(v: float) -> float:
    return _load().ssm_oracle_softplus(float(v))


def silu(z: float) -> float:
    return _load().ssm_oracle_silu(float(z))


def max_threads() -> int:
    return _load().ssm_oracle_max_threads()


def fwd(x, delta, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True,
        channels=None, nthreads=0, return_final_state=True, h0=None):
    """Serial fp64 forward selective scan.

    x, delta, z: [batch, dim, L]; B, C: [batch, dstate, L]; A: [dim, dstate];
    D, dt_bias: [dim].  Arrays are read as float32 (bf16 inputs must be passed
    as their exact float32 widening).  ``channels``: optional list of flat
    channel indices b*dim+d; the result rows follow that order.  ``h0``:
    optional start state [batch, dim, dstate] (read as float64; zeros if None).
    Returns (y [nchan, L] float64, final_state [nchan, dstate] float64 or None).
    """
    x = _f32(x)
    delta = _f32(delta)
    A = _f32(A)
    B = _f32(B)
    C = _f32(C)
    D = _f32(D)
    z = _f32(z)
    dt_bias = _f32(dt_bias)
    batch, dim, L = x.shape
    dstate = A.shape[1]
    assert delta.shape == x.shape and B.shape == (batch, dstate, L) and C.shape == B.shape
    assert A.shape == (dim, dstate)
    if z is not None:
        assert z.shape == x.shape
    if h0 is not None:
        h0 = _f64(h0)
        assert h0.shape == (batch, dim, dstate)
    if channels is None:
        chan = None
        nchan = batch * dim
    else:
        chan = np.ascontiguousarray(np.asarray(channels, dtype=np.int64)).astype(np.int64)
        nchan = chan.shape[0]
    y = np.empty((nchan, L), np.float64)
    fs = np.empty((nchan, dstate), np.float64) if return_final_state else None
    lp = ctypes.cast(None, _lp) if chan is None else chan.ctypes.data_as(_lp)
    rc = _load().ssm_oracle_fwd_from(_ptr(x, _fp), _ptr(delta, _fp), _ptr(A, _fp), _ptr(B, _fp),
                                     _ptr(C, _fp), _ptr(D, _fp), _ptr(z, _fp), _ptr(dt_bias, _fp),
                                     int(bool(delta_softplus)), _ptr(h0, _dp), _ptr(y, _dp),
                                     _ptr(fs, _dp) if fs is not None else ctypes.cast(None, _dp),
                                     batch, dim, dstate, L, lp, nchan, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle forward failed: {rc}")
    return y, fs


def step(state, x, delta, A, B, C, D=None, z=None, dt_bias=None, delta_softplus=True):
    """One token of the recurrence (decode mode), fp64.

    state: [batch, dim, dstate] (read as float64, not modified); x, delta, z:
    [batch, dim]; B, C: [batch, dstate]; A: [dim, dstate]; D, dt_bias: [dim].
    Returns (new_state [batch, dim, dstate] float64, y [batch, dim] float64).
    """
    h = np.array(state, dtype=np.float64, copy=True, order="C")
    x = _f32(x)
    delta = _f32(delta)
    A = _f32(A)
    B = _f32(B)
    C = _f32(C)
    D = _f32(D)
    z = _f32(z)
    dt_bias = _f32(dt_bias)
    batch, dim = x.shape
    dstate = A.shape[1]
    assert h.shape == (batch, dim, dstate) and delta.shape == x.shape
    assert B.shape == (batch, dstate) and C.shape == B.shape and A.shape == (dim, dstate)
    y = np.empty((batch, dim), np.float64)
    rc = _load().ssm_oracle_step(_ptr(h, _dp), _ptr(x, _fp), _ptr(delta, _fp), _ptr(A, _fp), _ptr(B, _fp),
                                 _ptr(C, _fp), _ptr(D, _fp), _ptr(z, _fp), _ptr(dt_bias, _fp),
                                 int(bool(delta_softplus)), _ptr(y, _dp), batch, dim, dstate)
    if rc != 0:
        raise RuntimeError(f"oracle step failed: {rc}")
    return h, y


def bwd(x, delta, A, B, C, dy, D=None, z=None, dt_bias=None, delta_softplus=True, h0=None, dfinal=None):
    """Gradients of the forward for a loss with dL/dy = dy [batch, dim, L]
    and dL/dfinal_state = dfinal [batch, dim, dstate] (None: zero), fp64.
    Returns a dict with dx, ddelta, dz (None without z), dA, dB, dC, dD,
    ddt_bias and dh0 (float64 arrays in the shapes of the inputs)."""
    x = _f32(x)
    delta = _f32(delta)
    A = _f32(A)
    B = _f32(B)
    C = _f32(C)
    D = _f32(D)
    z = _f32(z)
    dt_bias = _f32(dt_bias)
    batch, dim, L = x.shape
    dstate = A.shape[1]
    dy = _f64(dy)
    assert dy.shape == x.shape
    if h0 is not None:
        h0 = _f64(h0)
        assert h0.shape == (batch, dim, dstate)
    if dfinal is not None:
        dfinal = _f64(dfinal)
        assert dfinal.shape == (batch, dim, dstate)
    out = dict(dx=np.empty(x.shape), ddelta=np.empty(x.shape), dz=np.empty(x.shape) if z is not None else None,
               dA=np.empty(A.shape), dB=np.empty(B.shape), dC=np.empty(C.shape), dD=np.empty((dim,)),
               ddt_bias=np.empty((dim,)), dh0=np.empty((batch, dim, dstate)))
    rc = _load().ssm_oracle_bwd(_ptr(x, _fp), _ptr(delta, _fp), _ptr(A, _fp), _ptr(B, _fp), _ptr(C, _fp),
                                _ptr(D, _fp), _ptr(z, _fp), _ptr(dt_bias, _fp), int(bool(delta_softplus)),
                                _ptr(h0, _dp), _ptr(dy, _dp), _ptr(dfinal, _dp),
                                *[_ptr(out[k], _dp) for k in ("dx", "ddelta", "dA", "dB", "dC", "dD", "dz",
                                                              "ddt_bias", "dh0")],
                                batch, dim, dstate, L)
    if rc != 0:
        raise RuntimeError(f"oracle backward failed: {rc}")
    return out


def conv1d(x, w, bias=None, state_in=None, silu=True):
    """Causal depthwise convolution (K = w.shape[1] taps) with optional bias,
    start history state_in [batch, dim, K-1] and SiLU, fp64.
    Returns (y [batch, dim, L] float64, state_out [batch, dim, K-1] float64)."""
    x = _f32(x)
    w = _f32(w)
    bias = _f32(bias)
    state_in = _f32(state_in)
    batch, dim, L = x.shape
    K = w.shape[1]
    assert w.shape == (dim, K) and (bias is None or bias.shape == (dim,))
    assert state_in is None or state_in.shape == (batch, dim, K - 1)
    y = np.empty((batch, dim, L))
    st = np.empty((batch, dim, max(K - 1, 0)))
    rc = _load().ssm_oracle_conv1d(_ptr(x, _fp), _ptr(w, _fp), _ptr(bias, _fp), _ptr(state_in, _fp), int(bool(silu)),
                                   _ptr(y, _dp), _ptr(st, _dp), batch, dim, L, K)
    if rc != 0:
        raise RuntimeError(f"oracle conv1d failed: {rc}")
    return y, st


def pairs(x, delta, A, B, dt_bias, delta_softplus, b, d, n):
    """The exact (a_t, b_t) sequence of recurrence (b, d, n)."""
    x = _f32(x)
    delta = _f32(delta)
    A = _f32(A)
    B = _f32(B)
    dt_bias = _f32(dt_bias)
    batch, dim, L = x.shape
    dstate = A.shape[1]
    a_out = np.empty(L, np.float64)
    b_out = np.empty(L, np.float64)
    rc = _load().ssm_oracle_pairs(_ptr(x, _fp), _ptr(delta, _fp), _ptr(A, _fp), _ptr(B, _fp),
                                  _ptr(dt_bias, _fp), int(bool(delta_softplus)),
                                  batch, dim, dstate, L, b, d, n, _ptr(a_out, _dp), _ptr(b_out, _dp))
    if rc != 0:
        raise RuntimeError("oracle pairs: bad index")
    return a_out, b_out
