"""ctypes declarations of libssmscan.so (the C ABI in include/ssm_scan.h).

Argument marshalling only.  The library must have been built
(``selective_state_space_02_gb300.build.build()``); loading fails loudly if
it is missing -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libssmscan.so")
_lock = threading.Lock()
_lib = None

SSM_F32 = 0
SSM_BF16 = 1

VARIANTS = {"auto": 0, "fused": 1, "chunked": 2, "twopass": 3}
VARIANT_NAMES = {v: k for k, v in VARIANTS.items()}

# Entry points declared in include/ssm_scan.h: name -> (restype, argtypes)
_vp = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_FWD_ARGS = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _i, _i, _i, _i64, _i, _vp, _sz, _vp]
SIGNATURES = {
    "ssm_scan_version": (_i, []),
    "ssm_scan_status_string": (ctypes.c_char_p, [_i]),
    "ssm_scan_select_variant": (_i, [_i, _i, _i, _i64, _i]),
    "ssm_scan_fwd_workspace_size": (_sz, [_i, _i, _i, _i64, _i, _i]),
    "ssm_scan_fwd": (_i, list(_FWD_ARGS)),
    "ssm_scan_fwd_variant": (_i, list(_FWD_ARGS) + [_i]),
    "ssm_scan_device_status": (_i, [_vp, _i]),
    "ssm_scan_selftest_wait_timeout": (_i, [ctypes.c_longlong, _vp]),
    "ssm_scan_fwd_host_buffer_size": (_sz, [_i, _i, _i, _i64, _i, _i, _i, _i, _i, _i]),
    "ssm_scan_fwd_host": (_i, list(_FWD_ARGS) + [_i]),
    "ssm_scan_fwd_noalloc": (_i, list(_FWD_ARGS[:16]) + [_vp]),
    # x..softplus, initial_state, y, final_state, sizes, dtype, workspace, bytes, stream, variant
    "ssm_scan_fwd_from_state": (_i, list(_FWD_ARGS[:9]) + [_vp] + list(_FWD_ARGS[9:]) + [_i]),
    # state, x, delta, A, B, C, D, z, dt_bias, softplus, y, batch, dim, dstate, dtype, stream
    "ssm_scan_step": (_i, [_vp] * 9 + [_i, _vp, _i, _i, _i, _i, _vp]),
    # x, weight, bias, state_in, y, state_out, silu, batch, dim, seqlen, width, dtype, stream
    "ssm_conv1d_fwd": (_i, [_vp] * 6 + [_i, _i, _i, _i64, _i, _i, _vp]),
    # batch, dim, dstate, seqlen, width, dtype, mode
    "ssm_scan_fwd_conv_workspace_size": (_sz, [_i, _i, _i, _i64, _i, _i, _i]),
    # x, weight, bias, state, width, delta, A, B, C, D, z, dt_bias, softplus, y, final_state,
    # batch, dim, dstate, seqlen, dtype, workspace, bytes, stream, mode
    "ssm_scan_fwd_conv": (_i, [_vp] * 4 + [_i] + [_vp] * 7 + [_i, _vp, _vp, _i, _i, _i, _i64, _i, _vp, _sz, _vp, _i]),
    "ssm_scan_bwd_workspace_size": (_sz, [_i, _i, _i, _i64, _i]),
    "ssm_scan_bwd_kernel_count": (_i, [_i, _i, _i, _i64]),
    # x, delta, A, B, C, D, z, dt_bias, softplus, h0, dy, dfinal, dx, ddelta, dA, dB, dC, dD, dz, ddt_bias,
    # dh0, batch, dim, dstate, seqlen, dtype, workspace, bytes, stream
    "ssm_scan_bwd": (_i, [_vp] * 8 + [_i] + [_vp] * 12 + [_i, _i, _i, _i64, _i, _vp, _sz, _vp]),
    # checkpoints of the training forward, consumed by the backward
    "ssm_scan_ckpt_size": (_sz, [_i, _i, _i, _i64]),
    "ssm_scan_fwd_ckpt_workspace_size": (_sz, [_i, _i, _i, _i64, _i, _i]),
    # x..softplus, initial_state, y, final_state, ckpt, sizes, dtype, workspace, bytes, stream, variant
    "ssm_scan_fwd_ckpt": (_i, list(_FWD_ARGS[:9]) + [_vp] + list(_FWD_ARGS[9:11]) + [_vp] + list(_FWD_ARGS[11:])
                          + [_i]),
    "ssm_scan_bwd_ckpt_workspace_size": (_sz, [_i, _i, _i, _i64, _i]),
    "ssm_scan_bwd_ckpt_kernel_count": (_i, [_i, _i, _i, _i64]),
    # as ssm_scan_bwd with ckpt in the place of initial_state
    "ssm_scan_bwd_ckpt": (_i, [_vp] * 8 + [_i] + [_vp] * 12 + [_i, _i, _i, _i64, _i, _vp, _sz, _vp]),
}


class ScanError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


def lib_path() -> str:
    return _LIB_PATH


def load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"libssmscan.so not found at {_LIB_PATH}; build it with "
                    "`python -m selective_state_space_02_gb300.build` (needs nvcc)")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().ssm_scan_status_string(int(status)).decode()


def check(status: int):
    if status != 0:
        raise ScanError(status, status_string(status))
