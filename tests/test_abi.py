"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before launching
anything (every call below fails validation, so no kernel is launched and
no fake pointer is ever dereferenced)."""
import ctypes
import glob
import json
import os
import re

import pytest
import torch

import selective_state_space_02_gb300 as ssm
from selective_state_space_02_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssm_scan.h")
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))

OK, ERR_NULL, ERR_DIMS, ERR_ALIGN, ERR_DTYPE, ERR_WORKSPACE = 0, -1, -2, -3, -4, -5
ERR_ALIAS, ERR_VARIANT = -9, -10


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.load()


def _declared_functions():
    names = set()
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(ssm_[a-z_0-9]+)\s*\(", src, re.M))
    return sorted(names)


def test_header_declares_entry_points():
    names = _declared_functions()
    assert "ssm_scan_fwd" in names and "ssm_scan_fwd_host" in names and "ssm_scan_step" in names
    assert set(names) == set(_native.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_no_torch_in_the_abi():
    for h in HEADERS:
        src = open(h).read()
        assert "torch" not in src.lower().replace("pytorch", "") and "at::" not in src


def test_version_and_status_strings(lib):
    assert lib.ssm_scan_version() >> 16 == 1
    for s in (OK, ERR_NULL, ERR_DIMS, ERR_ALIGN, ERR_DTYPE, ERR_WORKSPACE, -6, -8, ERR_ALIAS, ERR_VARIANT, 12345):
        assert isinstance(_native.status_string(s), str) and _native.status_string(s)


def test_variant_selection_host_only(lib):
    assert ssm.select_variant(4, 1536, 16, 2048) == "fused"
    assert ssm.select_variant(8, 2048, 16, 4096) == "fused"
    assert ssm.select_variant(2, 5120, 64, 8192) == "fused"
    assert ssm.select_variant(1, 768, 16, 131072) == "twopass"
    assert ssm.select_variant(1, 64, 16, 1 << 20) == "twopass"
    assert ssm.select_variant(1, 64, 16, 256) == "chunked"
    assert ssm.select_variant(2, 1024, 16, 2048) == "fused"
    assert ssm.select_variant(1, 512, 16, 2048) == "chunked"
    assert ssm.select_variant(1, 512, 16, 4096) == "twopass"
    # measured crossovers that depend on the I/O type
    assert ssm.select_variant(1, 3072, 16, 8192) == "fused"
    assert ssm.select_variant(1, 3072, 16, 8192, torch.bfloat16) == "twopass"
    assert ssm.select_variant(1, 2048, 16, 1024) == "fused"
    assert ssm.select_variant(1, 2048, 16, 1024, torch.bfloat16) == "chunked"
    assert lib.ssm_scan_select_variant(1, 1, 0, 10, 0) == ERR_DIMS
    assert lib.ssm_scan_select_variant(1, 1, 65, 10, 0) == ERR_DIMS
    assert lib.ssm_scan_select_variant(1, 1, 16, 10, 3) == ERR_DTYPE


def _r256(n):
    return (n + 255) // 256 * 256


def test_workspace_sizes(lib):
    # chunked: B and C per chunk of 32 K steps as float4 per (state pair, step); K = 8, or 4 above 32 states
    assert ssm.workspace_size(4, 1536, 16, 2048, variant="chunked") == _r256(4 * 8 * 8 * 256 * 16)
    assert ssm.workspace_size(2, 5120, 64, 8192, variant="chunked") == _r256(2 * 64 * 32 * 128 * 16)
    assert ssm.workspace_size(1, 8, 5, 100, variant="chunked") == _r256(1 * 1 * 3 * 256 * 16)
    # fused: B and C prepared once as float32 rows [batch * L][2 * padded dstate + 16]
    assert ssm.workspace_size(4, 1536, 16, 2048, variant="fused") == _r256(4 * 2048 * 48 * 4)
    assert ssm.workspace_size(2, 5120, 64, 8192, variant="fused") == _r256(2 * 8192 * 144 * 4)
    assert ssm.workspace_size(1, 8, 5, 100, variant="fused") == _r256(100 * 32 * 4)
    for v in ("fused", "twopass"):
        assert ssm.workspace_size(1, 64, 16, 0, variant=v) == 0
    assert lib.ssm_scan_fwd_workspace_size(1, 1, 99, 10, 0, 0) == (1 << 64) - 1
    assert lib.ssm_scan_fwd_workspace_size(1, 1, 16, 10, 0, 7) == (1 << 64) - 1


def test_twopass_workspace_matches_chunk_state_ledger(lib):
    """The two-pass workspace holds one (batch, dim, dstate) fp32 state per
    chunk plus one sum of Delta per (batch, dim) and chunk.  The scan page's
    memory ledger (sect. 3.4) prints the per-chunk state of its example."""
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "ledger.json")))
    sh, pr = g["shape"], g["printed"]
    per_chunk = sh["batch"] * sh["d_inner"] * sh["d_state"]
    assert per_chunk == pr["elements_per_chunk_state"]
    assert per_chunk * 4 / 2 ** 20 == pytest.approx(pr["mb_per_chunk_state_fp32"])
    assert sh["seq_len"] // sh["chunk"] == pr["chunks"]
    assert round(pr["chunks"] * per_chunk * 4 / 1e6, 1) == pr["mb_all_chunk_states_fp32"]
    full = per_chunk * sh["seq_len"]
    assert float(f"{full:.2e}") == pr["elements_all_states"]
    assert round(full * 4 / 1e9, 1) == pr["gb_all_states_fp32"]
    # our workspace for that shape: K chunk states + K delta sums + the float32
    # B/C rows of the fused kernel, each 256-byte rounded
    ws = ssm.workspace_size(sh["batch"], sh["d_inner"], sh["d_state"], sh["seq_len"], variant="twopass")
    r256 = _r256
    bc = r256(sh["batch"] * sh["seq_len"] * (2 * sh["d_state"] + 16) * 4)
    ks = [k for k in range(1, 64)
          if r256(k * per_chunk * 4) + r256(k * sh["batch"] * sh["d_inner"] * 4) + bc == ws]
    assert len(ks) == 1, "workspace is not a whole number of chunk states"
    assert ws < full * 4 / 100, "the workspace must stay far below the full state tensor"


def _fwd(lib, x=8, delta=16 * 64, A=16 * 4096, B=16 * 8192, C=16 * 16384, D=None, z=None, dt=None,
         sp=1, y=16 * 32768, fs=None, batch=1, dim=2, dstate=4, L=8, dtype=0, ws=None, wsb=0, stream=None,
         variant=0):
    # fake, well-separated, 16-byte aligned addresses: every case below must
    # fail validation before any launch
    x = 16 * 2 if x == 8 else x
    return lib.ssm_scan_fwd_variant(x, delta, A, B, C, D, z, dt, sp, y, fs, batch, dim, dstate, L, dtype,
                                    ws, wsb, stream, variant)


def test_rejects_null_pointers(lib):
    assert _fwd(lib, x=None) == ERR_NULL
    assert _fwd(lib, delta=None) == ERR_NULL
    assert _fwd(lib, A=None) == ERR_NULL
    assert _fwd(lib, B=None) == ERR_NULL
    assert _fwd(lib, C=None) == ERR_NULL
    assert _fwd(lib, y=None) == ERR_NULL


def test_rejects_bad_sizes_and_dtype(lib):
    assert _fwd(lib, batch=-1) == ERR_DIMS
    assert _fwd(lib, dim=-3) == ERR_DIMS
    assert _fwd(lib, dstate=0) == ERR_DIMS
    assert _fwd(lib, dstate=65) == ERR_DIMS
    assert _fwd(lib, L=-1) == ERR_DIMS
    assert _fwd(lib, dtype=2) == ERR_DTYPE


def test_rejects_misaligned(lib):
    assert _fwd(lib, x=16 * 2 + 2) == ERR_ALIGN           # f32 needs 4-byte alignment
    assert _fwd(lib, A=16 * 4096 + 1) == ERR_ALIGN
    assert _fwd(lib, y=16 * 32768 + 1, dtype=1) == ERR_ALIGN


def test_rejects_aliasing(lib):
    assert _fwd(lib, y=16 * 2) == ERR_ALIAS                # y == x
    assert _fwd(lib, fs=16 * 4096) == ERR_ALIAS             # final state over A
    assert _fwd(lib, fs=16 * 32768 + 4) == ERR_ALIAS        # final state inside y


def test_rejects_missing_workspace_and_bad_variant(lib):
    assert _fwd(lib, variant=3) == ERR_WORKSPACE
    assert _fwd(lib, variant=3, ws=16 * 65536 + 16, wsb=1 << 20) == ERR_WORKSPACE   # not 256-aligned
    assert _fwd(lib, variant=3, ws=16 * 65536, wsb=4) == ERR_WORKSPACE               # too small
    assert _fwd(lib, variant=9) == ERR_VARIANT


def test_empty_problems_launch_nothing(lib):
    assert _fwd(lib, batch=0) == OK
    assert _fwd(lib, dim=0) == OK
    assert _fwd(lib, L=0) == OK                              # no final state requested


def test_binding_type_checks():
    import torch
    x = torch.zeros(1, 2, 8)
    A = torch.zeros(2, 4)
    B = torch.zeros(1, 4, 8)
    with pytest.raises(TypeError):
        ssm.scan_fwd(x.double(), x.double(), A, B, B)
    with pytest.raises(TypeError):
        ssm.scan_fwd(x, x.bfloat16(), A, B, B)
    with pytest.raises(ValueError):
        ssm.scan_fwd(x, x, A, B, B)                          # CPU tensors on the device path


def _from_state(lib, h0=16 * 65536, fs=None, y=16 * 32768, L=8, variant=0):
    return lib.ssm_scan_fwd_from_state(16 * 2, 16 * 64, 16 * 4096, 16 * 8192, 16 * 16384, None, None, None, 1,
                                       h0, y, fs, 1, 2, 4, L, 0, None, 0, None, variant)


def test_from_state_validation(lib):
    assert _from_state(lib, h0=16 * 65536 + 2) == ERR_ALIGN
    assert _from_state(lib, h0=16 * 32768 + 4) == ERR_ALIAS             # start state inside y
    assert _from_state(lib, h0=16 * 65536, fs=16 * 65536 + 8) == ERR_ALIAS   # partial overlap with final
    assert _from_state(lib, h0=16 * 65536, fs=16 * 65536, L=0, variant=1) == OK   # in place, empty: no copy
    assert _from_state(lib, variant=9) == ERR_VARIANT


def _step(lib, state=16 * 65536, x=16 * 2, delta=16 * 64, A=16 * 4096, B=16 * 8192, C=16 * 16384, y=16 * 32768,
          batch=1, dim=2, dstate=4, dtype=0):
    return lib.ssm_scan_step(state, x, delta, A, B, C, None, None, None, 1, y, batch, dim, dstate, dtype, None)


def test_step_validation(lib):
    assert _step(lib, batch=0) == OK
    assert _step(lib, state=None) == ERR_NULL
    assert _step(lib, y=None) == ERR_NULL
    assert _step(lib, dstate=0) == ERR_DIMS
    assert _step(lib, dstate=65) == ERR_DIMS
    assert _step(lib, dtype=5) == ERR_DTYPE
    assert _step(lib, state=16 * 65536 + 2) == ERR_ALIGN
    assert _step(lib, x=16 * 2 + 1, dtype=1) == ERR_ALIGN
    assert _step(lib, y=16 * 2) == ERR_ALIAS                 # y over x
    assert _step(lib, y=16 * 65536 + 4) == ERR_ALIAS         # y over the state
    assert _step(lib, state=16 * 4096) == ERR_ALIAS          # state over A


def _bwd(lib, dy=16 * 1024, dx=16 * 40000, ddelta=16 * 41000, dA=16 * 42000, dB=16 * 43000, dC=16 * 44000,
         D=None, dD=None, z=None, dz=None, ws=None, wsb=0, L=8, dtype=0):
    # fake, well-separated aligned addresses; every case fails validation before any launch
    return lib.ssm_scan_bwd(16 * 2, 16 * 64, 16 * 4096, 16 * 8192, 16 * 16384, D, z, None, 1, None, dy, None,
                            dx, ddelta, dA, dB, dC, dD, dz, None, None, 1, 2, 4, L, dtype, ws, wsb, None)


def test_bwd_validation(lib):
    assert lib.ssm_scan_bwd_workspace_size(1, 2, 4, 8, 0) > 0
    assert lib.ssm_scan_bwd_workspace_size(1, 2, 4, 0, 0) == 0
    assert lib.ssm_scan_bwd_workspace_size(1, 2, 65, 8, 0) == (1 << 64) - 1
    assert _bwd(lib, dy=None) == ERR_NULL
    assert _bwd(lib, dB=None) == ERR_NULL
    assert _bwd(lib, D=16 * 50000) == ERR_NULL                  # D without dD
    assert _bwd(lib, z=16 * 51000) == ERR_NULL                  # z without dz
    assert _bwd(lib, dx=16 * 2) == ERR_ALIAS                    # dx over x
    assert _bwd(lib, dC=16 * 43000 + 16) == ERR_ALIAS           # dC over dB
    assert _bwd(lib, dA=16 * 42000 + 2) == ERR_ALIGN
    assert _bwd(lib, dtype=7) == ERR_DTYPE
    assert _bwd(lib) == ERR_WORKSPACE                           # workspace required


def _conv(lib, x=16 * 2, w=16 * 4096, b=None, sin=None, y=16 * 8192, sout=None, width=4, L=8, dtype=0):
    # fake, well-separated aligned addresses; every case fails validation before any launch
    return lib.ssm_conv1d_fwd(x, w, b, sin, y, sout, 1, 1, 2, L, width, dtype, None)


def test_conv_validation(lib):
    assert _conv(lib, width=0) == ERR_DIMS
    assert _conv(lib, width=9) == ERR_DIMS
    assert _conv(lib, dtype=3) == ERR_DTYPE
    assert _conv(lib, x=None) == ERR_NULL
    assert _conv(lib, w=None) == ERR_NULL
    assert _conv(lib, x=16 * 2 + 1, dtype=1) == ERR_ALIGN
    assert _conv(lib, y=16 * 2) == ERR_ALIAS                         # y over x
    assert _conv(lib, sin=16 * 100, sout=16 * 100 + 4) == ERR_ALIAS   # state out over state in


def test_backward_kernel_count(lib):
    f = lib.ssm_scan_bwd_kernel_count
    # B/C re-layout + one whole-sequence pass storing the chunk-start states, one reverse walk
    assert f(4, 1536, 16, 2048) == 3
    assert f(8, 2048, 16, 4096) == 3
    assert f(2, 5120, 64, 8192) == 3
    # 768 channels: re-layout, chunk totals and carry scan, then a walk split into segments
    # (adjoint totals, their carry, the walk)
    assert f(1, 768, 16, 131072) == 6
    # one chunk: the carry scan alone gives its start state, one walk
    assert f(1, 8, 16, 20) == 2
    assert f(0, 8, 16, 20) == 0 and f(1, 8, 16, 0) == 0
    assert f(1, 8, 65, 20) == -1 and f(-1, 8, 16, 20) == -1


def test_backward_chunk_state_route_boundary(lib):
    """The chunk-start states come from one whole-sequence pass once the fused
    forward's configuration for the shape has at least 608 consumer warps (one
    per SM sub-partition), else from the totals pass and carry scan: one kernel
    more.  At 16 states that configuration goes down to 2 states a lane (4
    channels a warp); at 64 states a lane holds 16 (8 channels a warp)."""
    f = lib.ssm_scan_bwd_kernel_count
    # 16 states: 2432 channels = 608 warps; walks split into segments (+3)
    assert f(1, 2432, 16, 64) == 5 and f(1, 2428, 16, 64) == 6
    assert f(2, 1216, 13, 4096) == 5 and f(2, 1214, 13, 4096) == 6   # padded states count like 16
    # 64 states: 4864 channels = 608 warps; one walk
    assert f(1, 4864, 64, 64) == 3 and f(1, 4856, 64, 64) == 4


def test_checkpoint_sizes_and_refusals(lib):
    """The training pair's host side: checkpoint bytes (ceil(L / 32) chunk
    states), the forward's workspace (that of the variant it runs; none for
    CHUNKED), the backward's (segment sums only) and kernel count, and the
    checks that refuse before anything is launched."""
    SIZE_MAX = (1 << 64) - 1
    assert lib.ssm_scan_ckpt_size(4, 1536, 16, 2048) == 64 * 4 * 1536 * 16 * 4
    assert lib.ssm_scan_ckpt_size(2, 9, 5, 130) == 5 * 2 * 9 * 5 * 4
    assert lib.ssm_scan_ckpt_size(1, 8, 16, 0) == 0 and lib.ssm_scan_ckpt_size(1, 8, 65, 10) == SIZE_MAX
    fws = lib.ssm_scan_fwd_ckpt_workspace_size
    plain = lib.ssm_scan_fwd_workspace_size
    assert fws(4, 1536, 16, 2048, 1, 1) == plain(4, 1536, 16, 2048, 1, 1)         # FUSED
    assert fws(2, 9, 5, 130, 0, 3) == plain(2, 9, 5, 130, 0, 3)                     # TWOPASS
    assert lib.ssm_scan_select_variant(2, 9, 5, 130, 0) == 2                        # AUTO: CHUNKED ...
    assert fws(2, 9, 5, 130, 0, 0) == plain(2, 9, 5, 130, 0, 3)                     # ... taken as TWOPASS
    assert fws(2, 9, 5, 130, 0, 2) == SIZE_MAX                                      # CHUNKED: none
    assert lib.ssm_scan_bwd_ckpt_workspace_size(4, 1536, 16, 2048, 1) == 0          # one segment
    assert lib.ssm_scan_bwd_ckpt_workspace_size(1, 768, 16, 131072, 0) > 0         # segments
    assert lib.ssm_scan_bwd_ckpt_kernel_count(4, 1536, 16, 2048) == 1
    assert lib.ssm_scan_bwd_ckpt_kernel_count(1, 768, 16, 131072) == 3
    assert lib.ssm_scan_bwd_ckpt_kernel_count(0, 8, 16, 20) == 0
    # no checkpoint buffer: refused before any launch (no pointer is dereferenced)
    ERR_NULL = -1
    rc = lib.ssm_scan_fwd_ckpt(16, 16, 16, 16, 16, None, None, None, 1, None, 16, None, None,
                               1, 8, 16, 64, 0, None, 0, None, 1)
    assert rc == ERR_NULL
    rc = lib.ssm_scan_bwd_ckpt(16, 16, 16, 16, 16, None, None, None, 1, None, 16, None, 16, 16, 16, 16, 16,
                               None, None, None, None, 1, 8, 16, 64, 0, None, 0, None)
    assert rc == ERR_NULL
