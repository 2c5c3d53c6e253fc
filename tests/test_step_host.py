"""Host-side checks of fd_decode_mlp_step (no GPU): the argument checks reject bad calls
before any CUDA call, the unsupported shapes are reported as such, and a failed launch
surfaces as FD_ERR_CUDA. Every pointer below is a fake, aligned address: each call is
rejected on the host, so nothing is dereferenced or launched."""

import ctypes
from pathlib import Path

import pytest

from memory_bound_decode_fd_gb300 import _lib

TABLE, X0, RES, SCRATCH = 0x10000000, 0x20000000, 0x30000000, 0x40000000
HEADER = Path(__file__).resolve().parent.parent / "include" / "fd.h"
HIDDEN, INTER, GROUP = 4096, 14336, 128


def call(lib, table=TABLE, n_layers=32, x0=X0, residual=RES, eps=1e-5, hidden=HIDDEN,
         inter=INTER, group=GROUP, scratch=SCRATCH):
    vp = ctypes.c_void_p
    return lib.fd_decode_mlp_step(vp(table), n_layers, vp(x0), vp(residual), ctypes.c_float(eps),
                                  hidden, inter, group, vp(scratch), vp(0))


@pytest.mark.parametrize("field", ["table", "x0", "residual", "scratch"])
def test_null_pointers(fdlib, field):
    assert call(fdlib, **{field: 0}) == _lib.FD_ERR_NULL


@pytest.mark.parametrize("kw", [dict(n_layers=0), dict(n_layers=_lib.FD_STEP_MAX_LAYERS + 1),
                                dict(hidden=4100), dict(hidden=0), dict(inter=0), dict(group=0),
                                dict(eps=-1.0), dict(eps=float("nan")), dict(eps=float("inf"))])
def test_bad_shapes(fdlib, kw):
    assert call(fdlib, **kw) == _lib.FD_ERR_SHAPE


@pytest.mark.parametrize("kw", [dict(x0=X0 + 8), dict(residual=RES + 2), dict(table=TABLE + 8),
                                dict(scratch=SCRATCH + 4), dict(scratch=SCRATCH + 8)])
def test_misaligned(fdlib, kw):
    assert call(fdlib, **kw) == _lib.FD_ERR_ALIGN


@pytest.mark.parametrize("kw", [dict(residual=X0 + 4096), dict(scratch=RES + 16),
                                dict(scratch=X0 + 8000), dict(scratch=X0 - 32768)])
def test_overlaps(fdlib, kw):
    assert call(fdlib, **kw) == _lib.FD_ERR_OVERLAP


@pytest.mark.parametrize("kw", [dict(inter=4096), dict(group=64), dict(hidden=64 * 152 + 8)])
def test_unsupported_shapes_launch_nothing(fdlib, kw):
    assert call(fdlib, **kw) == _lib.FD_ERR_UNSUPPORTED


def test_failed_launch_is_a_cuda_error(fdlib):
    prev = fdlib.fd_get_launch_flags()
    assert fdlib.fd_set_launch_flags(prev | _lib.FD_LAUNCH_TEST_FAIL) == _lib.FD_OK
    try:
        assert call(fdlib) == _lib.FD_ERR_CUDA
    finally:
        fdlib.fd_set_launch_flags(prev)


def test_scratch_size():
    # one counter per layer padded to 16 bytes, then two rows of 32-bit tagged h words
    assert _lib.step_scratch_bytes(32, 4096) == 128 + 2 * 4096 * 4
    assert _lib.step_scratch_bytes(3, 2048) == 16 + 2 * 2048 * 4
    text = HEADER.read_text()
    assert "#define FD_STEP_SCRATCH_HROWS_OFFSET(n_layers) ((((size_t)(n_layers) * 4 + 15) / 16) * 16)" in text
    assert "(FD_STEP_SCRATCH_HROWS_OFFSET(n_layers) + (size_t)(hidden) * 8)" in text
