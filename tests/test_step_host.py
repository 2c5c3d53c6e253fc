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


# ---- the launch plan of the persistent step (fd_debug_plan_step), against the bulk-copy
# GEMV's (fd_debug_plan_gemv): the outputs are bit-identical to the separate GEMV only while
# both split the rows among the CTAs the same way.

# GB300: SMs, opt-in shared memory per CTA, shared memory per SM, reserved per CTA, a
# kernel's static shared memory, registers per thread
GB300_GEMV = (152, 232448, 233472, 1024, 256, 64)
GB300_STEP = (152, 232448, 233472, 1024, 384, 64)
STEP_FIELDS = ("grid", "rows_base", "rows_extra", "S", "w_rows", "smem", "rms_vpt", "rms_threads")


def step_plan(lib, hidden, inter=INTER, group=GROUP, device=GB300_STEP):
    dev = (ctypes.c_int * 6)(*device)
    out = (ctypes.c_int * 8)()
    st = lib.fd_debug_plan_step(dev, hidden, inter, group, out)
    return st, dict(zip(STEP_FIELDS, list(out)))


def gemv_plan(lib, N, K=INTER, group=GROUP, device=GB300_GEMV):
    dev = (ctypes.c_int * 6)(*device)
    out = (ctypes.c_int * 9)()
    st = lib.fd_debug_plan_gemv(dev, 1, K, N, group, 0, out)
    return st, list(out)


def test_decode_shape_plan(fdlib):
    st, p = step_plan(fdlib, 4096)
    assert st == _lib.FD_OK
    assert (p["grid"], p["rows_base"], p["rows_extra"], p["S"], p["w_rows"]) == (152, 26, 144, 4, 27)
    # 27 rows x 7 KB, 32 rows of scales, 28 warps x 64 partials, the normalised row
    assert p["smem"] == 27 * 7168 + 32 * 224 + 28 * 64 * 4 + 4096 * 2
    assert (p["rms_vpt"], p["rms_threads"]) == (2, 256)


def test_plan_rejects_bad_arguments(fdlib):
    out = (ctypes.c_int * 8)()
    dev = (ctypes.c_int * 6)(*GB300_STEP)
    assert fdlib.fd_debug_plan_step(None, 4096, INTER, GROUP, out) == _lib.FD_ERR_NULL
    assert fdlib.fd_debug_plan_step(dev, 4096, INTER, GROUP, None) == _lib.FD_ERR_NULL
    assert fdlib.fd_debug_plan_step(dev, 4100, INTER, GROUP, out) == _lib.FD_ERR_SHAPE
    assert fdlib.fd_debug_plan_step(dev, 0, INTER, GROUP, out) == _lib.FD_ERR_SHAPE
    assert fdlib.fd_debug_plan_step(dev, 4096, 4096, GROUP, out) == _lib.FD_ERR_UNSUPPORTED
    assert fdlib.fd_debug_plan_step(dev, 4096, INTER, 64, out) == _lib.FD_ERR_UNSUPPORTED


def row_kernel_block(hidden):
    """The add-RMSNorm row kernel's block for one row (its launcher's rule): vpt 1 up to 256
    vectors, 2 up to 512, 4 up to 1024, threads rounded up to whole warps."""
    nvec = hidden // 8
    vpt = 1 if nvec <= 256 else 2 if nvec <= 512 else 4 if nvec <= 1024 else 8
    return vpt, (-(-nvec // vpt) + 31) // 32 * 32


def test_plan_matches_the_gemv_partition_for_every_hidden(fdlib):
    supported = []
    for hidden in range(8, 64 * 152 + 1, 8):
        st, p = step_plan(fdlib, hidden)
        if st != _lib.FD_OK:
            assert st == _lib.FD_ERR_UNSUPPORTED
            continue
        supported.append(hidden)
        gst, g = gemv_plan(fdlib, hidden)
        assert gst == _lib.FD_OK
        # one CTA per SM in both, the same rows per CTA
        assert g[7] == 1, hidden
        assert (p["grid"], p["rows_base"], p["rows_extra"]) == tuple(g[:3]), hidden
        # every row owned once; every chunk of the largest CTA resident; within the budget
        assert p["grid"] * p["rows_base"] + p["rows_extra"] == hidden
        n_max = p["rows_base"] + (1 if p["rows_extra"] else 0)
        assert p["w_rows"] == n_max and p["S"] == -(-n_max // 8) and p["S"] <= 8
        assert p["smem"] <= GB300_STEP[1] - GB300_STEP[4]
        assert (p["rms_vpt"], p["rms_threads"]) == row_kernel_block(hidden), hidden
    # every hidden from 8 up to the largest that fits is supported (no holes), and the
    # largest is 29 rows on every SM
    assert supported == list(range(8, supported[-1] + 1, 8))
    assert supported[-1] == 29 * 152


@pytest.mark.parametrize("sms", [1, 2, 8, 100, 132, 152, 160])
def test_plan_on_other_sm_counts(fdlib, sms):
    # on any SM count the two plans split the rows the same way
    for hidden in (8, 64, 1000, 2048, 4096):
        st, p = step_plan(fdlib, hidden, device=(sms,) + GB300_STEP[1:])
        gst, g = gemv_plan(fdlib, hidden, device=(sms,) + GB300_GEMV[1:])
        if st != _lib.FD_OK:
            assert st == _lib.FD_ERR_UNSUPPORTED
            continue
        assert gst == _lib.FD_OK and g[7] == 1
        assert (p["grid"], p["rows_base"], p["rows_extra"]) == tuple(g[:3]), (sms, hidden)



def test_copy_rows_binding_rejects_bad_tensors():
    # checked before any CUDA call
    import torch

    from memory_bound_decode_fd_gb300 import kernels

    a = torch.zeros((4, 16), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="same shape"):
        kernels.copy_rows(a, torch.zeros((4, 8), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="same shape and dtype"):
        kernels.copy_rows(a, torch.zeros((4, 16), dtype=torch.float32))
    with pytest.raises(ValueError, match="contiguous"):
        kernels.copy_rows(a, torch.zeros((16, 4), dtype=torch.bfloat16).t())
    with pytest.raises(ValueError, match="CUDA tensor"):
        kernels.copy_rows(a, torch.zeros((4, 16), dtype=torch.bfloat16))
