"""Host-side checks of the NVFP4 kernel (no GPU): its launch plan (K split, padded batch,
shared-memory layout, tensor-memory columns, copy boxes) over a sweep of shapes, and the
argument checks of fd_nvfp4_scaled_mm, which reject bad calls before any CUDA call."""

import ctypes

import pytest

from memory_bound_decode_fd_gb300 import _lib

SMEM_OPTIN = 232448 - 128  # GB300 opt-in shared memory per CTA, less the kernel's static part
TMEM_COLS = 256
SF_COL0 = 128

KS = [256, 512, 768, 1024, 1536, 2048, 3072, 4096, 6144, 8192]


def plan(lib, M, K, N, budget=SMEM_OPTIN):
    p = (ctypes.c_int * 11)()
    st = lib.fd_debug_plan_nvfp4(M, K, N, budget, p)
    return st, list(p)


def test_qkv_workload_plan(fdlib):
    # M=64 K=4096 N=6144: four CTAs per cluster along K, 48 weight tiles, two CTAs per SM
    st, p = plan(fdlib, 64, 4096, 6144)
    assert st == _lib.FD_OK
    split, k_cta, stages, npad, tiles, off_x, off_wsf, off_xsf, recv, smem, fits = p
    assert (split, k_cta, stages, npad, tiles) == (4, 1024, 4, 64, 48)
    assert fits == 1 and 2 * (smem + 1024) <= 233472  # two resident CTAs per SM


@pytest.mark.parametrize("M", [1, 2, 15, 16, 17, 31, 33, 64, 65, 100, 128])
@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("N", [1, 127, 128, 6144])
def test_plan_invariants(fdlib, M, K, N):
    st, p = plan(fdlib, M, K, N)
    assert st == _lib.FD_OK, (M, K, N)
    split, k_cta, stages, npad, tiles, off_x, off_wsf, off_xsf, recv, smem, fits = p
    assert fits == 1
    assert split in (1, 2, 4, 8) and split * k_cta == K
    assert k_cta % 256 == 0 and k_cta <= 1024 and stages == k_cta // 256
    assert npad in (16, 32, 64, 128) and M <= npad and (npad == 16 or npad // 2 < M)
    assert tiles * 128 >= N > (tiles - 1) * 128
    # stage bases are 1024-byte aligned (128-byte swizzle atoms), regions in order, no overlap
    w_stage, x_stage, sf_row = 16384, npad * 128, k_cta // 16
    assert off_x == stages * w_stage and off_x % 1024 == 0 and x_stage % 1024 == 0
    assert off_wsf == off_x + stages * x_stage
    assert off_xsf == off_wsf + 128 * sf_row
    end = off_xsf + npad * sf_row
    assert smem >= max(end, recv) + 1024
    # at most two CTAs per SM (233472 bytes of shared memory, 1024 reserved per CTA), so two
    # 256-column TMEM allocations never exceed the SM's 512 columns
    assert 3 * (smem + 1024) > 233472
    # the scale tiles' copy boxes: inner extent a multiple of 16 bytes, at most 256
    assert sf_row % 16 == 0 and 16 <= sf_row <= 256 and off_wsf % 16 == 0 and off_xsf % 16 == 0
    # the reduction buffer [split][npad][128 / split] fp32 and the rows each rank finishes
    assert 128 % split == 0 and recv == split * npad * (128 // split) * 4
    # tensor memory: the accumulator's npad columns, then 8 scale columns per K = 64 step
    assert npad <= SF_COL0 and SF_COL0 + 8 * (k_cta // 64) <= TMEM_COLS


def test_tmem_and_smem_addresses_replayed(fdlib):
    # Replay, for the workload shape, every address the kernel forms: the MMA descriptors'
    # start addresses (weights and activations, 32 bytes per K = 64 step inside a 128-byte
    # row), the scale columns and the reduction stores.
    st, p = plan(fdlib, 64, 4096, 6144)
    split, k_cta, stages, npad, tiles, off_x, off_wsf, off_xsf, recv, smem, fits = p
    for s in range(stages):
        for j in range(4):
            kb = 4 * s + j
            a = s * 16384 + 32 * j
            b = off_x + s * npad * 128 + 32 * j
            # an MMA reads 128 (resp. npad) rows of 32 bytes from 1024-byte swizzle atoms
            assert a + 127 * 128 + 32 <= off_x and b + (npad - 1) * 128 + 32 <= off_wsf
            assert SF_COL0 + 8 * kb + 8 <= TMEM_COLS
            # scale bytes read for this step: rows 0..127 (npad) at 4 kb .. 4 kb + 3
            assert off_wsf + 127 * (k_cta // 16) + 4 * kb + 4 <= off_xsf
            assert off_xsf + (npad - 1) * (k_cta // 16) + 4 * kb + 4 <= smem - 1024
    rows_own = 128 // split
    for rank in range(split):
        for r in range(128):
            owner, rr = divmod(r, rows_own)
            assert owner < split
            for j in range(npad):
                addr = ((rank * npad + j) * rows_own + rr) * 4
                assert 0 <= addr and addr + 4 <= recv <= smem - 1024


@pytest.mark.parametrize("K", [0, 128, 300, 4097])
def test_bad_k_is_a_shape_error(fdlib, K):
    st, _ = plan(fdlib, 64, K, 128)
    assert st == _lib.FD_ERR_UNSUPPORTED
    assert call(fdlib, K=K) == _lib.FD_ERR_SHAPE


@pytest.mark.parametrize("K", [1280, 2304, 4352, 8448, 16384])
def test_k_without_a_split_is_unsupported(fdlib, K):
    assert call(fdlib, K=K) == _lib.FD_ERR_UNSUPPORTED


# Fake, aligned "device" addresses: every call below is rejected on the host before any
# CUDA call, so nothing is dereferenced or launched.
X, XS, W, WS, AL, O = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000, 0x60000000


def call(lib, x=X, xs=XS, w=W, ws=WS, alpha=AL, out=O, M=64, K=4096, N=6144):
    return lib.fd_nvfp4_scaled_mm(ctypes.c_void_p(x), ctypes.c_void_p(xs), ctypes.c_void_p(w),
                                  ctypes.c_void_p(ws), ctypes.c_void_p(alpha), ctypes.c_void_p(out),
                                  M, K, N, None)


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), _lib.FD_ERR_SHAPE),
    (dict(N=-1), _lib.FD_ERR_SHAPE),
    (dict(M=257), _lib.FD_ERR_UNSUPPORTED),
    (dict(x=0), _lib.FD_ERR_NULL),
    (dict(ws=0), _lib.FD_ERR_NULL),
    (dict(alpha=0), _lib.FD_ERR_NULL),
    (dict(out=O + 8), _lib.FD_ERR_ALIGN),
    (dict(xs=XS + 4), _lib.FD_ERR_ALIGN),
    (dict(alpha=AL + 2), _lib.FD_ERR_ALIGN),
    (dict(out=X), _lib.FD_ERR_OVERLAP),
    (dict(out=WS + 16), _lib.FD_ERR_OVERLAP),
    (dict(alpha=O + 64), _lib.FD_ERR_OVERLAP),
])
def test_rejects_bad_arguments_without_launching(fdlib, kw, status):
    assert call(fdlib, **kw) == status


def test_empty_call_reads_nothing(fdlib):
    assert call(fdlib, x=0, xs=0, w=0, ws=0, alpha=0, out=0, M=0) == _lib.FD_OK
    assert call(fdlib, x=0, xs=0, w=0, ws=0, alpha=0, out=0, N=0) == _lib.FD_OK


def test_fake_launch_failure_reports_cuda_error(fdlib):
    prev = fdlib.fd_get_launch_flags()
    assert fdlib.fd_set_launch_flags(_lib.FD_LAUNCH_TEST_FAIL) == _lib.FD_OK
    try:
        assert call(fdlib) == _lib.FD_ERR_CUDA
        assert fdlib.fd_last_cuda_error() != 0
    finally:
        fdlib.fd_set_launch_flags(prev)
