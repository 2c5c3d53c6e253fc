"""Host-side checks of the NVFP4 kernel (no GPU): its launch plan (K split, padded batch,
shared-memory layout, tensor-memory columns, copy boxes) over a sweep of shapes, and the
argument checks of fd_nvfp4_scaled_mm, which reject bad calls before any CUDA call."""

import ctypes

import pytest

from memory_bound_decode_fd_gb300 import _lib

SMEM_OPTIN = 232448 - 256  # GB300 opt-in shared memory per CTA, less the kernel's static part
SF_COL0 = 128

KS = [256, 512, 768, 1024, 1280, 1536, 2048, 3072, 4096, 6144, 8192, 12288, 16384]


def plan(lib, M, K, N, budget=SMEM_OPTIN):
    p = (ctypes.c_int * 13)()
    st = lib.fd_debug_plan_nvfp4(M, K, N, budget, p)
    keys = ("split", "s_total", "max_stages", "npad", "n_tiles", "tmem_cols", "cols_own",
            "sf_row", "off_x", "off_wsf", "off_xsf", "recv", "smem")
    return st, dict(zip(keys, list(p)))


def test_qkv_workload_plan(fdlib):
    # M=64 K=4096 N=6144 (48 weight tiles of 128 rows, 16 stages of 256 k): four CTAs per
    # cluster along K, 192 CTAs of 4 stages, two per SM by shared memory.
    st, p = plan(fdlib, 64, 4096, 6144)
    assert st == _lib.FD_OK
    assert (p["split"], p["max_stages"], p["npad"], p["n_tiles"]) == (4, 4, 64, 48)
    assert p["tmem_cols"] == 256 and 2 * (p["smem"] + 256 + 1024) <= 233472


def first_stage(r, s_total, split):
    return r * s_total // split


@pytest.mark.parametrize("M", [1, 2, 15, 16, 17, 31, 33, 64, 65, 100, 128])
@pytest.mark.parametrize("K", KS)
@pytest.mark.parametrize("N", [1, 127, 128, 6144, 40000])
def test_plan_invariants_and_replay(fdlib, M, K, N):
    st, p = plan(fdlib, M, K, N)
    if st != _lib.FD_OK and M > 64:
        # 128 padded rows do not fit shared memory at this K: the library runs such a
        # batch in launches of 64 rows, which always have a plan
        assert K > 12288 and plan(fdlib, 64, K, N)[0] == _lib.FD_OK
        return
    assert st == _lib.FD_OK, (M, K, N)
    split, S, ms, npad = p["split"], p["s_total"], p["max_stages"], p["npad"]
    assert 1 <= split <= 8 and S * 256 == K and ms == -(-S // split) <= 12
    # the smallest split with at most 4 stages per CTA where one exists
    if S <= 32:
        assert ms <= 4 and (split == 1 or -(-S // (split - 1)) > 4)
    assert npad in (16, 32, 64, 128) and M <= npad and (npad == 16 or npad // 2 < M)
    assert p["n_tiles"] * 128 >= N > (p["n_tiles"] - 1) * 128
    # every stage of K in exactly one rank's slice; no slice longer than max_stages
    sizes = [first_stage(r + 1, S, split) - first_stage(r, S, split) for r in range(split)]
    assert sum(sizes) == S and max(sizes) == ms and min(sizes) >= 1
    # tensor memory: accumulator columns below 128, 32 scale columns per stage above
    assert npad <= SF_COL0 and SF_COL0 + 32 * ms <= p["tmem_cols"] in (256, 512)
    # at most two CTAs per SM with 256 columns, one with 512 (SM: 233472 bytes, 1 KB
    # reserved per CTA), so the allocations always fit the SM's 512 columns
    per_sm = 233472 // (p["smem"] + 256 + 1024)
    assert per_sm * p["tmem_cols"] <= 512 and p["smem"] <= SMEM_OPTIN
    # shared memory: stage bases 1024-byte aligned, regions in order
    w_stage, x_stage, sf_row = 16384, npad * 128, p["sf_row"]
    assert sf_row == 16 * ms and sf_row <= 256
    assert p["off_x"] == ms * w_stage and x_stage % 1024 == 0
    assert p["off_wsf"] == p["off_x"] + ms * x_stage and p["off_xsf"] == p["off_wsf"] + 128 * sf_row
    end = p["off_xsf"] + npad * sf_row
    assert p["smem"] >= max(end, p["recv"]) + 1024
    # the reduction buffers, receive slots [split][cols_own][128 rows] then the CTA's own
    # accumulator [split * cols_own][128 rows], and the output columns (activation rows)
    # each rank finishes
    cols = p["cols_own"]
    chunk = cols * 128 * 4
    assert cols == -(-npad // split) and chunk % 16 == 0
    assert p["recv"] == 2 * split * chunk
    # replay of one CTA per rank: copies and operand reads inside their regions, global
    # coordinates inside the tensors (the scale box may run past K: zero-filled)
    for r in range(split):
        s0, n_st = first_stage(r, S, split), sizes[r]
        assert 0 <= s0 and s0 + n_st <= S and (s0 * 128) % 16 == 0 and (s0 * 16) % 16 == 0
        for s in range(n_st):
            for j in range(4):
                a = s * w_stage + 32 * j
                b = p["off_x"] + s * x_stage + 32 * j
                assert a + 127 * 128 + 32 <= p["off_x"] and b + (npad - 1) * 128 + 32 <= p["off_wsf"]
                assert SF_COL0 + 32 * s + 8 * j + 8 <= p["tmem_cols"]
            assert p["off_wsf"] + 127 * sf_row + 16 * s + 16 <= p["off_xsf"]
            assert p["off_xsf"] + (npad - 1) * sf_row + 16 * s + 16 <= p["smem"] - 1024
        # rank r's partial sum of column j, row `row`, lands in the owner of j at
        # [r][j - owner cols_own][row]; every column of the batch has an owner
        for j in (0, min(M, npad) - 1):
            owner, jj = divmod(j, cols)
            assert owner < split
            for row in (0, 127):
                slot = r * chunk + (jj * 128 + row) * 4  # in the owner's receive slots
                own = split * chunk + (j * 128 + row) * 4  # in rank r's accumulator
                assert slot + 4 <= split * chunk and split * chunk <= own and own + 4 <= p["recv"]
            # the chunk rank r sends to `owner` lies inside its accumulator
            assert split * chunk + (owner + 1) * chunk <= p["recv"]

@pytest.mark.parametrize("K", [0, 128, 300, 4097])
def test_bad_k_is_a_shape_error(fdlib, K):
    st, _ = plan(fdlib, 64, K, 128)
    assert st == _lib.FD_ERR_UNSUPPORTED
    assert call(fdlib, K=K) == _lib.FD_ERR_SHAPE


@pytest.mark.parametrize("K", [16640, 32768])
def test_k_above_the_maximum_is_unsupported(fdlib, K):
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
