"""Host-side tests (no GPU) of the tensor-core GEMV's shared-memory planner, through the C
ABI (fd_debug_plan_tc): the decode shape's plan, and for a sweep of shapes the invariants
the kernel relies on: the k step by batch size, regions in order and on 1024-byte
boundaries (the 128-byte-swizzled tensor-map destinations), operand stages in pairs (the
two halves the MMA thread commits), the scale window, room for the cluster reduction in
the rings, and the budget."""

import ctypes
import itertools

import pytest

from memory_bound_decode_fd_gb300 import _lib

# the opt-in shared memory of a GB300 CTA less the kernel's static shared memory
BUDGET = 232448 - 816
FIELDS = ("npad", "stepk", "s_w", "s_gu", "s_op", "sg", "off_gu", "off_op", "off_sc", "smem")


def plan(lib, M, K, N, group=128, budget=BUDGET):
    out = (ctypes.c_int * 10)()
    st = lib.fd_debug_plan_tc(M, K, N, group, budget, out)
    return st, dict(zip(FIELDS, list(out)))


def test_decode_batch_plan(fdlib):
    st, p = plan(fdlib, 64, 14336, 4096)
    assert st == _lib.FD_OK
    assert (p["npad"], p["stepk"]) == (64, 128)
    # 48 KB operand stages: two of them and two 32 KB gate/up stages leave room for 3
    # weight tiles of 16 KB
    assert (p["s_w"], p["s_gu"], p["s_op"]) == (3, 2, 2)
    assert p["sg"] == 40  # 28 groups of a K quarter + the 8-aligned window
    st, p = plan(fdlib, 128, 14336, 4096)
    assert st == _lib.FD_OK and (p["npad"], p["stepk"]) == (128, 64)


def test_wide_k_small_groups_fall_back_to_64k_steps(fdlib):
    # K = 32768, group 64: the 136-column scale window leaves too little room for 128-k
    # stages at 64 rows, so the kernel runs 64-k steps (still on the tensor cores)
    st, p = plan(fdlib, 64, 32768, 256, 64)
    assert st == _lib.FD_OK and (p["npad"], p["stepk"], p["sg"]) == (64, 64, 136)
    st, p = plan(fdlib, 20, 32768, 256, 64)
    assert st == _lib.FD_OK and (p["npad"], p["stepk"]) == (32, 128)


def test_rejects(fdlib):
    out = (ctypes.c_int * 10)()
    assert fdlib.fd_debug_plan_tc(64, 14336, 4096, 128, BUDGET, None) == _lib.FD_ERR_NULL
    assert fdlib.fd_debug_plan_tc(0, 14336, 4096, 128, BUDGET, out) == _lib.FD_ERR_SHAPE
    assert fdlib.fd_debug_plan_tc(64, 14336, 4000, 128, BUDGET, out) == _lib.FD_ERR_UNSUPPORTED  # N % 128
    assert fdlib.fd_debug_plan_tc(64, 2048, 256, 32, BUDGET, out) == _lib.FD_ERR_UNSUPPORTED  # group % 64
    assert fdlib.fd_debug_plan_tc(64, 14336, 4096, 128, 64 * 1024, out) == _lib.FD_ERR_UNSUPPORTED


SWEEP = list(itertools.product(
    (1, 16, 17, 32, 33, 64, 65, 128, 256),            # M
    (1024, 2048, 4096, 9216, 14336, 16384, 32768),    # K
    (64, 128, 256, 512),                              # group
))


@pytest.mark.parametrize("M,K,group", SWEEP)
def test_plan_invariants(fdlib, M, K, group):
    st, p = plan(fdlib, M, K, 256, group)
    if K % 1024 or K % group or (K // group) % 8:
        assert st == _lib.FD_ERR_UNSUPPORTED
        return
    assert st == _lib.FD_OK, (M, K, group)
    npad, stepk = p["npad"], p["stepk"]
    m = min(M, 128)
    assert npad == next(n for n in (16, 32, 64, 128) if m <= n)
    k_cta = K // 4
    # 128-k steps up to 64 rows unless even their smallest layout (2 weight tiles, 2 gate/up
    # and 2 operand stages) exceeds the budget; then 64-k steps
    sg = (-(-k_cta // group) + 14) & ~7
    sc = -(-128 * sg * 2 // 1024) * 1024
    fits128 = 1024 + 2 * 16384 + sc + 2 * (4 * npad * 128) + 2 * (128 * 256 + npad * 256) <= BUDGET
    assert stepk == (128 if npad <= 64 and fits128 else 64), (M, K, group)
    assert k_cta % stepk == 0 and k_cta % 256 == 0
    gu_stage = 2 * (stepk // 64) * npad * 128
    op_stage = 128 * stepk * 2 + npad * stepk * 2
    # regions in order, each on a 1024-byte boundary
    assert p["off_gu"] == p["s_w"] * 16384
    assert p["off_op"] == p["off_gu"] + p["s_gu"] * gu_stage
    assert p["off_sc"] == p["off_op"] + p["s_op"] * op_stage
    for v in (p["off_gu"], p["off_op"], p["off_sc"], gu_stage, op_stage, npad * 128):
        assert v % 1024 == 0
    assert 2 <= p["s_w"] <= 4 and 2 <= p["s_gu"] <= 4 and p["s_op"] in (2, 4)
    # the scale window: every group of the K quarter, from an 8-aligned first column
    groups = -(-k_cta // group)
    assert p["sg"] % 8 == 0 and groups + 7 <= p["sg"] <= 256
    sc_bytes = -(-128 * p["sg"] * 2 // 1024) * 1024
    assert p["smem"] == p["off_sc"] + sc_bytes + 1024 <= BUDGET
    # the cluster reduction ([4 ranks][npad][32 rows] fp32) fits the two rings it reuses
    assert 4 * npad * 32 * 4 <= p["off_sc"] - p["off_gu"]
