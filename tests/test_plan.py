"""Host-side tests (no GPU) of the bulk-copy GEMV kernel's launch planner, through the C ABI
(fd_debug_plan_gemv): the plans of the workload shapes, and for a sweep of shapes and
device facts the invariants the kernel relies on (every row owned once, stages within the
mbarrier slots, shared memory within each CTA's share, the activation copy never
overlapping a stage filled before it is read)."""

import ctypes
import itertools

import pytest

from memory_bound_decode_fd_gb300 import _lib

# GB300: SMs, opt-in shared memory per CTA, shared memory per SM, reserved per CTA,
# the kernel's static shared memory, registers per thread
GB300 = (152, 232448, 233472, 1024, 256, 64)
FIELDS = ("grid", "rows_base", "rows_extra", "S", "w_rows", "act_first_stage", "ring",
          "per_sm", "smem")


def plan(lib, M, K, N, group=128, plain=0, device=GB300):
    dev = (ctypes.c_int * 6)(*device)
    out = (ctypes.c_int * 9)()
    st = lib.fd_debug_plan_gemv(dev, M, K, N, group, plain, out)
    return st, dict(zip(FIELDS, list(out)))


def test_workload_plans(fdlib):
    st, p = plan(fdlib, 1, 14336, 4096)       # decode-step down projection
    assert st == 0 and p["ring"] == 0 and p["per_sm"] == 1 and p["grid"] == 152
    assert (p["S"], p["w_rows"], p["act_first_stage"]) == (4, 27, 2)  # gate/up overlays rows 19-26
    st, p = plan(fdlib, 1, 9216, 2560)        # gate/up in a stage of its own
    assert st == 0 and p["ring"] == 0 and (p["S"], p["w_rows"], p["act_first_stage"]) == (4, 32, 3)
    st, p = plan(fdlib, 1, 4096, 28672, plain=1)  # gate/up projection: three CTAs per SM
    assert st == 0 and p["per_sm"] == 3 and p["grid"] == 456 and p["ring"] == 1 and p["S"] == 4
    st, p = plan(fdlib, 1, 14336, 8192)       # larger share: a ring
    assert st == 0 and p["ring"] == 1 and p["S"] == 3 and p["act_first_stage"] == 2


def test_rejects_bad_arguments(fdlib):
    out = (ctypes.c_int * 9)()
    dev = (ctypes.c_int * 6)(*GB300)
    assert fdlib.fd_debug_plan_gemv(None, 1, 1024, 8, 128, 0, out) == _lib.FD_ERR_NULL
    assert fdlib.fd_debug_plan_gemv(dev, 1, 1000, 8, 128, 0, out) == _lib.FD_ERR_SHAPE
    assert fdlib.fd_debug_plan_gemv(dev, 0, 1024, 8, 128, 0, out) == _lib.FD_ERR_SHAPE


SWEEP = list(itertools.product(
    (1, 2, 3, 16),                                   # M
    (1024, 2048, 4096, 9216, 14336, 15360),          # K
    (7, 100, 256, 1000, 2560, 4096, 8192, 28672),    # N
    (0, 1),                                          # plain
    (40, 64, 128),                                   # registers
))


@pytest.mark.parametrize("M,K,N,plain,regs", SWEEP)
def test_plan_invariants(fdlib, M, K, N, plain, regs):
    group, R = 128, 8
    sms, optin, per_sm_smem, reserved, static, _ = GB300
    st, p = plan(fdlib, M, K, N, group, plain, (sms, optin, per_sm_smem, reserved, static, regs))
    MB, LPS = (1, 2) if M == 1 else (2, 1)
    w_row, s_row = K // 2, (K // group) * 2
    red = (LPS * (K // 32) // 32) * 64 * MB * 4
    if st != 0:
        # not launched: only when even a two-stage ring does not fit one CTA
        assert st == _lib.FD_ERR_UNSUPPORTED
        assert red + 2 * R * (w_row + s_row) > optin - static or M == 1
        return
    # every row owned exactly once
    assert p["rows_base"] >= 1 and 0 <= p["rows_extra"] < p["grid"]
    assert p["grid"] * p["rows_base"] + p["rows_extra"] == N
    # stages within the mbarrier slots, layout bytes as the kernel computes them
    assert 1 <= p["S"] <= 8
    assert p["smem"] == p["w_rows"] * w_row + p["S"] * R * s_row + red
    assert p["smem"] <= optin - static
    # resident CTAs per SM fit the SM: shared memory, threads, registers
    c = p["per_sm"]
    threads = LPS * (K // 32) + 32
    warps = (threads + 31) // 32
    assert 1 <= c <= 4
    if c > 1:  # one CTA always fits: the kernel's launch bounds cap its registers
        assert c * threads <= 2048
        assert c * warps * ((regs * 32 + 255) // 256) * 256 <= 65536
        assert c * (p["smem"] + reserved + static) <= per_sm_smem
    n_max = p["rows_base"] + (p["rows_extra"] > 0)
    if not p["ring"]:
        # one pass, every chunk in a stage of its own
        assert M <= MB and p["w_rows"] >= n_max and -(-n_max // R) <= p["S"]
    if M == 1:
        act = K * (2 if plain else 4)
        # the activation copy fits the weight rows and stays clear of every stage that is
        # filled before the consumers have read it
        assert p["w_rows"] * w_row >= act
        assert p["act_first_stage"] * R * w_row <= p["w_rows"] * w_row - act
        if p["ring"]:
            assert p["act_first_stage"] >= (3 if c > 1 else 2)


def producer_schedule(p, M, N, MB, R):
    """The bulk-copy kernel's producer, replayed on the host: for every CTA, the chunks it
    issues in order, as (chunk index, stage, first row, rows)."""
    for b in range(p["grid"]):
        n_begin = b * p["rows_base"] + min(b, p["rows_extra"])
        n_cnt = p["rows_base"] + (1 if b < p["rows_extra"] else 0)
        n_chunks = -(-n_cnt // R)
        total = n_chunks * -(-M // MB)
        ps = pnc = 0
        for c in range(total):
            yield b, c, ps, n_begin + pnc * R, min(R, n_cnt - pnc * R), total
            ps = (ps + 1) % p["S"]
            pnc = (pnc + 1) % n_chunks


@pytest.mark.parametrize("M,K,N,plain,regs", SWEEP)
def test_producer_copies_stay_in_bounds(fdlib, M, K, N, plain, regs):
    group, R = 128, 8
    sms, optin, per_sm_smem, reserved, static, _ = GB300
    st, p = plan(fdlib, M, K, N, group, plain, (sms, optin, per_sm_smem, reserved, static, regs))
    if st != 0:
        return
    MB = 1 if M == 1 else 2
    w_row = K // 2
    act = K * (2 if plain else 4)
    owned = [0] * N
    for b, c, stage, n0, rows, total in producer_schedule(p, M, N, MB, R):
        assert rows >= 1 and 0 <= n0 and n0 + rows <= N            # global rows in range
        assert stage * R + rows <= p["w_rows"]                      # inside the weight rows
        if M == 1 and c < p["act_first_stage"]:
            # filled before the consumers have read the activation: clear of its bytes
            assert (stage * R + rows) * w_row <= p["w_rows"] * w_row - act
        if not p["ring"]:
            assert total <= p["S"]                                  # no stage is reused
        if c < -(-(p["rows_base"] + (b < p["rows_extra"])) // R):   # first activation pass
            for n in range(n0, n0 + rows):
                owned[n] += 1
    assert owned == [1] * N                                         # every row streamed once per pass
