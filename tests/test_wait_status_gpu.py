"""A bounded device wait that runs out is reported to the host and leaves the context
usable. The test-only launch flag FD_LAUNCH_TEST_WAIT_TIMEOUT gives the M = 1 cluster GEMV
a wait limit of about 2^20 SM clocks and makes its copy thread leave the first weight chunk
of every CTA uncopied, so the consumers' wait for that chunk runs out: no fault, no hang,
no copy left in flight. The call's outputs are NaN, fd_device_status reports
FD_DEVICE_STATUS_WAIT_TIMEOUT once, and the next call is correct."""

import time

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
import oracle
from memory_bound_decode_fd_gb300 import _lib, inputs
from fd_check import check_gemv, dev_bf16, dev_i32, host_bits

pytestmark = pytest.mark.gpu


def run(d, out=None):
    y = fd.swiglu_w4a16_gemv(dev_bf16(d["gate"]), dev_bf16(d["up"]), dev_i32(d["qweight"]),
                             dev_bf16(d["scales"]), out=out, group=d["group"])
    torch.cuda.synchronize()
    return host_bits(y)


def test_wait_timeout_is_reported_and_the_context_stays_usable(cuda_device):
    lib = fd.load_library()
    d = inputs.gemv_inputs(1, 14336, 4096, 128, seed=40)
    prev_path = fd.set_gemv_path("auto")
    try:
        run(d)  # load the kernel (and its cached launch facts) outside the timed call
        assert fd.device_status(clear=True) == 0
        flags = lib.fd_get_launch_flags()
        assert lib.fd_set_launch_flags(flags | _lib.FD_LAUNCH_TEST_WAIT_TIMEOUT) == _lib.FD_OK
        try:
            t0 = time.perf_counter()
            y = run(d)
            elapsed = time.perf_counter() - t0
        finally:
            lib.fd_set_launch_flags(flags)
        assert elapsed < 5.0, elapsed  # the short limit, not the second-long default
        assert np.all(np.isnan(oracle.bf16_to_f32(y)))
        st = fd.device_status(clear=True)
        assert st & _lib.FD_DEVICE_STATUS_WAIT_TIMEOUT
        assert fd.device_status(clear=True) == 0  # cleared
        # the context is usable and the kernel correct again
        check_gemv(run(d), d["gate"], d["up"], d["qweight"], d["scales"], 128)
        assert fd.device_status(clear=True) == 0
    finally:
        fd.set_gemv_path(prev_path)


def test_status_is_clean_after_ordinary_calls(cuda_device):
    d = inputs.gemv_inputs(1, 9216, 2560, 128, seed=41)
    fd.device_status(clear=True)
    for path in ("auto", "bulk", "cuda_core"):
        prev = fd.set_gemv_path(path)
        try:
            run(d)
        finally:
            fd.set_gemv_path(prev)
    assert fd.device_status(clear=False) == 0
