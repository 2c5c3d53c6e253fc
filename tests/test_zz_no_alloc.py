"""fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc: the GEMV with the next layer's add-RMSNorm
folded in, for callers that cannot allocate device memory when they call (a stream being
captured into a CUDA graph, a plugin inside another runtime with no allocator of its own,
a process whose device memory belongs to an arena it does not control). It takes no scratch
argument: the library keeps the fold's counter and partial sums in its own static device
array. Called here through the C ABI, two calls in a row on different inputs, each checked
against the existing entry point (which takes a caller-allocated scratch buffer) on the same
inputs, within the tolerances the other tests use. This file is collected last; it passes
alone in a fresh process as well as after the other tests."""

import ctypes

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
from memory_bound_decode_fd_gb300 import _lib, inputs
from fd_check import bf16_f64, dev_bf16, dev_i32, host_bits, stated_bar

pytestmark = pytest.mark.gpu

EPS = 1e-5
K, N, GROUP = 14336, 4096, 128


def make(seed):
    d = inputs.gemv_inputs(1, K, N, GROUP, seed=seed)
    rng = np.random.default_rng(seed + 100)
    return {
        "gate": dev_bf16(d["gate"]), "up": dev_bf16(d["up"]),
        "qweight": dev_i32(d["qweight"]), "scales": dev_bf16(d["scales"]),
        "residual": dev_bf16(inputs.normal_bf16(rng, (1, N))),
        "rms_weight": dev_bf16(inputs.normal_bf16(rng, (N,), 1.0, 0.1)),
    }


def no_alloc_call(t):
    """The new entry point through the C ABI, every output preallocated by the test."""
    y = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
    normed = torch.empty_like(y)
    res_out = torch.empty_like(y)
    lib = fd.load_library()
    stream = torch.cuda.current_stream()
    p = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    st = lib.fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc(
        p(t["gate"]), p(t["up"]), p(t["qweight"]), p(t["scales"]), p(y), p(t["residual"]),
        p(t["rms_weight"]), ctypes.c_float(EPS), p(normed), p(res_out), K, N, GROUP,
        ctypes.c_void_p(stream.cuda_stream))
    assert st == _lib.FD_OK, fd.status_string(st)
    torch.cuda.synchronize()
    return host_bits(y), host_bits(normed), host_bits(res_out)


def existing_call(t):
    """The existing entry point on the same inputs, with a caller-allocated scratch."""
    y, normed, res_out = fd.swiglu_w4a16_gemv_add_rmsnorm(
        t["gate"], t["up"], t["qweight"], t["scales"], t["residual"], t["rms_weight"], EPS,
        fd.fold_scratch(), group=GROUP)
    torch.cuda.synchronize()
    return host_bits(y), host_bits(normed), host_bits(res_out)


def test_no_alloc_entry_point_matches_the_existing_one_twice(cuda_device):
    prev = fd.set_gemv_path("auto")
    try:
        for seed in (91, 92):  # two calls in a row, on different inputs
            t = make(seed)
            got = no_alloc_call(t)
            ref = existing_call(t)
            for name, g, r in zip(("y", "normed", "residual_out"), got, ref):
                stated_bar(bf16_f64(g), bf16_f64(r))
            # the new residual is bf16(y + residual): exact wherever y agrees
            same_y = got[0] == ref[0]
            assert np.array_equal(got[2][same_y], ref[2][same_y])
    finally:
        fd.set_gemv_path(prev)
