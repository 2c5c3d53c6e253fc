"""GPU parity of fd_swiglu_w4a16_gemv_add_rmsnorm: the SwiGLU-W4A16 GEMV of one row with the
next layer's residual add + RMSNorm folded into its tail, called through the C ABI. Every
output is checked against the oracle on the GPU's own inputs: y within the GEMV's derived
bound, the new residual bit-exact (h = bf16(y + residual) from the bf16 y) and the
normalised row within the add-RMSNorm element bound. The fold's scratch must come back
zero after every call."""

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
import oracle
from memory_bound_decode_fd_gb300 import _lib, inputs
from fd_check import check_add_rmsnorm, check_gemv, dev_bf16, dev_i32, host_bits

pytestmark = pytest.mark.gpu

EPS = 1e-5


def make(K, N, seed):
    d = inputs.gemv_inputs(1, K, N, 128, seed=seed)
    rng = np.random.default_rng(seed + 100)
    d["residual"] = inputs.normal_bf16(rng, (1, N))
    d["rms_weight"] = inputs.normal_bf16(rng, (N,), 1.0, 0.1)
    return d


def run_fold(d, scratch, in_place=False):
    res = dev_bf16(d["residual"])
    y, normed, res_out = fd.swiglu_w4a16_gemv_add_rmsnorm(
        dev_bf16(d["gate"]), dev_bf16(d["up"]), dev_i32(d["qweight"]), dev_bf16(d["scales"]),
        res, dev_bf16(d["rms_weight"]), EPS, scratch,
        residual_out=res if in_place else None, group=d["group"])
    torch.cuda.synchronize()
    return host_bits(y), host_bits(normed), host_bits(res_out)


def check_fold(d, y, normed, res_out):
    check_gemv(y, d["gate"], d["up"], d["qweight"], d["scales"], d["group"])
    # the add-RMSNorm on the GPU's own y: residual bit-exact, normed within its bound
    check_add_rmsnorm(normed, res_out, y, d["residual"], d["rms_weight"], EPS)


@pytest.mark.parametrize("K,N", [(14336, 4096), (9216, 2560), (4096, 1024), (1024, 256)])
def test_fold_matches_oracle(cuda_device, K, N):
    d = make(K, N, seed=50 + K % 97)
    scratch = fd.fold_scratch()
    out = run_fold(d, scratch)
    check_fold(d, *out)
    assert int(scratch[:4].view(torch.int32).item()) == 0  # the counter is reset


def test_fold_twice_in_a_row_and_in_place(cuda_device):
    d = make(14336, 4096, seed=61)
    scratch = fd.fold_scratch()
    a = run_fold(d, scratch)
    b = run_fold(d, scratch, in_place=True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    check_fold(d, *b)
    assert int(scratch[:4].view(torch.int32).item()) == 0


def test_fold_fallback_to_two_kernels(cuda_device):
    # With the CUDA-core kernel selected the call runs that GEMV and then the separate
    # add-RMSNorm kernel: the same outputs within the bounds, the scratch untouched.
    d = make(14336, 4096, seed=62)
    scratch = fd.fold_scratch()
    prev = fd.set_gemv_path("cuda_core")
    try:
        out = run_fold(d, scratch)
    finally:
        fd.set_gemv_path(prev)
    check_fold(d, *out)
    assert int(scratch.sum().item()) == 0


def test_fold_in_a_graph_with_pdl(cuda_device):
    # Three folded calls back to back in a CUDA graph with programmatic dependent launch
    # (the counter is reused by each), equal to eager calls bit for bit.
    d = make(14336, 4096, seed=63)
    g, u = dev_bf16(d["gate"]), dev_bf16(d["up"])
    q, s = dev_i32(d["qweight"]), dev_bf16(d["scales"])
    w = dev_bf16(d["rms_weight"])
    res0 = dev_bf16(d["residual"])
    scratch = fd.fold_scratch()
    outs = [torch.empty((1, 4096), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    norms = [torch.empty_like(outs[0]) for _ in range(3)]
    res = res0.clone()

    def chain():
        for i in range(3):
            fd.swiglu_w4a16_gemv_add_rmsnorm(g, u, q, s, res, w, EPS, scratch, y=outs[i],
                                             normed=norms[i], residual_out=res)

    stream = torch.cuda.Stream()
    prev = fd.set_pdl(True)
    try:
        with torch.cuda.stream(stream):
            chain()
        stream.synchronize()
        eager = [host_bits(t) for t in outs + norms + [res]]
        res.copy_(res0)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            chain()
        res.copy_(res0)
        graph.replay()
        torch.cuda.synchronize()
    finally:
        fd.set_pdl(prev)
    for a, b in zip(eager, [host_bits(t) for t in outs + norms + [res]]):
        assert np.array_equal(a, b)
    assert int(scratch[:4].view(torch.int32).item()) == 0


def test_fold_wait_timeout_gives_nan_and_resets(cuda_device):
    # A bounded wait that runs out (FD_LAUNCH_TEST_WAIT_TIMEOUT) makes every output NaN,
    # the normalised row too, and still leaves the counter at zero for the next call.
    lib = fd.load_library()
    d = make(14336, 4096, seed=64)
    scratch = fd.fold_scratch()
    run_fold(d, scratch)
    fd.device_status(clear=True)
    flags = lib.fd_get_launch_flags()
    lib.fd_set_launch_flags(flags | _lib.FD_LAUNCH_TEST_WAIT_TIMEOUT)
    try:
        y, normed, _ = run_fold(d, scratch)
    finally:
        lib.fd_set_launch_flags(flags)
    assert np.all(np.isnan(oracle.bf16_to_f32(y))) and np.all(np.isnan(oracle.bf16_to_f32(normed)))
    assert fd.device_status(clear=True) & _lib.FD_DEVICE_STATUS_WAIT_TIMEOUT
    assert int(scratch[:4].view(torch.int32).item()) == 0
    check_fold(d, *run_fold(d, scratch))
