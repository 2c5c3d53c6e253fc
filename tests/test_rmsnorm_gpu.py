"""GPU parity of fd_add_rmsnorm against the CPU oracle, through the C ABI."""

import gc

import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
from memory_bound_decode_fd_gb300 import inputs
from fd_check import GuardedBuffer, check_add_rmsnorm, dev_bf16, host_bits

pytestmark = pytest.mark.gpu


def run(d, eps, out=None, residual_out=None):
    x, r, w = dev_bf16(d["x"]), dev_bf16(d["residual"]), dev_bf16(d["weight"])
    y, h = fd.add_rmsnorm(x, r, w, eps, out=out, residual_out=residual_out)
    torch.cuda.synchronize()
    return host_bits(y), host_bits(h)


def test_rmsnorm_8192x4096_full(cuda_device):
    # add-RMSNorm rows=8192 hidden=4096 eps=1e-6, seed 1: every output checked.
    d = inputs.rmsnorm_inputs(8192, 4096, seed=1)
    y, h = run(d, 1e-6)
    res = check_add_rmsnorm(y, h, d["x"], d["residual"], d["weight"], 1e-6)
    assert res["frac_exact"] > 0.99


def test_rmsnorm_batched_64x4096(cuda_device):
    d = inputs.batched_inputs()["rmsnorm"]
    y, h = run(d, 1e-5)
    check_add_rmsnorm(y, h, d["x"], d["residual"], d["weight"], 1e-5)


@pytest.mark.parametrize("rows,hidden", [
    (1, 4096), (1, 8), (3, 16), (5, 24), (7, 2048), (2, 2056), (9, 4104), (4, 8192),
    (3, 8200), (2, 16384), (2, 32768), (1000, 4096), (152 * 6 + 1, 4096), (4097, 512),
])
def test_rmsnorm_shapes(cuda_device, rows, hidden):
    d = inputs.rmsnorm_inputs(rows, hidden, seed=rows * 7 + hidden)
    for eps in (1e-6, 1e-5):
        y, h = run(d, eps)
        check_add_rmsnorm(y, h, d["x"], d["residual"], d["weight"], eps)


def test_rmsnorm_in_place(cuda_device):
    d = inputs.rmsnorm_inputs(33, 4096, seed=3)
    x, r, w = dev_bf16(d["x"]), dev_bf16(d["residual"]), dev_bf16(d["weight"])
    y, h = fd.add_rmsnorm(x, r, w, 1e-6, out=x, residual_out=r)
    torch.cuda.synchronize()
    assert y.data_ptr() == x.data_ptr() and h.data_ptr() == r.data_ptr()
    check_add_rmsnorm(host_bits(x), host_bits(r), d["x"], d["residual"], d["weight"], 1e-6)


def test_rmsnorm_guard_bands_untouched(cuda_device):
    d = inputs.rmsnorm_inputs(17, 4104, seed=4)
    yb, hb = GuardedBuffer((17, 4104)), GuardedBuffer((17, 4104))
    run(d, 1e-6, out=yb.tensor, residual_out=hb.tensor)
    assert yb.guards_intact() and hb.guards_intact()
    check_add_rmsnorm(host_bits(yb.tensor), host_bits(hb.tensor), d["x"], d["residual"],
                      d["weight"], 1e-6)


def test_rmsnorm_allocates_nothing(cuda_device):
    d = inputs.rmsnorm_inputs(512, 4096, seed=5)
    x, r, w = dev_bf16(d["x"]), dev_bf16(d["residual"]), dev_bf16(d["weight"])
    y, h = torch.empty_like(x), torch.empty_like(x)
    fd.add_rmsnorm(x, r, w, 1e-6, out=y, residual_out=h)
    gc.collect()  # tensors of earlier tests are freed now, not during the measurement
    gc.disable()
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    torch.cuda.reset_peak_memory_stats()
    for _ in range(5):
        fd.add_rmsnorm(x, r, w, 1e-6, out=y, residual_out=h)
    torch.cuda.synchronize()
    gc.enable()
    assert torch.cuda.memory_allocated() == before
    assert torch.cuda.max_memory_allocated() == before
    assert torch.cuda.mem_get_info()[0] == free_before


def test_rmsnorm_rejects_partial_overlap(cuda_device):
    d = inputs.rmsnorm_inputs(4, 64, seed=6)
    x, r, w = dev_bf16(d["x"]), dev_bf16(d["residual"]), dev_bf16(d["weight"])
    big = torch.empty((5, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fd.FdError) as e:
        fd.add_rmsnorm(x, r, w, 1e-6, out=big[:4], residual_out=big[1:5])
    assert e.value.status == fd.FD_ERR_OVERLAP
