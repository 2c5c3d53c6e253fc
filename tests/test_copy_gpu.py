"""fd_copy through the C ABI: device <-> device and pinned host <-> device, bit for bit,
for one vector, a ragged count and a decode step's input block, without touching the
bytes around the destination; and under programmatic dependent launch after a kernel
that writes the source. fd_copy_rows: rows at different pitches on both sides (the decode
step's interleaved gate and up rows), from device, pinned and pageable host memory, with
the bytes between the destination rows untouched."""

import pytest
import torch

import memory_bound_decode_fd_gb300 as fd

pytestmark = pytest.mark.gpu

SIZES = [16, 16 * 12345, 1_851_392]  # one vector, ragged, 32 layers of gate/up + x + residual


def _src(n, device):
    g = torch.Generator().manual_seed(n)
    t = torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)
    return t.to(device) if device == "cuda" else t.pin_memory()


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("src_dev,dst_dev", [("cuda", "cuda"), ("pinned", "cuda"), ("cuda", "pinned")])
def test_copy_bit_exact_with_guards(cuda_device, n, src_dev, dst_dev):
    src = _src(n, src_dev)
    guard = 64
    if dst_dev == "cuda":
        buf = torch.full((n + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
    else:
        buf = torch.full((n + 2 * guard,), 0xA5, dtype=torch.uint8).pin_memory()
    dst = buf[guard:guard + n]
    fd.copy(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src.cpu())
    rest = torch.cat([buf[:guard], buf[guard + n:]]).cpu()
    assert bool((rest == 0xA5).all())


def test_copy_with_pdl_after_a_writing_kernel(cuda_device):
    # the source is written by the kernel just before (add_rmsnorm's residual_out); the
    # copy must read it only after that kernel completes
    hidden = 4096
    x = torch.randn((1, hidden), device="cuda").to(torch.bfloat16)
    r = torch.randn((1, hidden), device="cuda").to(torch.bfloat16)
    w = torch.ones((hidden,), device="cuda", dtype=torch.bfloat16)
    out, h = torch.empty_like(x), torch.empty_like(x)
    host = torch.zeros((1, hidden), dtype=torch.bfloat16).pin_memory()
    prev = fd.set_pdl(True)
    try:
        for _ in range(3):
            h.zero_()
            fd.add_rmsnorm(x, r, w, 1e-5, out=out, residual_out=h)
            fd.copy(host, h)
            torch.cuda.synchronize()
            assert torch.equal(host.view(torch.int16), h.cpu().view(torch.int16))
    finally:
        fd.set_pdl(prev)
    expect = (x.float() + r.float()).to(torch.bfloat16).cpu()
    assert torch.equal(host.view(torch.int16), expect.view(torch.int16))


@pytest.mark.parametrize("rows,width,src_kind,dst_kind", [
    (1, 8, "cuda", "cuda"),
    (32, 14336, "pinned", "cuda"),    # a decode step's gate rows into the interleaved block
    (32, 14336, "pageable", "cuda"),  # host memory a kernel cannot reach: cudaMemcpy2DAsync
    (7, 24, "cuda", "pinned"),
])
def test_copy_rows_strided(cuda_device, rows, width, src_kind, dst_kind):
    g = torch.Generator().manual_seed(rows * width)
    src_full = torch.randint(-30000, 30000, (rows, 3 * width), dtype=torch.int16, generator=g)
    src = src_full[:, width:2 * width]  # pitch 3 x width
    if src_kind == "cuda":
        src_full = src_full.cuda()
        src = src_full[:, width:2 * width]
    elif src_kind == "pinned":
        src_full = src_full.pin_memory()
        src = src_full[:, width:2 * width]
    fill = torch.full((rows, 2, width), 0x5A5A, dtype=torch.int16)
    buf = fill.cuda() if dst_kind == "cuda" else fill.pin_memory()
    dst = buf[:, 0, :]  # pitch 2 x width: every other row of the buffer is a guard
    fd.copy_rows(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), src.cpu())
    assert bool((buf[:, 1, :].cpu() == 0x5A5A).all())


def test_copy_rows_with_pdl_after_a_writing_kernel(cuda_device):
    # the rows are written by the kernel just before (add_rmsnorm's residual_out, 4 rows);
    # the strided copy must read them only after that kernel completes
    rows, hidden = 4, 1024
    x = torch.randn((rows, hidden), device="cuda").to(torch.bfloat16)
    r = torch.randn((rows, hidden), device="cuda").to(torch.bfloat16)
    w = torch.ones((hidden,), device="cuda", dtype=torch.bfloat16)
    out, h = torch.empty_like(x), torch.empty_like(x)
    host = torch.zeros((rows, 2, hidden), dtype=torch.bfloat16).pin_memory()
    prev = fd.set_pdl(True)
    try:
        for _ in range(3):
            h.zero_()
            fd.add_rmsnorm(x, r, w, 1e-5, out=out, residual_out=h)
            fd.copy_rows(host[:, 1, :], h)
            torch.cuda.synchronize()
            assert torch.equal(host[:, 1, :].view(torch.int16), h.cpu().view(torch.int16))
    finally:
        fd.set_pdl(prev)
    expect = (x.float() + r.float()).to(torch.bfloat16).cpu()
    assert torch.equal(host[:, 1, :].view(torch.int16), expect.view(torch.int16))
    assert not host[:, 0, :].view(torch.int16).any()  # the rows between were not written
