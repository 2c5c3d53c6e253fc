"""Host-side tests (no GPU): the C-ABI library loads and exports every symbol the header
declares, rejects bad arguments before any CUDA call, and the Python binding, packing,
input generators and byte models behave."""

import ctypes
import re
from pathlib import Path

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
from memory_bound_decode_fd_gb300 import _lib, inputs, traffic

HEADER = Path(__file__).resolve().parent.parent / "include" / "fd.h"


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fd_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fd_swiglu_w4a16_gemv", "fd_swiglu_w4a16_gemv_residual", "fd_add_rmsnorm",
              "fd_status_string", "fd_w4_dequant_debug"):
        assert n in names


def test_library_exports_every_declared_symbol(fdlib):
    for name in declared_functions():
        assert hasattr(fdlib, name), name
        assert name in _lib.SIGNATURES, name


def test_header_constants_match_binding():
    text = HEADER.read_text()
    for name in ("FD_MAX_K", "FD_MAX_M", "FD_MAX_HIDDEN", "FD_LAUNCH_PDL", "FD_LAUNCH_TEST_FAIL",
                 "FD_STEP_MAX_LAYERS",
                 "FD_LAUNCH_TEST_WAIT_TIMEOUT", "FD_DEVICE_STATUS_WAIT_TIMEOUT", "FD_NVFP4_MAX_K"):
        m = re.search(rf"#define {name} (\d+)", text)
        assert int(m.group(1)) == getattr(_lib, name)
    for name in ("FD_OK", "FD_ERR_NULL", "FD_ERR_SHAPE", "FD_ERR_ALIGN", "FD_ERR_UNSUPPORTED",
                 "FD_ERR_CUDA", "FD_ERR_OVERLAP"):
        m = re.search(rf"{name} = (\d+)", text)
        assert int(m.group(1)) == getattr(_lib, name)


def test_status_strings(fdlib):
    for code in range(0, 7):
        s = fdlib.fd_status_string(code).decode()
        assert s.startswith("FD_")
    assert fdlib.fd_status_string(99).decode() == "fd: unknown status"
    assert fdlib.fd_version() >= 10000


# Fake, 16-byte aligned "device" addresses: every call below is rejected by the host-side
# checks before any CUDA call, so nothing is dereferenced or launched.
A = 0x10000000
B = 0x20000000
C = 0x30000000
D = 0x40000000
E = 0x50000000


def gemv(lib, gate=A, up=B, qw=C, sc=D, out=E, M=1, K=1024, N=256, group=128):
    return lib.fd_swiglu_w4a16_gemv(gate, up, qw, sc, out, M, K, N, group, None)


@pytest.mark.parametrize("kw,status", [
    (dict(gate=None), _lib.FD_ERR_NULL),
    (dict(up=None), _lib.FD_ERR_NULL),
    (dict(qw=None), _lib.FD_ERR_NULL),
    (dict(sc=None), _lib.FD_ERR_NULL),
    (dict(out=None), _lib.FD_ERR_NULL),
    (dict(M=-1), _lib.FD_ERR_SHAPE),
    (dict(N=-1), _lib.FD_ERR_SHAPE),
    (dict(M=0, K=1000), _lib.FD_ERR_SHAPE),    # an empty call still has valid sizes
    (dict(K=0), _lib.FD_ERR_SHAPE),
    (dict(K=1000), _lib.FD_ERR_SHAPE),
    (dict(K=1024, group=48), _lib.FD_ERR_SHAPE),
    (dict(K=1056, group=128), _lib.FD_ERR_SHAPE),
    (dict(group=0), _lib.FD_ERR_SHAPE),
    (dict(M=257), _lib.FD_ERR_UNSUPPORTED),
    (dict(K=32768 + 128), _lib.FD_ERR_UNSUPPORTED),
    (dict(gate=A + 2), _lib.FD_ERR_ALIGN),
    (dict(out=E + 8), _lib.FD_ERR_ALIGN),
    (dict(qw=C + 4), _lib.FD_ERR_ALIGN),
    (dict(out=A), _lib.FD_ERR_OVERLAP),
    (dict(out=C + 16), _lib.FD_ERR_OVERLAP),
])
def test_gemv_rejects_bad_arguments_without_launching(fdlib, kw, status):
    assert gemv(fdlib, **kw) == status


F = 0x60000000


def gemv_res(lib, gate=A, up=B, qw=C, sc=D, res=F, out=E, M=1, K=1024, N=256, group=128):
    return lib.fd_swiglu_w4a16_gemv_residual(gate, up, qw, sc, res, out, M, K, N, group, None)


@pytest.mark.parametrize("kw,status", [
    (dict(res=None), _lib.FD_ERR_NULL),
    (dict(gate=None), _lib.FD_ERR_NULL),
    (dict(M=-1), _lib.FD_ERR_SHAPE),
    (dict(K=1000), _lib.FD_ERR_SHAPE),
    (dict(M=257), _lib.FD_ERR_UNSUPPORTED),
    (dict(res=F + 2), _lib.FD_ERR_ALIGN),
    (dict(res=E + 16), _lib.FD_ERR_OVERLAP),   # partial overlap with out (== out is allowed)
    (dict(res=A), _lib.FD_ERR_OVERLAP),        # residual over gate
    (dict(res=B + 64), _lib.FD_ERR_OVERLAP),   # residual inside up
    (dict(res=C + 32), _lib.FD_ERR_OVERLAP),   # residual inside qweight
    (dict(res=D), _lib.FD_ERR_OVERLAP),        # residual over scales
    (dict(out=A), _lib.FD_ERR_OVERLAP),        # out over gate
])
def test_gemv_residual_rejects_bad_arguments_without_launching(fdlib, kw, status):
    assert gemv_res(fdlib, **kw) == status


def gate_up(lib, x=A, qw=C, sc=D, g=E, u=F, M=1, K=1024, I=128, group=128):
    return lib.fd_w4a16_gate_up_gemv(x, qw, sc, g, u, M, K, I, group, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), _lib.FD_ERR_NULL),
    (dict(g=None), _lib.FD_ERR_NULL),
    (dict(u=None), _lib.FD_ERR_NULL),
    (dict(qw=None), _lib.FD_ERR_NULL),
    (dict(I=-1), _lib.FD_ERR_SHAPE),
    (dict(M=-1), _lib.FD_ERR_SHAPE),
    (dict(K=1000), _lib.FD_ERR_SHAPE),
    (dict(group=48), _lib.FD_ERR_SHAPE),
    (dict(M=257), _lib.FD_ERR_UNSUPPORTED),
    (dict(I=2**30), _lib.FD_ERR_UNSUPPORTED),
    (dict(x=A + 2), _lib.FD_ERR_ALIGN),
    (dict(u=F + 8), _lib.FD_ERR_ALIGN),
    (dict(u=E + 64), _lib.FD_ERR_OVERLAP),     # up over gate
    (dict(g=A), _lib.FD_ERR_OVERLAP),          # gate over x
    (dict(u=C + 16), _lib.FD_ERR_OVERLAP),     # up inside qweight
    (dict(g=D), _lib.FD_ERR_OVERLAP),          # gate over scales
])
def test_gate_up_rejects_bad_arguments_without_launching(fdlib, kw, status):
    assert gate_up(fdlib, **kw) == status


@pytest.mark.parametrize("args,status", [
    ((None, B, 1024), _lib.FD_ERR_NULL),
    ((A, None, 1024), _lib.FD_ERR_NULL),
    ((A, B, 1000), _lib.FD_ERR_SHAPE),
    ((A + 8, B, 1024), _lib.FD_ERR_ALIGN),
    ((A, B + 4, 1024), _lib.FD_ERR_ALIGN),
    ((A, A + 512, 1024), _lib.FD_ERR_OVERLAP),
])
def test_copy_rejects_bad_arguments_without_launching(fdlib, args, status):
    assert fdlib.fd_copy(*args, None) == status


@pytest.mark.parametrize("args,status", [
    # dst, dst_pitch, src, src_pitch, row_bytes, rows
    ((None, 64, B, 64, 32, 4), _lib.FD_ERR_NULL),
    ((A, 64, None, 64, 32, 4), _lib.FD_ERR_NULL),
    ((A, 64, B, 64, 24, 4), _lib.FD_ERR_SHAPE),       # row not a multiple of 16 bytes
    ((A, 40, B, 64, 32, 4), _lib.FD_ERR_SHAPE),       # pitch not a multiple of 16
    ((A, 16, B, 64, 32, 4), _lib.FD_ERR_SHAPE),       # pitch below the row
    ((A + 8, 64, B, 64, 32, 4), _lib.FD_ERR_ALIGN),
    ((A, 64, B + 4, 64, 32, 4), _lib.FD_ERR_ALIGN),
    ((A, 64, A + 32, 64, 32, 4), _lib.FD_ERR_OVERLAP),  # interleaved rows
    ((A + 192, 64, A, 64, 32, 4), _lib.FD_ERR_OVERLAP),  # the last source row meets dst
])
def test_copy_rows_rejects_bad_arguments_without_launching(fdlib, args, status):
    assert fdlib.fd_copy_rows(*args, None) == status


def test_copy_rows_empty_and_failed_launch(fdlib):
    assert fdlib.fd_copy_rows(None, 0, None, 0, 0, 4, None) == _lib.FD_OK
    assert fdlib.fd_copy_rows(None, 0, None, 0, 32, 0, None) == _lib.FD_OK
    prev = fdlib.fd_get_launch_flags()
    assert fdlib.fd_set_launch_flags(prev | _lib.FD_LAUNCH_TEST_FAIL) == _lib.FD_OK
    try:
        assert fdlib.fd_copy_rows(A, 64, B, 64, 32, 4, None) == _lib.FD_ERR_CUDA
    finally:
        fdlib.fd_set_launch_flags(prev)


def rms(lib, x=A, r=B, w=C, eps=1e-6, out=D, rout=E, rows=4, hidden=4096):
    return lib.fd_add_rmsnorm(x, r, w, ctypes.c_float(eps), out, rout, rows, hidden, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), _lib.FD_ERR_NULL),
    (dict(w=None), _lib.FD_ERR_NULL),
    (dict(rout=None), _lib.FD_ERR_NULL),
    (dict(rows=-1), _lib.FD_ERR_SHAPE),
    (dict(rows=0, hidden=12), _lib.FD_ERR_SHAPE),
    (dict(hidden=12), _lib.FD_ERR_SHAPE),
    (dict(hidden=0), _lib.FD_ERR_SHAPE),
    (dict(eps=-1e-6), _lib.FD_ERR_SHAPE),
    (dict(eps=float("nan")), _lib.FD_ERR_SHAPE),
    (dict(eps=float("inf")), _lib.FD_ERR_SHAPE),
    (dict(hidden=32768 + 8), _lib.FD_ERR_UNSUPPORTED),
    (dict(r=B + 2), _lib.FD_ERR_ALIGN),
    (dict(rout=E + 4), _lib.FD_ERR_ALIGN),
    (dict(out=E), _lib.FD_ERR_OVERLAP),            # both outputs in one buffer
    (dict(out=A + 16), _lib.FD_ERR_OVERLAP),       # partial overlap with x
    (dict(out=B), _lib.FD_ERR_OVERLAP),            # out over residual
    (dict(rout=A), _lib.FD_ERR_OVERLAP),           # residual_out over x
    (dict(rout=B + 32), _lib.FD_ERR_OVERLAP),      # partial overlap with residual
    (dict(w=D + 64), _lib.FD_ERR_OVERLAP),         # weight inside out
])
def test_rmsnorm_rejects_bad_arguments_without_launching(fdlib, kw, status):
    assert rms(fdlib, **kw) == status


def test_empty_calls_return_ok_without_reading_pointers(fdlib):
    # nothing to compute: FD_OK at once, NULL pointers never read, nothing launched
    N0 = None
    assert gemv(fdlib, gate=N0, up=N0, qw=N0, sc=N0, out=N0, M=0) == _lib.FD_OK
    assert gemv(fdlib, gate=N0, up=N0, qw=N0, sc=N0, out=N0, N=0) == _lib.FD_OK
    assert gemv_res(fdlib, gate=N0, up=N0, qw=N0, sc=N0, res=N0, out=N0, M=0) == _lib.FD_OK
    assert gate_up(fdlib, x=N0, qw=N0, sc=N0, g=N0, u=N0, M=0) == _lib.FD_OK
    assert gate_up(fdlib, x=N0, qw=N0, sc=N0, g=N0, u=N0, I=0) == _lib.FD_OK
    assert fdlib.fd_copy(N0, N0, 0, None) == _lib.FD_OK
    assert rms(fdlib, x=N0, r=N0, w=N0, out=N0, rout=N0, rows=0) == _lib.FD_OK
    assert fdlib.fd_w4_dequant_debug(N0, N0, N0, 1024, 0, 128, None) == _lib.FD_OK


def test_dequant_debug_rejects_bad_arguments(fdlib):
    f = fdlib.fd_w4_dequant_debug
    assert f(A, B, None, 1024, 4, 128, None) == _lib.FD_ERR_NULL
    assert f(A, B, C, 1000, 4, 128, None) == _lib.FD_ERR_SHAPE
    assert f(A + 4, B, C, 1024, 4, 128, None) == _lib.FD_ERR_ALIGN
    assert f(A, B, A, 1024, 4, 128, None) == _lib.FD_ERR_OVERLAP


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(_lib.FdLibraryMissing):
        _lib.load(tmp_path / "libfd.so")


def test_binding_rejects_cpu_tensors():
    g = torch.zeros(1, 64, dtype=torch.bfloat16)
    q = torch.zeros(4, 8, dtype=torch.int32)
    s = torch.zeros(4, 2, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fd.swiglu_w4a16_gemv(g, g, q, s, group=32)
    with pytest.raises(ValueError, match="CUDA"):
        fd.add_rmsnorm(g, g, g[0], 1e-6)


class _FakeCuda:
    """Stands in for a CUDA tensor or stream in the binding's device checks."""

    def __init__(self, index, is_cuda=True):
        self.is_cuda = is_cuda
        self.device = torch.device("cuda", index) if is_cuda else torch.device("cpu")
        self.cuda_stream = 1234


def test_binding_requires_one_device_per_call():
    from memory_bound_decode_fd_gb300 import kernels
    a, b, host = _FakeCuda(0), _FakeCuda(1), _FakeCuda(None, is_cuda=False)
    assert kernels._device_of(a, a, host) == torch.device("cuda", 0)
    assert kernels._device_of(host, host) is None
    with pytest.raises(ValueError, match="one device"):
        kernels._device_of(a, b)
    # a stream must belong to the tensors' device
    assert kernels._stream_handle(_FakeCuda(1), torch.device("cuda", 1)).value == 1234
    with pytest.raises(ValueError, match="stream is on"):
        kernels._stream_handle(_FakeCuda(0), torch.device("cuda", 1))


def test_pack_int4_layout_and_checks():
    q = np.arange(-8, 8, dtype=np.int8).reshape(2, 8)
    w = fd.pack_int4(q).view(np.uint32)
    assert w[0, 0] == 0xFEDCBA98  # -8..-1 -> nibbles 8..F, nibble 0 first
    assert w[1, 0] == 0x76543210
    with pytest.raises(ValueError):
        fd.pack_int4(np.zeros((2, 7), np.int8))
    with pytest.raises(ValueError):
        fd.pack_int4(np.full((1, 8), 8, np.int8))


def test_inputs_are_deterministic_and_shaped():
    a = inputs.gemv_inputs(1, 1024, 256, 128, seed=0)
    b = inputs.gemv_inputs(1, 1024, 256, 128, seed=0)
    for k in ("gate", "up", "qweight", "scales"):
        assert np.array_equal(a[k], b[k])
    assert a["gate"].shape == (1, 1024) and a["gate"].dtype == np.uint16
    assert a["qweight"].shape == (256, 128) and a["qweight"].dtype == np.int32
    assert a["scales"].shape == (256, 8)
    s = a["scales"].astype(np.uint32) << 16
    sf = s.view(np.float32)
    assert sf.min() >= 0.0049 and sf.max() <= 0.0201  # bounds after bf16 rounding
    r = inputs.rmsnorm_inputs(4, 64, seed=1)
    assert r["x"].shape == (4, 64) and r["weight"].shape == (64,)


def test_ideal_bytes_of_the_workloads():
    assert traffic.gemv_bytes(1, 1024, 256, 128) == 139_776
    assert traffic.add_rmsnorm_bytes(8192, 4096) == 268_443_648
    assert traffic.gemv_bytes(1, 9216, 2560, 128) == 12_207_104
    assert traffic.decode_step_bytes(32, 4096, 14336, 128) == 972_292_096
    # gate/up of the same MLP: 28672 x 4096 int4 + scales + x + g and u
    assert traffic.gate_up_bytes(1, 4096, 14336, 128) == (
        28672 * 2048 + 28672 * 32 * 2 + 4096 * 2 + 28672 * 2)
    assert traffic.gemv_bytes(64, 14336, 4096, 128) == 34_471_936
    assert traffic.add_rmsnorm_bytes(64, 4096) == 2_105_344
