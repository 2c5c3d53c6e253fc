"""ctypes loader for ``libfd.so`` (argument marshalling only; no compute here)."""

from __future__ import annotations

import ctypes
import threading
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "libfd.so"

FD_OK = 0
FD_ERR_NULL = 1
FD_ERR_SHAPE = 2
FD_ERR_ALIGN = 3
FD_ERR_UNSUPPORTED = 4
FD_ERR_CUDA = 5
FD_ERR_OVERLAP = 6

FD_GEMV_AUTO = 0
FD_GEMV_CUDA_CORE = 1
FD_GEMV_BULK = 2
FD_GEMV_TENSOR = 3

FD_LAUNCH_PDL = 1
FD_LAUNCH_TEST_FAIL = 256
FD_LAUNCH_TEST_WAIT_TIMEOUT = 512
FD_DEVICE_STATUS_WAIT_TIMEOUT = 1

FD_MAX_K = 32768
FD_MAX_M = 256
FD_MAX_HIDDEN = 32768
FD_NVFP4_MAX_K = 16384
FD_FOLD_SCRATCH_BYTES = 4096
FD_STEP_MAX_LAYERS = 1024




def step_scratch_bytes(n_layers: int, hidden: int) -> int:
    """FD_STEP_SCRATCH_BYTES(n_layers, hidden) of include/fd.h: the layer counters padded
    to 16 bytes, then two rows of 32-bit tagged h words."""
    return (n_layers * 4 + 15) // 16 * 16 + hidden * 8

# Every symbol include/fd.h declares, with its ctypes signature.
_VP = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "fd_swiglu_w4a16_gemv": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    "fd_swiglu_w4a16_gemv_residual": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    "fd_swiglu_w4a16_gemv_add_rmsnorm": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_float,
                                             _VP, _VP, _VP, _I, _I, _I, _VP]),
    "fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                                     ctypes.c_float, _VP, _VP, _I, _I, _I, _VP]),
    "fd_w4a16_gate_up_gemv": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP]),
    "fd_copy": (_I, [_VP, _VP, ctypes.c_size_t, _VP]),
    "fd_copy_rows": (_I, [_VP, ctypes.c_size_t, _VP, ctypes.c_size_t, ctypes.c_size_t,
                          ctypes.c_size_t, _VP]),
    "fd_debug_plan_gemv": (_I, [_VP, _I, _I, _I, _I, _I, _VP]),
    "fd_device_status": (_I, [_VP, _VP, _I]),
    "fd_decode_mlp_step": (_I, [_VP, _I, _VP, _VP, ctypes.c_float, _I, _I, _I, _VP, _VP]),
    "fd_debug_plan_step": (_I, [_VP, _I, _I, _I, _VP]),
    "fd_debug_plan_tc": (_I, [_I, _I, _I, _I, _I, _VP]),
    "fd_nvfp4_scaled_mm": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _VP]),
    "fd_debug_plan_nvfp4": (_I, [_I, _I, _I, _I, _VP]),
    "fd_add_rmsnorm": (_I, [_VP, _VP, _VP, ctypes.c_float, _VP, _VP, _I, _I, _VP]),
    "fd_w4_dequant_debug": (_I, [_VP, _VP, _VP, _I, _I, _I, _VP]),
    "fd_status_string": (ctypes.c_char_p, [_I]),
    "fd_last_cuda_error": (_I, []),
    "fd_version": (_I, []),
    "fd_set_gemv_path": (_I, [_I]),
    "fd_get_gemv_path": (_I, []),
    "fd_gemv_uses_tensor_cores": (_I, [_I, _I, _I, _I]),
    "fd_set_launch_flags": (_I, [ctypes.c_uint]),
    "fd_get_launch_flags": (ctypes.c_uint, []),
}


class FdLibraryMissing(RuntimeError):
    """libfd.so is not built: the fused kernels have no fallback and cannot run."""


class FdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: Path | None = None) -> ctypes.CDLL:
    """Load libfd.so once and attach the signatures. Raises FdLibraryMissing if absent."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = Path(path) if path is not None else LIB_PATH
        if not p.exists():
            raise FdLibraryMissing(
                f"{p} is missing; build it with memory_bound_decode_fd_gb300.build.build() "
                "(nvcc, sm_103a). There is no CPU fallback."
            )
        lib = ctypes.CDLL(str(p))
        for name, (restype, argtypes) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = restype
            fn.argtypes = argtypes
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().fd_status_string(int(status)).decode()


def check(status: int) -> None:
    if status != FD_OK:
        msg = status_string(status)
        if status == FD_ERR_CUDA:
            msg += f" (cudaError {load().fd_last_cuda_error()})"
        raise FdError(status, msg)
