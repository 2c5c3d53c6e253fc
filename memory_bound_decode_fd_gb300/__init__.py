"""fd - fused memory-bound decode kernels for GB300 (sm_103a).

* ``swiglu_w4a16_gemv``: y = (silu(g) * u) . dequant(W_int4)^T, one kernel, int4 in HBM only.
* ``swiglu_w4a16_gemv_residual``: the same GEMV with a residual-add epilogue (out =
  residual + y, the new residual stream written by the down projection).
* ``w4a16_gate_up_gemv``: the gate and up projections as one W4A16 GEMV (horizontal
  fusion), writing the g and u that ``swiglu_w4a16_gemv`` consumes.
* ``add_rmsnorm``: residual add + RMSNorm, one pass, two outputs.
* ``swiglu_w4a16_gemv_add_rmsnorm``: the GEMV with the next layer's add-RMSNorm folded into
  its tail (one launch per decode layer).
* ``nvfp4_scaled_mm``: the NVFP4 (packed FP4, E4M3 1x16 block scales) matmul with its fp32
  output multiplier folded in, on the tensor cores' block-scaled MMA.
* ``decode_mlp_step``: L layers of the two, in stream order.
* ``decode_mlp_step_persistent``: the same L layers as one persistent launch, bit-identical.

The compute runs in ``libfd.so`` (C ABI in ``include/fd.h``); this package marshals
PyTorch CUDA tensors into it. Build the library with ``build.build()``. There is no CPU
fallback: calling a kernel without the library raises ``FdLibraryMissing``.
"""

from ._lib import (  # noqa: F401
    FD_ERR_ALIGN,
    FD_ERR_CUDA,
    FD_ERR_NULL,
    FD_ERR_OVERLAP,
    FD_ERR_SHAPE,
    FD_ERR_UNSUPPORTED,
    FD_LAUNCH_TEST_FAIL,
    FD_MAX_HIDDEN,
    FD_MAX_K,
    FD_MAX_M,
    FD_NVFP4_MAX_K,
    FD_OK,
    LIB_PATH,
    FdError,
    FdLibraryMissing,
    status_string,
)
from ._lib import load as load_library  # noqa: F401
from .kernels import (  # noqa: F401
    GEMV_PATHS,
    add_rmsnorm,
    copy,
    copy_rows,
    decode_mlp_step,
    decode_mlp_step_persistent,
    device_status,
    fold_scratch,
    gemv_uses_tensor_cores,
    nvfp4_scaled_mm,
    set_gemv_path,
    set_pdl,
    step_layer_table,
    step_scratch,
    swiglu_w4a16_gemv,
    swiglu_w4a16_gemv_add_rmsnorm,
    swiglu_w4a16_gemv_add_rmsnorm_noalloc,
    swiglu_w4a16_gemv_residual,
    w4_dequant_debug,
    w4a16_gate_up_gemv,
)
from .packing import pack_int4  # noqa: F401
from .traffic import (  # noqa: F401
    add_rmsnorm_bytes,
    decode_step_bytes,
    gate_up_bytes,
    gemv_bytes,
    gemv_flops,
    nvfp4_bytes,
    nvfp4_flops,
)

__version__ = "1.0.0"
