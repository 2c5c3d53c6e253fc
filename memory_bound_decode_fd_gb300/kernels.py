"""Python binding of the fd C ABI (include/fd.h) for PyTorch CUDA tensors.

Argument marshalling only: every step of the computation runs in libfd.so's CUDA
kernels, launched on the caller's current PyTorch stream. PyTorch provides the device
memory and the stream; nothing here computes.
"""

from __future__ import annotations

import contextlib
import ctypes

import torch

from . import _lib


GEMV_PATHS = {"auto": _lib.FD_GEMV_AUTO, "cuda_core": _lib.FD_GEMV_CUDA_CORE,
              "bulk": _lib.FD_GEMV_BULK, "tensor": _lib.FD_GEMV_TENSOR}


def set_gemv_path(path: str) -> str:
    """Select the GEMV kernel process-wide ("auto", "cuda_core", "bulk" or "tensor"); returns the
    previous selection. See fd_set_gemv_path in include/fd.h."""
    lib = _lib.load()
    prev = {v: k for k, v in GEMV_PATHS.items()}[lib.fd_get_gemv_path()]
    _lib.check(lib.fd_set_gemv_path(GEMV_PATHS[path]))
    return prev


def gemv_uses_tensor_cores(M: int, K: int, N: int, group: int = 128) -> bool:
    """Whether, under the current kernel selection, this GEMV shape runs on the
    tensor-core kernel (bf16-rounded MMA operands). See fd_gemv_uses_tensor_cores."""
    return bool(_lib.load().fd_gemv_uses_tensor_cores(M, K, N, group))


def set_pdl(enabled: bool) -> bool:
    """Turn programmatic dependent launch on or off for every later fd launch in this
    process; returns the previous setting. See FD_LAUNCH_PDL in include/fd.h for the
    condition under which it is safe (no in-flight kernel writes the weight tensors)."""
    lib = _lib.load()
    prev = bool(lib.fd_get_launch_flags() & _lib.FD_LAUNCH_PDL)
    _lib.check(lib.fd_set_launch_flags(_lib.FD_LAUNCH_PDL if enabled else 0))
    return prev


def device_status(clear: bool = True, stream: torch.cuda.Stream | None = None) -> int:
    """The FD_DEVICE_STATUS_* bits kernels recorded on the current device since the last
    clear (a bounded wait that gave up sets FD_DEVICE_STATUS_WAIT_TIMEOUT). Synchronises
    `stream` (default: the current stream). See fd_device_status in include/fd.h."""
    lib = _lib.load()
    out = ctypes.c_uint(0)
    _lib.check(lib.fd_device_status(_stream_handle(stream, None), ctypes.byref(out), int(bool(clear))))
    return int(out.value)


def _device_of(*tensors) -> torch.device | None:
    """The one CUDA device of a call's CUDA tensors (None if it has none, e.g. a copy
    between two pinned host buffers). Tensors on two devices are an error: the kernels
    dereference every pointer on the device they run on."""
    devs = {t.device for t in tensors if t.is_cuda}
    if len(devs) > 1:
        raise ValueError(f"all CUDA tensors of a call must be on one device, got {sorted(map(str, devs))}")
    return devs.pop() if devs else None


def _stream_handle(stream, device: torch.device | None) -> ctypes.c_void_p:
    """The handle of `stream`, else of the current stream of `device`; a stream of
    another device is an error."""
    s = stream if stream is not None else torch.cuda.current_stream(device)
    if device is not None and s.device != device:
        raise ValueError(f"stream is on {s.device} but the tensors are on {device}")
    return ctypes.c_void_p(int(s.cuda_stream))


def _on_device(device: torch.device | None):
    """Make `device` current for the library call (it launches on, and reads the facts
    of, the calling thread's current device); a no-op when it already is."""
    if device is None or device.index is None or device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(device)


def _check_tensor(name: str, t: torch.Tensor, dtype: torch.dtype, shape: tuple | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the fd kernels have no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def swiglu_w4a16_gemv(
    gate: torch.Tensor,
    up: torch.Tensor,
    qweight: torch.Tensor,
    scales: torch.Tensor,
    out: torch.Tensor | None = None,
    group: int = 128,
    stream: torch.cuda.Stream | None = None,
) -> torch.Tensor:
    """out[m, n] = bf16(sum_k silu(gate[m, k]) * up[m, k] * q[n, k] * scales[n, k // group]).

    gate, up: bf16 [M, K]; qweight: int32 [N, K/8] (nibble j of word p = q[n, 8p + j]);
    scales: bf16 [N, K/group]; out: bf16 [M, N] (allocated if None).
    """
    if gate.dim() == 1:
        gate = gate.unsqueeze(0)
        up = up.unsqueeze(0)
    if gate.dim() != 2 or qweight.dim() != 2 or scales.dim() != 2:
        raise ValueError("gate/up must be [M, K]; qweight [N, K/8]; scales [N, K/group]")
    M, K = gate.shape
    N = qweight.shape[0]
    _check_tensor("gate", gate, torch.bfloat16)
    _check_tensor("up", up, torch.bfloat16, (M, K))
    _check_tensor("qweight", qweight, torch.int32, (N, K // 8))
    if group <= 0 or K % group != 0:
        raise ValueError(f"K={K} must be a multiple of group={group}")
    _check_tensor("scales", scales, torch.bfloat16, (N, K // group))
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=gate.device)
    _check_tensor("out", out, torch.bfloat16, (M, N))
    dev = _device_of(gate, up, qweight, scales, out)
    lib = _lib.load()
    with _on_device(dev):
        st = lib.fd_swiglu_w4a16_gemv(
            _ptr(gate), _ptr(up), _ptr(qweight), _ptr(scales), _ptr(out),
            int(M), int(K), int(N), int(group), _stream_handle(stream, dev),
        )
    _lib.check(st)
    return out


def swiglu_w4a16_gemv_residual(
    gate: torch.Tensor,
    up: torch.Tensor,
    qweight: torch.Tensor,
    scales: torch.Tensor,
    residual: torch.Tensor,
    out: torch.Tensor | None = None,
    group: int = 128,
    stream: torch.cuda.Stream | None = None,
) -> torch.Tensor:
    """The GEMV with a residual-add epilogue: out[m, n] = bf16(f32(residual[m, n]) +
    sum_k silu(gate[m, k]) * up[m, k] * q[n, k] * scales[n, k // group]), one rounding.

    residual: bf16 [M, N] (a 1-D tensor is one row); out may be residual (in place).
    Other arguments as ``swiglu_w4a16_gemv``.
    """
    if gate.dim() == 1:
        gate = gate.unsqueeze(0)
        up = up.unsqueeze(0)
    if residual.dim() == 1:
        residual = residual.unsqueeze(0)
    if gate.dim() != 2 or qweight.dim() != 2 or scales.dim() != 2:
        raise ValueError("gate/up must be [M, K]; qweight [N, K/8]; scales [N, K/group]")
    M, K = gate.shape
    N = qweight.shape[0]
    _check_tensor("gate", gate, torch.bfloat16)
    _check_tensor("up", up, torch.bfloat16, (M, K))
    _check_tensor("qweight", qweight, torch.int32, (N, K // 8))
    if group <= 0 or K % group != 0:
        raise ValueError(f"K={K} must be a multiple of group={group}")
    _check_tensor("scales", scales, torch.bfloat16, (N, K // group))
    _check_tensor("residual", residual, torch.bfloat16, (M, N))
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=gate.device)
    elif out.dim() == 1:
        out = out.unsqueeze(0)
    _check_tensor("out", out, torch.bfloat16, (M, N))
    dev = _device_of(gate, up, qweight, scales, residual, out)
    lib = _lib.load()
    with _on_device(dev):
        st = lib.fd_swiglu_w4a16_gemv_residual(
            _ptr(gate), _ptr(up), _ptr(qweight), _ptr(scales), _ptr(residual), _ptr(out),
            int(M), int(K), int(N), int(group), _stream_handle(stream, dev),
        )
    _lib.check(st)
    return out


def fold_scratch(device=None) -> torch.Tensor:
    """A zeroed scratch buffer for swiglu_w4a16_gemv_add_rmsnorm (FD_FOLD_SCRATCH_BYTES
    bytes); every completed call leaves it zero again. One per stream."""
    return torch.zeros(_lib.FD_FOLD_SCRATCH_BYTES, dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def swiglu_w4a16_gemv_add_rmsnorm(
    gate: torch.Tensor,
    up: torch.Tensor,
    qweight: torch.Tensor,
    scales: torch.Tensor,
    residual: torch.Tensor,
    rms_weight: torch.Tensor,
    eps: float,
    scratch: torch.Tensor,
    y: torch.Tensor | None = None,
    normed: torch.Tensor | None = None,
    residual_out: torch.Tensor | None = None,
    group: int = 128,
    stream: torch.cuda.Stream | None = None,
) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(y, normed, residual_out): the SwiGLU-W4A16 GEMV of one row with the next layer's
    residual add + RMSNorm folded into its tail: y = gemv(...), residual_out = bf16(y +
    residual), normed = RMSNorm(residual_out) * rms_weight. residual_out may be residual (in
    place). scratch: fold_scratch(). See fd_swiglu_w4a16_gemv_add_rmsnorm in include/fd.h."""
    if gate.dim() == 1:
        gate = gate.unsqueeze(0)
        up = up.unsqueeze(0)
    if residual.dim() == 1:
        residual = residual.unsqueeze(0)
    if gate.dim() != 2 or gate.shape[0] != 1 or qweight.dim() != 2 or scales.dim() != 2:
        raise ValueError("gate/up must be [1, K]; qweight [N, K/8]; scales [N, K/group]")
    K = gate.shape[1]
    N = qweight.shape[0]
    _check_tensor("gate", gate, torch.bfloat16)
    _check_tensor("up", up, torch.bfloat16, (1, K))
    _check_tensor("qweight", qweight, torch.int32, (N, K // 8))
    if group <= 0 or K % group != 0:
        raise ValueError(f"K={K} must be a multiple of group={group}")
    _check_tensor("scales", scales, torch.bfloat16, (N, K // group))
    _check_tensor("residual", residual, torch.bfloat16, (1, N))
    _check_tensor("rms_weight", rms_weight, torch.bfloat16, (N,))
    _check_tensor("scratch", scratch, torch.uint8, (_lib.FD_FOLD_SCRATCH_BYTES,))
    outs = []
    for name, t in (("y", y), ("normed", normed), ("residual_out", residual_out)):
        if t is None:
            t = torch.empty((1, N), dtype=torch.bfloat16, device=gate.device)
        elif t.dim() == 1:
            t = t.unsqueeze(0)
        _check_tensor(name, t, torch.bfloat16, (1, N))
        outs.append(t)
    y, normed, residual_out = outs
    dev = _device_of(gate, up, qweight, scales, residual, rms_weight, scratch, y, normed, residual_out)
    lib = _lib.load()
    with _on_device(dev):
        st = lib.fd_swiglu_w4a16_gemv_add_rmsnorm(
            _ptr(gate), _ptr(up), _ptr(qweight), _ptr(scales), _ptr(y), _ptr(residual),
            _ptr(rms_weight), ctypes.c_float(float(eps)), _ptr(normed), _ptr(residual_out),
            _ptr(scratch), int(K), int(N), int(group), _stream_handle(stream, dev),
        )
    _lib.check(st)
    return y, normed, residual_out


def step_layer_table(layers, normed, y, device=None) -> torch.Tensor:
    """The device array of fd_step_layer that decode_mlp_step_persistent reads: per layer
    the pointers (gate, up, qweight, scales, rms_weight, normed, y), as int64. ``layers``:
    dicts of gate and up [1, inter] (or [inter]), qweight [hidden, inter/8] int32, scales
    [hidden, inter/group] and rms_weight [hidden] bf16; ``normed`` and ``y``: per-layer
    [1, hidden] bf16 outputs. The tensors must stay alive while the table is used."""
    rows = []
    for i, (l, n, yy) in enumerate(zip(layers, normed, y)):
        hidden, k8 = l["qweight"].shape
        _check_tensor(f"layers[{i}].qweight", l["qweight"], torch.int32, (hidden, k8))
        for name in ("gate", "up"):
            _check_tensor(f"layers[{i}].{name}", l[name], torch.bfloat16)
            if l[name].numel() != 8 * k8:
                raise ValueError(f"layers[{i}].{name} must hold inter={8 * k8} elements")
        _check_tensor(f"layers[{i}].scales", l["scales"], torch.bfloat16)
        _check_tensor(f"layers[{i}].rms_weight", l["rms_weight"], torch.bfloat16, (hidden,))
        for name, t in (("normed", n), ("y", yy)):
            _check_tensor(f"{name}[{i}]", t, torch.bfloat16)
            if t.numel() != hidden:
                raise ValueError(f"{name}[{i}] must hold hidden={hidden} elements")
        ptrs = [l["gate"].data_ptr(), l["up"].data_ptr(), l["qweight"].data_ptr(),
                l["scales"].data_ptr(), l["rms_weight"].data_ptr(), n.data_ptr(), yy.data_ptr()]
        # the kernel reads these with 16-byte loads and bulk copies; the C ABI cannot check
        # pointers that live in device memory, so they are checked here
        for name, ptr in zip(("gate", "up", "qweight", "scales", "rms_weight", "normed", "y"), ptrs):
            if ptr % 16:
                raise ValueError(f"layers[{i}].{name} is not 16-byte aligned")
        rows.append(ptrs)
    dev = device if device is not None else layers[0]["qweight"].device
    return torch.tensor(rows, dtype=torch.int64, device=dev)


def step_scratch(n_layers: int, hidden: int, device=None) -> torch.Tensor:
    """The scratch of decode_mlp_step_persistent (a counter per layer and two rows of
    tagged h words; every call zeroes it)."""
    return torch.zeros(_lib.step_scratch_bytes(n_layers, hidden), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def decode_mlp_step_persistent(x, residual, table, eps, inter, group, scratch, stream=None):
    """A whole decode step in one launch (fd_decode_mlp_step): for every layer of
    ``table`` (step_layer_table), add-RMSNorm of (x_l, residual) into the layer's normed,
    then its GEMV into its y, with x_0 = x and x_{l+1} = y_l; ``residual`` is left as the
    last layer's h. Every output is bit-identical to decode_mlp_step's chain of separate
    calls. ``inter`` is the GEMV's K. Nothing is allocated here."""
    n_layers = int(table.shape[0])
    hidden = x.numel()
    _check_tensor("x", x, torch.bfloat16)
    _check_tensor("residual", residual, torch.bfloat16)
    if residual.numel() != hidden:
        raise ValueError("residual must hold hidden elements")
    _check_tensor("table", table, torch.int64, (n_layers, 7))
    _check_tensor("scratch", scratch, torch.uint8)
    if scratch.numel() < _lib.step_scratch_bytes(n_layers, hidden):
        raise ValueError("scratch is too small (step_scratch)")
    dev = _device_of(x, residual, table, scratch)
    lib = _lib.load()
    with _on_device(dev):
        st = lib.fd_decode_mlp_step(_ptr(table), n_layers, _ptr(x), _ptr(residual),
                                    ctypes.c_float(float(eps)), int(hidden), int(inter),
                                    int(group), _ptr(scratch), _stream_handle(stream, dev))
    _lib.check(st)


def swiglu_w4a16_gemv_add_rmsnorm_noalloc(
    gate: torch.Tensor,
    up: torch.Tensor,
    qweight: torch.Tensor,
    scales: torch.Tensor,
    residual: torch.Tensor,
    rms_weight: torch.Tensor,
    eps: float,
    y: torch.Tensor,
    normed: torch.Tensor,
    residual_out: torch.Tensor,
    group: int = 128,
    stream: torch.cuda.Stream | None = None,
) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """swiglu_w4a16_gemv_add_rmsnorm without a scratch buffer, for callers that cannot
    allocate device memory when they call (see fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc in
    include/fd.h): the library uses its own static array, shared by every call, so calls
    must not overlap on the GPU. Every output is passed in (nothing is allocated here
    either); residual_out may be residual (in place)."""
    if gate.dim() == 1:
        gate = gate.unsqueeze(0)
        up = up.unsqueeze(0)
    K = gate.shape[-1]
    N = qweight.shape[0]
    _check_tensor("gate", gate, torch.bfloat16, (1, K))
    _check_tensor("up", up, torch.bfloat16, (1, K))
    _check_tensor("qweight", qweight, torch.int32, (N, K // 8))
    if group <= 0 or K % group != 0:
        raise ValueError(f"K={K} must be a multiple of group={group}")
    _check_tensor("scales", scales, torch.bfloat16, (N, K // group))
    _check_tensor("rms_weight", rms_weight, torch.bfloat16, (N,))
    for name, t in (("residual", residual), ("y", y), ("normed", normed), ("residual_out", residual_out)):
        _check_tensor(name, t, torch.bfloat16)
        if t.numel() != N:
            raise ValueError(f"{name} must hold N={N} elements")
    dev = _device_of(gate, up, qweight, scales, residual, rms_weight, y, normed, residual_out)
    lib = _lib.load()
    with _on_device(dev):
        st = lib.fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc(
            _ptr(gate), _ptr(up), _ptr(qweight), _ptr(scales), _ptr(y), _ptr(residual),
            _ptr(rms_weight), ctypes.c_float(float(eps)), _ptr(normed), _ptr(residual_out),
            int(K), int(N), int(group), _stream_handle(stream, dev),
        )
    _lib.check(st)
    return y, normed, residual_out


def w4a16_gate_up_gemv(
    x: torch.Tensor,
    qweight: torch.Tensor,
    scales: torch.Tensor,
    gate_out: torch.Tensor | None = None,
    up_out: torch.Tensor | None = None,
    group: int = 128,
    stream: torch.cuda.Stream | None = None,
) -> tuple[torch.Tensor, torch.Tensor]:
    """(gate, up) = the gate and up projections of x as one W4A16 GEMV over the stacked
    weights: qweight int32 [2I, K/8] (gate rows, then up rows), scales bf16 [2I, K/group].

    gate[m, j] = bf16(sum_k x[m, k] * W[j, k]), up[m, j] = bf16(sum_k x[m, k] * W[I + j, k]).
    x: bf16 [M, K] (a 1-D tensor is one row); gate_out, up_out: bf16 [M, I] (allocated if
    None). They are the gate and up inputs of ``swiglu_w4a16_gemv``.
    """
    if x.dim() == 1:
        x = x.unsqueeze(0)
    if x.dim() != 2 or qweight.dim() != 2 or scales.dim() != 2:
        raise ValueError("x must be [M, K]; qweight [2I, K/8]; scales [2I, K/group]")
    M, K = x.shape
    N = qweight.shape[0]
    if N % 2 != 0:
        raise ValueError(f"qweight has {N} rows: expected 2I (gate rows, then up rows)")
    inter = N // 2
    _check_tensor("x", x, torch.bfloat16)
    _check_tensor("qweight", qweight, torch.int32, (N, K // 8))
    if group <= 0 or K % group != 0:
        raise ValueError(f"K={K} must be a multiple of group={group}")
    _check_tensor("scales", scales, torch.bfloat16, (N, K // group))
    if gate_out is None:
        gate_out = torch.empty((M, inter), dtype=torch.bfloat16, device=x.device)
    if up_out is None:
        up_out = torch.empty((M, inter), dtype=torch.bfloat16, device=x.device)
    _check_tensor("gate_out", gate_out, torch.bfloat16, (M, inter))
    _check_tensor("up_out", up_out, torch.bfloat16, (M, inter))
    dev = _device_of(x, qweight, scales, gate_out, up_out)
    lib = _lib.load()
    with _on_device(dev):
        st = lib.fd_w4a16_gate_up_gemv(
            _ptr(x), _ptr(qweight), _ptr(scales), _ptr(gate_out), _ptr(up_out),
            int(M), int(K), int(inter), int(group), _stream_handle(stream, dev),
        )
    _lib.check(st)
    return gate_out, up_out


def nvfp4_scaled_mm(
    x: torch.Tensor,
    x_sf: torch.Tensor,
    w: torch.Tensor,
    w_sf: torch.Tensor,
    alpha: torch.Tensor,
    out: torch.Tensor | None = None,
    stream: torch.cuda.Stream | None = None,
) -> torch.Tensor:
    """out[m, n] = bf16(alpha * sum_k X[m, k] * W[n, k]) for NVFP4 operands, the output
    multiplier folded into the GEMM.

    x: uint8 [M, K/2] packed FP4 (element 2p in the low nibble of byte p); x_sf: uint8
    [M, K/16] E4M3 scale codes (one per 16 k); w: uint8 [N, K/2]; w_sf: uint8 [N, K/16];
    alpha: a one-element float32 CUDA tensor (the 0-dim multiplier, read by the kernel);
    out: bf16 [M, N] (allocated if None). See fd_nvfp4_scaled_mm in include/fd.h.
    """
    if x.dim() != 2 or w.dim() != 2 or x_sf.dim() != 2 or w_sf.dim() != 2:
        raise ValueError("x [M, K/2], x_sf [M, K/16], w [N, K/2], w_sf [N, K/16]")
    M, K2 = x.shape
    N = w.shape[0]
    K = 2 * K2
    _check_tensor("x", x, torch.uint8)
    _check_tensor("x_sf", x_sf, torch.uint8, (M, K // 16))
    _check_tensor("w", w, torch.uint8, (N, K2))
    _check_tensor("w_sf", w_sf, torch.uint8, (N, K // 16))
    if not isinstance(alpha, torch.Tensor) or not alpha.is_cuda or alpha.dtype != torch.float32 \
            or alpha.numel() != 1:
        raise ValueError("alpha must be a one-element float32 CUDA tensor")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check_tensor("out", out, torch.bfloat16, (M, N))
    dev = _device_of(x, x_sf, w, w_sf, alpha, out)
    lib = _lib.load()
    with _on_device(dev):
        st = lib.fd_nvfp4_scaled_mm(
            _ptr(x), _ptr(x_sf), _ptr(w), _ptr(w_sf), _ptr(alpha), _ptr(out),
            int(M), int(K), int(N), _stream_handle(stream, dev),
        )
    _lib.check(st)
    return out


def copy(dst: torch.Tensor, src: torch.Tensor, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """dst <- src (same number of bytes, contiguous, 16-byte aligned) with one kernel:
    either side may be a CUDA tensor or a pinned host tensor (read or written by the GPU
    over NVLink-C2C). Falls back to one cudaMemcpyAsync for memory a kernel cannot reach."""
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy: dst and src must be contiguous")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("copy: dst and src differ in size")
    for name, t in (("dst", dst), ("src", src)):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"copy: {name} must be a CUDA tensor or pinned host memory")
    dev = _device_of(dst, src)
    lib = _lib.load()
    with _on_device(dev):
        _lib.check(lib.fd_copy(_ptr(dst), _ptr(src), nbytes, _stream_handle(stream, dev)))
    return dst


def copy_rows(dst: torch.Tensor, src: torch.Tensor,
              stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """dst <- src for two 2-D tensors of the same shape and dtype whose rows are contiguous
    (unit inner stride) but may lie at any row stride, with one kernel (fd_copy_rows): either
    side may be a CUDA tensor or host memory (pinned memory is read or written by the GPU
    over NVLink-C2C; other host memory goes through one cudaMemcpy2DAsync)."""
    if dst.dim() != 2 or src.dim() != 2 or dst.shape != src.shape or dst.dtype != src.dtype:
        raise ValueError("copy_rows: dst and src must be 2-D tensors of the same shape and dtype")
    if dst.stride(1) != 1 or src.stride(1) != 1:
        raise ValueError("copy_rows: rows must be contiguous")
    es = dst.element_size()
    rows, row_bytes = dst.shape[0], dst.shape[1] * es
    if not (dst.is_cuda or src.is_cuda):
        raise ValueError("copy_rows: one side must be a CUDA tensor")
    dev = _device_of(dst, src)
    lib = _lib.load()
    with _on_device(dev):
        _lib.check(lib.fd_copy_rows(_ptr(dst), dst.stride(0) * es, _ptr(src), src.stride(0) * es,
                                    row_bytes, rows, _stream_handle(stream, dev)))
    return dst


def add_rmsnorm(
    x: torch.Tensor,
    residual: torch.Tensor,
    weight: torch.Tensor,
    eps: float,
    out: torch.Tensor | None = None,
    residual_out: torch.Tensor | None = None,
    stream: torch.cuda.Stream | None = None,
) -> tuple[torch.Tensor, torch.Tensor]:
    """(out, residual_out) with residual_out = bf16(x + residual) and
    out = bf16(bf16(h * rstd) * weight), rstd = 1/sqrt(mean(h^2) + eps) per row.

    x, residual: bf16 [rows, hidden] (a 1-D tensor is one row); weight: bf16 [hidden].
    out may be x and residual_out may be residual (in place).
    """
    squeeze = x.dim() == 1
    if squeeze:
        x = x.unsqueeze(0)
        residual = residual.unsqueeze(0)
    if x.dim() != 2:
        raise ValueError("x must be [rows, hidden]")
    rows, hidden = x.shape
    _check_tensor("x", x, torch.bfloat16)
    _check_tensor("residual", residual, torch.bfloat16, (rows, hidden))
    _check_tensor("weight", weight, torch.bfloat16, (hidden,))
    if out is None:
        out = torch.empty_like(x)
    elif squeeze and out.dim() == 1:
        out = out.unsqueeze(0)
    if residual_out is None:
        residual_out = torch.empty_like(x)
    elif squeeze and residual_out.dim() == 1:
        residual_out = residual_out.unsqueeze(0)
    _check_tensor("out", out, torch.bfloat16, (rows, hidden))
    _check_tensor("residual_out", residual_out, torch.bfloat16, (rows, hidden))
    dev = _device_of(x, residual, weight, out, residual_out)
    lib = _lib.load()
    with _on_device(dev):
        st = lib.fd_add_rmsnorm(
            _ptr(x), _ptr(residual), _ptr(weight), ctypes.c_float(float(eps)), _ptr(out),
            _ptr(residual_out), int(rows), int(hidden), _stream_handle(stream, dev),
        )
    _lib.check(st)
    if squeeze:
        return out.squeeze(0), residual_out.squeeze(0)
    return out, residual_out


def w4_dequant_debug(
    qweight: torch.Tensor,
    scales: torch.Tensor,
    group: int = 128,
    out: torch.Tensor | None = None,
    stream: torch.cuda.Stream | None = None,
) -> torch.Tensor:
    """fp32 [N, K] dequantised weights from the GEMV prologue's unpack (test support)."""
    _check_tensor("qweight", qweight, torch.int32)
    if qweight.dim() != 2:
        raise ValueError("qweight must be [N, K/8]")
    N, K8 = qweight.shape
    K = K8 * 8
    if group <= 0 or K % group != 0:
        raise ValueError(f"K={K} must be a multiple of group={group}")
    _check_tensor("scales", scales, torch.bfloat16, (N, K // group))
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=qweight.device)
    _check_tensor("out", out, torch.float32, (N, K))
    dev = _device_of(qweight, scales, out)
    lib = _lib.load()
    with _on_device(dev):
        st = lib.fd_w4_dequant_debug(
            _ptr(qweight), _ptr(scales), _ptr(out), int(K), int(N), int(group),
            _stream_handle(stream, dev),
        )
    _lib.check(st)
    return out


def decode_mlp_step(
    x: torch.Tensor,
    residual: torch.Tensor,
    layers: list[dict],
    eps: float,
    group: int = 128,
    normed: list[torch.Tensor] | None = None,
    y: list[torch.Tensor] | None = None,
    stream: torch.cuda.Stream | None = None,
    scratch: torch.Tensor | None = None,
) -> tuple[torch.Tensor, torch.Tensor]:
    """One decode step over L layers of ("09 - Operator fusion", "The fusion boundary
    problem"): (normed_l, residual) = add_rmsnorm(x_l, residual); y_l = down(g_l, u_l);
    x_{l+1} = y_l. Two kernel launches per layer, in stream order; ``residual`` is
    updated in place. ``layers`` holds per-layer device tensors ``rms_weight``, ``gate``,
    ``up``, ``qweight``, ``scales``. ``normed``/``y`` are optional preallocated outputs
    (one [1, hidden] tensor per layer) so the step allocates nothing and can be captured
    in a CUDA graph. With ``scratch`` (fold_scratch()) each layer's add-RMSNorm after the
    first is folded into the previous layer's GEMV (swiglu_w4a16_gemv_add_rmsnorm): L + 1
    launches instead of 2L, the same dataflow. Returns (x_L, residual).
    """
    if scratch is not None:
        n_out = normed[0] if normed is not None else None
        n_out, _ = add_rmsnorm(x, residual, layers[0]["rms_weight"], eps, out=n_out,
                               residual_out=residual, stream=stream)
        cur = x
        for i, layer in enumerate(layers):
            y_out = y[i] if y is not None else None
            if i + 1 < len(layers):
                nxt = normed[i + 1] if normed is not None else None
                cur, _, _ = swiglu_w4a16_gemv_add_rmsnorm(
                    layer["gate"], layer["up"], layer["qweight"], layer["scales"], residual,
                    layers[i + 1]["rms_weight"], eps, scratch, y=y_out, normed=nxt,
                    residual_out=residual, group=group, stream=stream)
            else:
                cur = swiglu_w4a16_gemv(layer["gate"], layer["up"], layer["qweight"],
                                        layer["scales"], out=y_out, group=group, stream=stream)
        return cur, residual
    cur = x
    for i, layer in enumerate(layers):
        n_out = normed[i] if normed is not None else None
        n_out, _ = add_rmsnorm(cur, residual, layer["rms_weight"], eps, out=n_out,
                               residual_out=residual, stream=stream)
        y_out = y[i] if y is not None else None
        cur = swiglu_w4a16_gemv(layer["gate"], layer["up"], layer["qweight"], layer["scales"],
                                out=y_out, group=group, stream=stream)
    return cur, residual
