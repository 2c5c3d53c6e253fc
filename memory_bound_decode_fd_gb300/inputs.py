"""Seeded synthetic inputs for the fused decode kernels (shared by tests and bench).

Holds random draws only, none of the kernels' arithmetic. Each generator draws from
``numpy.random.default_rng(seed)`` (PCG64) in a fixed order and returns host arrays:
bf16 tensors as uint16 bit patterns (normal draws are made in float64, narrowed to
float32, and rounded to bf16 by ``torch.Tensor.to(torch.bfloat16)``), packed int4
weights as int32 words. Drawing each 32-bit word uniformly makes every nibble an
independent uniform integer in [-8, 7] (two's complement), which is the weight
distribution of the workloads; scales are uniform in [0.005, 0.02].

Workloads (name: sizes, seed):
  gemv_small     GEMV M=1 K=1024 N=256 group 128, seed 0
  rmsnorm_big    add-RMSNorm rows=8192 hidden=4096 eps=1e-6, seed 1
  gemv_94mb      GEMV M=1 K=9216 N=2560 group 128 (its fp32 (1,K,N) product is 94 MB), seed 2
  decode_step    32 x [add-RMSNorm 1x4096 eps=1e-5 + GEMV K=14336 N=4096], seed 3
  batched_m64    GEMV M=64 K=14336 N=4096 + add-RMSNorm 64x4096 eps=1e-5, seed 4
  gemv_residual  the decode-step GEMV with the residual-add epilogue, seed 3
  gate_up        gate/up GEMV M=1 K=4096 I=14336 (28672 stacked rows), seed 3
  nvfp4_qkv      NVFP4 scaled matmul M=64 K=4096 N=6144 (``nvfp4_inputs``), seed 5

NVFP4 operands (``nvfp4_inputs``; M=64 K=4096 N=6144 is a Llama-3.1-8B QKV projection at
batch 64, seed 5) are drawn as codes: packed FP4 bytes uniform (every nibble one of the
16 E2M1 codes with equal odds), E4M3 block-scale codes with sign 0, exponent field
uniform in 3..9 and mantissa uniform in 0..7 (scales from 2^-4 to 7.5), and the fp32
output multiplier uniform in [0.5, 2).
"""

from __future__ import annotations

import numpy as np
import torch


def to_bf16_bits(x) -> np.ndarray:
    """float array -> bf16 bit patterns (uint16), rounded by torch (nearest-even)."""
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=np.float32)))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, mean: float = 0.0, std: float = 1.0):
    return to_bf16_bits(rng.normal(mean, std, size=shape))


def int4_words(rng: np.random.Generator, n: int, k: int) -> np.ndarray:
    """Packed weights [n, k/8] int32 with i.i.d. uniform nibbles (q uniform in [-8, 7])."""
    return rng.integers(0, 2**32, size=(n, k // 8), dtype=np.uint32).view(np.int32)


def scales_bf16(rng: np.random.Generator, n: int, k: int, group: int):
    return to_bf16_bits(rng.uniform(0.005, 0.02, size=(n, k // group)))


def gemv_inputs(M: int, K: int, N: int, group: int = 128, seed: int = 0, rng=None) -> dict:
    """Draw order: gate, up, qweight, scales."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    return {
        "gate": normal_bf16(rng, (M, K)),
        "up": normal_bf16(rng, (M, K)),
        "qweight": int4_words(rng, N, K),
        "scales": scales_bf16(rng, N, K, group),
        "M": M, "K": K, "N": N, "group": group,
    }


def rmsnorm_inputs(rows: int, hidden: int, seed: int = 1, rng=None) -> dict:
    """Draw order: x, residual, weight (weight ~ N(1, 0.1))."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    return {
        "x": normal_bf16(rng, (rows, hidden)),
        "residual": normal_bf16(rng, (rows, hidden)),
        "weight": normal_bf16(rng, (hidden,), 1.0, 0.1),
        "rows": rows, "hidden": hidden,
    }


def decode_step_inputs(layers: int = 32, hidden: int = 4096, inter: int = 14336,
                       group: int = 128, seed: int = 3) -> dict:
    """Draw order: x0, residual0, then per layer: rms_weight, gate, up, qweight, scales."""
    rng = np.random.default_rng(seed)
    x0 = normal_bf16(rng, (1, hidden))
    res0 = normal_bf16(rng, (1, hidden))
    per_layer = []
    for _ in range(layers):
        per_layer.append({
            "rms_weight": normal_bf16(rng, (hidden,), 1.0, 0.1),
            "gate": normal_bf16(rng, (1, inter)),
            "up": normal_bf16(rng, (1, inter)),
            "qweight": int4_words(rng, hidden, inter),
            "scales": scales_bf16(rng, hidden, inter, group),
        })
    return {"x": x0, "residual": res0, "layers": per_layer, "hidden": hidden,
            "inter": inter, "group": group}


def batched_inputs(M: int = 64, K: int = 14336, N: int = 4096, group: int = 128,
                   seed: int = 4) -> dict:
    """GEMV draws (gate, up, qweight, scales) then RMSNorm draws (x, residual, weight)."""
    rng = np.random.default_rng(seed)
    g = gemv_inputs(M, K, N, group, rng=rng)
    r = rmsnorm_inputs(M, N, rng=rng)
    return {"gemv": g, "rmsnorm": r}


def fp4_bytes(rng: np.random.Generator, rows: int, k: int) -> np.ndarray:
    """Packed FP4 operand [rows, k/2] uint8, every nibble i.i.d. uniform over the 16 codes."""
    return rng.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)


def e4m3_scale_codes(rng: np.random.Generator, rows: int, k: int) -> np.ndarray:
    """Block-scale codes [rows, k/16] uint8: sign 0, exponent field 3..9, mantissa 0..7."""
    e = rng.integers(3, 10, size=(rows, k // 16), dtype=np.uint8)
    m = rng.integers(0, 8, size=(rows, k // 16), dtype=np.uint8)
    return (e << np.uint8(3)) | m


def nvfp4_inputs(M: int = 64, K: int = 4096, N: int = 6144, seed: int = 5, rng=None) -> dict:
    """Draw order: x, x_sf, w, w_sf, alpha."""
    rng = rng if rng is not None else np.random.default_rng(seed)
    return {
        "x": fp4_bytes(rng, M, K),
        "x_sf": e4m3_scale_codes(rng, M, K),
        "w": fp4_bytes(rng, N, K),
        "w_sf": e4m3_scale_codes(rng, N, K),
        "alpha": np.float32(rng.uniform(0.5, 2.0)),
        "M": M, "K": K, "N": N,
    }


WORKLOADS = {
    "gemv_small": dict(kind="gemv", M=1, K=1024, N=256, group=128, seed=0),
    "rmsnorm_big": dict(kind="rmsnorm", rows=8192, hidden=4096, eps=1e-6, seed=1),
    "gemv_94mb": dict(kind="gemv", M=1, K=9216, N=2560, group=128, seed=2),
    "decode_step": dict(kind="decode", layers=32, hidden=4096, inter=14336, group=128,
                        eps=1e-5, seed=3),
    "batched_m64": dict(kind="batched", M=64, K=14336, N=4096, group=128, eps=1e-5, seed=4),
    # the decode-step down projection with the residual-add epilogue (new_residual = x + out)
    "gemv_residual": dict(kind="gemv_residual", M=1, K=14336, N=4096, group=128, seed=3),
    # the gate and up projections of the same MLP as one horizontally fused W4A16 GEMV
    "gate_up": dict(kind="gate_up", M=1, K=4096, I=14336, group=128, seed=3),
    # the NVFP4 QKV projection at batch 64 (Llama-3.1-8B: 32 query + 8 key/value heads of 128)
    "nvfp4_qkv": dict(kind="nvfp4", M=64, K=4096, N=6144, seed=5),
}
