"""Algorithmic (ideal) HBM bytes of one call of each fused kernel.

The roofline numerator: every input read once and every output written once, nothing
else ("Kernel Fusion, torch.compile and CUDA Graphs, Measured", "Measured": effective
GB/s divides the fused kernel's bytes by the time, so it measures the job, not the
traffic).
"""

from __future__ import annotations


def gemv_bytes(M: int, K: int, N: int, group: int) -> int:
    """int4 weights + bf16 scales + bf16 gate and up + bf16 output."""
    return N * K // 2 + N * (K // group) * 2 + 2 * M * K * 2 + M * N * 2


def gate_up_bytes(M: int, K: int, inter: int, group: int) -> int:
    """The stacked [2I, K] int4 weights and their bf16 scales, x once, g and u written."""
    N = 2 * inter
    return N * K // 2 + N * (K // group) * 2 + M * K * 2 + M * N * 2


def gemv_flops(M: int, K: int, N: int) -> int:
    return 2 * M * K * N


def add_rmsnorm_bytes(rows: int, hidden: int) -> int:
    """x and residual read, out and residual_out written (2 bytes each), weight once."""
    return 8 * rows * hidden + 2 * hidden


def decode_step_bytes(layers: int, hidden: int, inter: int, group: int) -> int:
    return layers * (add_rmsnorm_bytes(1, hidden) + gemv_bytes(1, inter, hidden, group))


def nvfp4_bytes(M: int, K: int, N: int) -> int:
    """Packed FP4 weights and activations (K/2 bytes per row), their E4M3 scales (K/16
    bytes per row) and the bf16 output; alpha's 4 bytes are not counted."""
    return (N + M) * (K // 2 + K // 16) + M * N * 2


def nvfp4_flops(M: int, K: int, N: int) -> int:
    return 2 * M * K * N
