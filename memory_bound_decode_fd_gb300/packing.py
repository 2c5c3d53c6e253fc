"""Host-side int4 weight packing into the layout fd_swiglu_w4a16_gemv reads.

q [N, K] int8 in [-8, 7] -> int32 [N, K/8]: nibble j (bits 4j..4j+3) of word p in row n
holds q[n, 8p + j] as a 4-bit two's complement integer ("09 - Operator fusion", section
5, taxonomy item 4: only this packed form crosses HBM).
"""

from __future__ import annotations

import numpy as np


def pack_int4(q) -> np.ndarray:
    """Pack int8 q [N, K] (values in [-8, 7], K % 8 == 0) into int32 [N, K/8]."""
    q = np.asarray(q)
    if q.ndim != 2 or q.shape[1] % 8 != 0:
        raise ValueError("q must be [N, K] with K % 8 == 0")
    if q.size and (q.min() < -8 or q.max() > 7):
        raise ValueError("q must lie in [-8, 7]")
    nib = (q.astype(np.int64) & 0xF).astype(np.uint32).reshape(q.shape[0], -1, 8)
    words = np.zeros(nib.shape[:2], dtype=np.uint32)
    for j in range(8):
        words |= nib[:, :, j] << np.uint32(4 * j)
    return words.view(np.int32)
