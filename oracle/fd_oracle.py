"""Plain, slow, unfused CPU oracle for the SwiGLU-prologue W4A16 GEMV and fused
residual-add + RMSNorm.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline legs of ``bench.py``, never by the product path. It shares no code,
constants or helpers with the CUDA library; it reads the same input bytes.

Every floating-point step is done in float64 unless a page fixes a narrower
precision (the residual add is fp32-then-bf16, as the pages' kernel does). Each
function cites the passage it follows, by page title and section:

* [FIX]   "PyTorch Community Proposes Fusion Fix as Large Intermediate Buffers May Slow
          Single-Token Decoding in Quantized LLMs" - "Reproduction and analysis",
          "Fix proposal".
* [SGL13] "Chapter 13 - torch.compile" (learning-sglang) - "The two halves of one tool,
          and what each is worth".
* [FUSE]  "09 - Operator fusion" (inference engineering, part IV) - section 5 "Technical
          explanation": "The taxonomy of fusions", "The fusion boundary problem".
* [KFM]   "Kernel Fusion, torch.compile and CUDA Graphs, Measured" - "Step 1: why
          elementwise kernels are memory-bound", "Step 2: fusing them by hand in
          Triton", "Step 3: what torch.compile generates".
* [NVFP4] "PyTorch folds NVFP4 output scaling into NVGEMM candidates for decode
          workloads" - body (eligibility: packed FP4 operands, E4M3 1x16 block scales, a
          zero-dimensional fp32 output multiplier; the ATen candidate that runs the scaled
          matmul and the multiplication separately).

Where the pages are silent the plainest reading is taken (symmetric two's-complement
int4, eight nibbles per 32-bit word along K, nibble j of word p holding k = 8p + j,
bf16 scales [N, K/group] with w = q * s; for NVFP4, E2M1 elements packed two per byte
with the even k in the low nibble, E4M3 scales [rows, K/16] row-major, and a bf16
output). Every function here is pinned by
``tests/test_oracle_pins.py`` to something other than itself; none is "parity
unpinned".
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_to_f32",
    "f32_to_bf16_rne",
    "silu",
    "swiglu_activation",
    "unpack_int4",
    "dequant_w4",
    "contract",
    "swiglu_w4a16_gemv",
    "swiglu_w4a16_gemv_residual",
    "w4a16_gemv",
    "gate_up_gemv",
    "add_rmsnorm",
    "decode_mlp_step",
    "unpack_fp4",
    "e2m1_to_f64",
    "e4m3_to_f64",
    "nvfp4_dequant",
    "nvfp4_scaled_mm",
    "unfused_product_bytes",
    "eager_add_rmsnorm_kernels",
    "eager_add_rmsnorm_bytes_per_elem",
    "eager_swiglu_bytes_per_elem",
    "fused_swiglu_bytes_per_elem",
]


# --------------------------------------------------------------------------------------
# bfloat16 <-> float32 (bit level)
# --------------------------------------------------------------------------------------

def bf16_to_f32(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32. Exact: a bf16 value is the top
    half of the float32 with the same value."""
    b = np.asarray(bits).astype(np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_rne(x) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even), returned as
    uint16 bit patterns. NaN stays NaN (quiet bit set); +-inf stays inf.

    [KFM] Step 2: every bf16 value the pages' kernel stores is a float32 rounded to
    bf16 (`.to(tl.bfloat16)`), which rounds to nearest-even.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    upper = u >> np.uint64(16)
    lower = u & np.uint64(0xFFFF)
    half = np.uint64(0x8000)
    round_up = (lower > half) | ((lower == half) & ((upper & np.uint64(1)) == np.uint64(1)))
    out = upper + round_up.astype(np.uint64)
    is_nan = np.isnan(f)
    out = np.where(is_nan, upper | np.uint64(0x0040), out)
    return out.astype(np.uint16)


# --------------------------------------------------------------------------------------
# SwiGLU prologue
# --------------------------------------------------------------------------------------

def silu(x) -> np.ndarray:
    """silu(x) = x * sigmoid(x) = x / (1 + exp(-x)), in float64.

    [KFM] Step 1: SwiGLU's activation "computes g / (1 + exp(-g)) * u".
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def swiglu_activation(gate_bits, up_bits) -> np.ndarray:
    """a = silu(g) * u in float64 from bf16 gate and up (uint16 bits), unrounded.

    [KFM] Step 1 (silu(g) * u); [FUSE] "The fusion boundary problem" (act = silu(gate) *
    up feeding the down projection). The fused kernel never stores `a`; the oracle keeps
    it in float64.
    """
    g = bf16_to_f32(gate_bits).astype(np.float64)
    u = bf16_to_f32(up_bits).astype(np.float64)
    return silu(g) * u


# --------------------------------------------------------------------------------------
# int4 weights
# --------------------------------------------------------------------------------------

def unpack_int4(qweight) -> np.ndarray:
    """Unpack int32 words [N, K/8] into int8 q [N, K] with q in [-8, 7].

    Nibble j (bits 4j..4j+3) of word p in row n is q[n, 8p + j], a 4-bit two's
    complement integer. [FUSE] taxonomy item 4 ("GEMM prologue fusion": the INT4 form is
    what crosses HBM); the bit layout is this library's reading, the pages give none.
    """
    w = np.ascontiguousarray(qweight).view(np.uint32)
    n_rows, n_words = w.shape
    q = np.empty((n_rows, n_words * 8), dtype=np.int8)
    for j in range(8):
        nib = ((w >> np.uint32(4 * j)) & np.uint32(0xF)).astype(np.int16)
        nib = np.where(nib >= 8, nib - 16, nib)
        q[:, j::8] = nib.astype(np.int8)
    return q


def dequant_w4(qweight, scale_bits, group: int) -> np.ndarray:
    """Dequantised weights W[n, k] = q[n, k] * s[n, k // group] as float32 [N, K].

    [FUSE] taxonomy item 4 (dequantize weights -> matmul). The product of a 4-bit integer
    and a bf16 scale has at most 12 significant bits, so the float32 result is exact; it
    is computed in float64 and then narrowed.
    """
    q = unpack_int4(qweight).astype(np.float64)
    s = bf16_to_f32(scale_bits).astype(np.float64)
    n_rows, k = q.shape
    if k % group != 0 or s.shape != (n_rows, k // group):
        raise ValueError("scales must be [N, K/group]")
    w = q * np.repeat(s, group, axis=1)
    return w.astype(np.float32)


def contract(a, w) -> np.ndarray:
    """y[m, n] = sum_k a[m, k] * w[n, k] in float64, one output at a time.

    The matrix product of an nn.Linear layer (out = x @ W^T, [FIX] "Reproduction and
    analysis") written as the plain loop over outputs (m, n); only the innermost sum over
    k is one vectorised float64 dot product. No blocking or reordering beyond that.
    """
    a = np.asarray(a, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    if a.ndim != 2 or w.ndim != 2 or a.shape[1] != w.shape[1]:
        raise ValueError("contract: a is [M, K] and w is [N, K]")
    y = np.empty((a.shape[0], w.shape[0]), dtype=np.float64)
    for m in range(a.shape[0]):
        for n in range(w.shape[0]):
            y[m, n] = np.dot(a[m], w[n])
    return y


def swiglu_w4a16_gemv(gate_bits, up_bits, qweight, scale_bits, group: int) -> np.ndarray:
    """y[m, n] = sum_k a[m, k] * W[n, k] with a = silu(g) * u, as float64 [M, N].

    Unfused on purpose: the activation, the dequantised weight matrix and the product
    are each formed in full before the next step. [FIX] "Reproduction and analysis"
    (single-row matmul y = x @ W with a SwiGLU pre-operation and int4 weights);
    [FUSE] "The fusion boundary problem" (out = act @ W_down). The contraction is the
    plain per-output sum of ``contract``.
    """
    a = swiglu_activation(gate_bits, up_bits)
    if a.ndim == 1:
        a = a[None, :]
    w = dequant_w4(qweight, scale_bits, group).astype(np.float64)
    if a.shape[1] != w.shape[1]:
        raise ValueError("gate/up K does not match the weights")
    return contract(a, w)


def swiglu_w4a16_gemv_residual(gate_bits, up_bits, qweight, scale_bits, residual_bits,
                               group: int):
    """The down projection with a residual-add epilogue: new_residual = x + out.

    [FUSE] "The fusion boundary problem": kernel 3 of a fused layer is GEMM(act, W_down)
    with a residual-add epilogue writing new_residual = x + out, x being the pre-norm
    residual stream (the first output of kernel 1, add_rmsnorm). [FUSE] "The taxonomy of
    fusions", item 3: the elementwise op is applied to the accumulator before the output
    is written.

    Returns ``(ref, eager_bits)``:
      * ``ref``        float64 [M, N], f32(residual) + y with y from swiglu_w4a16_gemv,
                       nothing rounded;
      * ``eager_bits`` uint16, the unfused chain's two roundings: out = bf16(y) is stored,
                       then a separate add kernel stores bf16(f32(x) + f32(out)).
    """
    y = swiglu_w4a16_gemv(gate_bits, up_bits, qweight, scale_bits, group)
    r = bf16_to_f32(np.asarray(residual_bits, dtype=np.uint16)).astype(np.float64)
    r = r.reshape(y.shape)
    ref = r + y
    out_bits = f32_to_bf16_rne(y.astype(np.float32))
    s32 = bf16_to_f32(out_bits) + r.astype(np.float32)  # float32 add, IEEE RNE
    eager_bits = f32_to_bf16_rne(s32)
    return ref, eager_bits


def w4a16_gemv(x_bits, qweight, scale_bits, group: int) -> np.ndarray:
    """y[m, n] = sum_k x[m, k] * W[n, k] as float64 [M, N], x a plain bf16 activation.

    [FUSE] "The taxonomy of fusions", item 4 (dequantise the int4 weights, then the
    matmul) with no pre-operation on the activation. Unfused: W is formed in full, then
    the plain per-output sum of ``contract``.
    """
    x = bf16_to_f32(np.asarray(x_bits, dtype=np.uint16)).astype(np.float64)
    if x.ndim == 1:
        x = x[None, :]
    w = dequant_w4(qweight, scale_bits, group).astype(np.float64)
    if x.shape[1] != w.shape[1]:
        raise ValueError("x K does not match the weights")
    return contract(x, w)


def gate_up_gemv(x_bits, qweight, scale_bits, group: int):
    """(g, u), each float64 [M, I]: the gate and up projections of x as one GEMV.

    [FUSE] "The taxonomy of fusions", item 5 (horizontal fusion: gate_proj and up_proj,
    two matmuls on the same input, become one gate_up_proj) and "The fusion boundary
    problem" (gate, up = h @ W_gate_up). The stacked weight holds the gate projection's I
    rows, then the up projection's I rows.
    """
    y = w4a16_gemv(x_bits, qweight, scale_bits, group)
    if y.shape[1] % 2 != 0:
        raise ValueError("the stacked weight must have 2I rows")
    inter = y.shape[1] // 2
    return y[:, :inter], y[:, inter:]


# --------------------------------------------------------------------------------------
# Residual add + RMSNorm
# --------------------------------------------------------------------------------------

def add_rmsnorm(x_bits, residual_bits, weight_bits, eps: float):
    """Residual add followed by RMSNorm over the last axis.

    Follows the order of [KFM] Step 2's hand-written kernel:
      h = bf16(f32(x) + f32(r))              (float32 add, rounded to bf16; stored)
      rstd = 1 / sqrt(mean_j f32(h_j)^2 + eps)   (here in float64)
      y = h * rstd * w

    Returns ``(h_bits, y_ref, y_eager_bits)``:
      * ``h_bits``      uint16, the new residual (bit-exact target);
      * ``y_ref``       float64, h * rstd * w with no rounding;
      * ``y_eager_bits`` uint16, bf16(bf16(h * rstd) * w), the page's two roundings
                        (normalised value rounded to bf16, then scaled by w).
    The mean divides by the row length ([KFM] Step 3 divides by 4096.0 for hidden 4096).
    """
    x = bf16_to_f32(x_bits)
    r = bf16_to_f32(residual_bits)
    h_bits = f32_to_bf16_rne(x + r)  # numpy float32 + float32 -> float32 (IEEE RNE)
    h = bf16_to_f32(h_bits).astype(np.float64)
    w = bf16_to_f32(weight_bits).astype(np.float64)
    ms = np.mean(h * h, axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(ms + float(eps))
    normed = h * rstd
    y_ref = normed * w
    t_bits = f32_to_bf16_rne(normed.astype(np.float32))
    prod = bf16_to_f32(t_bits).astype(np.float64) * w  # exact: 8-bit x 8-bit significands
    y_eager_bits = f32_to_bf16_rne(prod.astype(np.float32))
    return h_bits, y_ref, y_eager_bits


# --------------------------------------------------------------------------------------
# The decode MLP step (add-RMSNorm, then the SwiGLU-prologue down projection)
# --------------------------------------------------------------------------------------

def decode_mlp_step(x_bits, residual_bits, layers, eps: float, group: int):
    """Run L layers of: (normed, residual) = add_rmsnorm(x, residual); y = down(g, u);
    x_next = bf16(y).

    ``layers`` is a sequence of dicts with keys ``rms_weight``, ``gate``, ``up``,
    ``qweight``, ``scales`` (bf16 bits / int32 words). [FUSE] "The fusion boundary
    problem": kernel 1 is add_rmsnorm(residual, attn_out) -> (x, h) with two outputs and
    the down projection's output joins the residual stream at the next add. The gate/up
    projection between them is not part of this path, so each layer's g and u are given
    inputs. The value handed to the next layer is the bf16-rounded GEMV output, as the
    bf16 layer output of a model would be.

    Returns per-layer lists of (h_bits, y_norm_ref, y_norm_eager_bits, y_gemv_ref) and
    the final (x_bits, residual_bits).
    """
    x = np.asarray(x_bits, dtype=np.uint16)
    res = np.asarray(residual_bits, dtype=np.uint16)
    record = []
    for layer in layers:
        h_bits, y_norm, y_norm_eager = add_rmsnorm(x, res, layer["rms_weight"], eps)
        y = swiglu_w4a16_gemv(layer["gate"], layer["up"], layer["qweight"], layer["scales"], group)
        record.append((h_bits, y_norm, y_norm_eager, y))
        res = h_bits
        x = f32_to_bf16_rne(y.astype(np.float32)).reshape(x.shape)
    return record, x, res


# --------------------------------------------------------------------------------------
# NVFP4 scaled matmul with the output scale folded in
# --------------------------------------------------------------------------------------

def unpack_fp4(packed) -> np.ndarray:
    """Split packed FP4 bytes [R, K/2] into 4-bit codes [R, K] (uint8, 0..15).

    [NVFP4]: the operands are "packed FP4", two 4-bit elements per byte. The page gives
    no order; the reading here is element 2p in the low nibble (bits 0..3) of byte p
    and element 2p + 1 in the high nibble.
    """
    b = np.ascontiguousarray(packed).astype(np.uint8)
    if b.ndim != 2:
        raise ValueError("packed FP4 operands are [rows, K/2] bytes")
    codes = np.empty((b.shape[0], b.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = b & np.uint8(0x0F)
    codes[:, 1::2] = b >> np.uint8(4)
    return codes


def e2m1_to_f64(codes) -> np.ndarray:
    """Value of 4-bit E2M1 codes: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.

    An exponent field of 0 is subnormal, m * 2^-1; otherwise (1 + m/2) * 2^(e - 1). The
    format has no infinity or NaN, so every code is finite (largest magnitude 6). This
    is the element type of NVFP4 ([NVFP4] "packed FP4"); the page does not spell the
    encoding out, and the reading is the standard FP4 E2M1 definition.
    """
    c = np.asarray(codes).astype(np.int64)
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return sign * mag


def e4m3_to_f64(codes) -> np.ndarray:
    """Value of 8-bit E4M3 codes: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits
    2..0. An exponent field of 0 is subnormal, (m/8) * 2^-6. S.1111.111 is NaN and there
    is no infinity, so S.1111.110 = 448 is the largest magnitude.

    [NVFP4]: the block scales are "E4M3 1x16" scales.
    """
    c = np.asarray(codes).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def nvfp4_dequant(packed, sf_codes) -> np.ndarray:
    """Dequantised NVFP4 operand X[r, k] = e2m1(x[r, k]) * e4m3(sf[r, k // 16]), float64
    [R, K].

    [NVFP4]: one E4M3 scale per 1x16 block, i.e. per 16 consecutive elements of a row
    along K. A 2-bit significand times a 4-bit one is exact in float64.
    """
    x = e2m1_to_f64(unpack_fp4(packed))
    sf = e4m3_to_f64(np.asarray(sf_codes))
    rows, k = x.shape
    if k % 16 != 0 or sf.shape != (rows, k // 16):
        raise ValueError("block scales must be [rows, K/16]")
    return x * np.repeat(sf, 16, axis=1)


def nvfp4_scaled_mm(x_packed, x_sf, w_packed, w_sf, alpha):
    """out[m, n] = alpha * sum_k X[m, k] * W[n, k] with X, W the dequantised NVFP4
    activations [M, K] and weights [N, K] (an nn.Linear's x @ W^T).

    [NVFP4] body: the scaled matmul of two packed-FP4 operands with E4M3 1x16 block
    scales, and the zero-dimensional fp32 output multiplier alpha that the fold applies
    inside the GEMM instead of in a separate multiplication. Unfused here: both operands
    are dequantised in full, then the plain per-output sum of ``contract``, then the
    multiplication.

    Returns ``(ref, eager_bits)``:
      * ``ref``        float64 [M, N], alpha * the sum, nothing rounded;
      * ``eager_bits`` uint16, the unfolded sequence the page's ATen candidate keeps: the
                       scaled matmul stores bf16(sum), then a separate multiplication by
                       alpha computes in float32 and stores bf16 again.
    """
    x = nvfp4_dequant(x_packed, x_sf)
    w = nvfp4_dequant(w_packed, w_sf)
    if x.shape[1] != w.shape[1]:
        raise ValueError("activation K does not match the weights")
    a32 = np.float32(alpha)
    acc = contract(x, w)
    ref = float(a32) * acc
    mm_bits = f32_to_bf16_rne(acc.astype(np.float32))
    eager_bits = f32_to_bf16_rne(bf16_to_f32(mm_bits) * a32)  # float32 multiply, IEEE RNE
    return ref, eager_bits


# --------------------------------------------------------------------------------------
# Byte models of the unfused forms the fused kernels replace
# --------------------------------------------------------------------------------------

def unfused_product_bytes(m: int, k: int, n: int, elem_bytes: int = 4) -> int:
    """Size of the (M, K, N) broadcast product an M=1 matmul decomposed into a
    multiply and a sum materialises. [FIX] "Reproduction and analysis": K=9216, N=2560
    writes and reads back about 94 MB."""
    return m * k * n * elem_bytes


def eager_add_rmsnorm_kernels():
    """The eager residual add + Qwen2-style RMSNorm chain, one entry per kernel:
    (name, bytes read per element, bytes written per element). [KFM] "Why it matters"
    and Step 1 (9 kernels, 42 bytes per element on bf16; the page's per-element table
    did not survive, so the split is reconstructed from the listed operations: add,
    cast to fp32, square, mean, add eps, rsqrt, multiply, cast to bf16, multiply by w;
    the eps add and rsqrt touch one value per row and the mean writes one per row)."""
    return [
        ("add", 4, 2),
        ("to_fp32", 2, 4),
        ("pow", 4, 4),
        ("mean", 4, 0),
        ("add_eps", 0, 0),
        ("rsqrt", 0, 0),
        ("mul_rstd", 4, 4),
        ("to_bf16", 4, 2),
        ("mul_weight", 2, 2),
    ]


def eager_add_rmsnorm_bytes_per_elem() -> int:
    return sum(r + w for _, r, w in eager_add_rmsnorm_kernels())


def eager_swiglu_bytes_per_elem() -> int:
    """silu then multiply as two bf16 kernels: read g, write s; read s and u, write a.
    [KFM] Step 1: 10 bytes per element."""
    return (2 + 2) + (2 + 2 + 2)


def fused_swiglu_bytes_per_elem() -> int:
    """One kernel: read g and u, write a. [KFM] Step 1: 6 bytes per element."""
    return 2 + 2 + 2
