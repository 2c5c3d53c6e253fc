"""Shared helpers of the GPU parity tests: host<->device marshalling of bf16 bit patterns
and the comparisons against the oracle.

Tolerances
  * Stated bar (both kernels): max |y - ref| <= 2e-2 * max |ref| and mean relative error
    sum |y - ref| / sum |ref| <= 4e-3, per output tensor (ref in float64).
  * GEMV, elementwise bound derived from the kernel's arithmetic. Per 32-k slice the
    kernel computes a = silu(g) * u in fp32 as (g u / 2)(1 + tanh(g / 2)) with
    tanh.approx.f32 (relative error below 2^-10.5 here, so a_k is off by at most
    2^-10.5 |g_k u_k / 2|), encodes it as a16 = rint(a * 32767 / amax_slice), so each a_k
    is represented within amax_slice / 65534 (+ a few ulp of a from the scale's
    rounding); the slice's sum of a16 * q is exact in int32; then two fp32 scalings, the
    5-level warp butterfly and up to 16 cross-warp adds follow. So the fp32 result differs
    from the exact sum by at most
    delta = 64 * 2^-24 * sum_k |a_k| |W_nk| + 1.05 * sum_k (amax_slice(k) / 65534) |W_nk|
            + 1.01 * 2^-10.5 * sum_k |g_k u_k / 2| |W_nk|,
    and the single bf16 rounding adds at most 2^-8 of the value:
    |y - ref| <= 2^-8 * |ref| + 1.01 * delta.
  * GEMV on the tensor-core path (fd_gemv_uses_tensor_cores): both MMA operands are
    rounded to bf16, a' = bf16(silu(g) * u) with silu in its tanh form (tanh.approx.f32,
    relative error below 2^-10.5 here; the error it leaves in a is at most
    2^-10.5 * |g u / 2|) and w' = bf16(q * s); bf16 x bf16 products are exact in fp32
    and the tensor core accumulates in fp32, one rounding per K = 16 step (allowed
    2^-22 of the running magnitude each). So
    delta = 1.01 * (2^-8 * sum_k |a_k| |W_nk| + 2^-10.5 * sum_k |g_k u_k / 2| |W_nk|)
            + (K / 16 + 8) * 2^-22 * sum_k |a_k| |W_nk|,
    |y - ref| <= 2^-8 * |ref| + delta.
  * add-RMSNorm: residual_out bit-exact. out against the oracle's two-rounding form
    t = bf16(h * rstd), y = bf16(t * w): the kernel's rstd is fp32, so where h * rstd sits
    next to a bf16 rounding boundary t can land one step (ulp(t)) away; that moves t * w
    by |w| ulp(t), and the second rounding adds at most one ulp(y). So per element
    |y - y_eager| <= |w| ulp_bf16(t) + ulp_bf16(y). The page's own observation (at most
    one bf16 step, 0.031, at the outputs' largest magnitude) is reported as
    `max_abs_vs_eager`, and the stated bar is checked against the unrounded float64 form.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle


def dev_bf16(bits, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def dev_i32(words, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(words)).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_f64(bits) -> np.ndarray:
    return oracle.bf16_to_f32(bits).astype(np.float64)


def stated_bar(y: np.ndarray, ref: np.ndarray, max_abs_rel=2e-2, mean_rel=4e-3) -> dict:
    err = np.abs(y - ref)
    scale = np.max(np.abs(ref))
    res = {
        "max_abs_err": float(err.max(initial=0.0)),
        "max_abs_ref": float(scale),
        "mean_rel_err": float(err.sum() / max(np.abs(ref).sum(), 1e-300)),
    }
    assert res["max_abs_err"] <= max_abs_rel * scale, res
    assert res["mean_rel_err"] <= mean_rel, res
    return res


TANH_REL = 2.0**-10.5


def gemv_reference(gate, up, qweight, scales, group, rows=None):
    """(ref, abs_sum, enc_err, tanh_err), each [M, n], for all or the selected weight rows:
    the float64 result, sum_k |a_k| |W_nk|, sum_k (amax_slice(k) / 65534) |W_nk| and
    sum_k |g_k u_k / 2| |W_nk|."""
    if rows is not None:
        qweight = qweight[rows]
        scales = scales[rows]
    ref = oracle.swiglu_w4a16_gemv(gate, up, qweight, scales, group)
    a = np.abs(oracle.swiglu_activation(gate, up))
    if a.ndim == 1:
        a = a[None, :]
    w = np.abs(oracle.dequant_w4(qweight, scales, group).astype(np.float64))
    M, K = a.shape
    gu = 0.5 * np.abs(bf16_f64(gate) * bf16_f64(up)).reshape(M, K)
    amax = a.reshape(M, K // 32, 32).max(axis=2)
    enc = np.repeat(amax / 65534.0, 32, axis=1)
    return ref, a @ w.T, enc @ w.T, gu @ w.T


def gemv_sum_error(K, abs_sum, enc_err, tanh_err, tensor_cores):
    """Bound on |fp32 sum of the kernel - float64 sum| before the final bf16 rounding:
    bf16 operands (tensor cores) or the 16-bit activation encoding (CUDA cores), the
    tanh form of silu, and fp32 accumulation."""
    if tensor_cores:
        return 1.01 * (2.0**-8 * abs_sum + TANH_REL * tanh_err) + (K / 16 + 8) * 2.0**-22 * abs_sum
    return 1.01 * (64 * 2.0**-24 * abs_sum + 1.05 * enc_err + 1.01 * TANH_REL * tanh_err)


def check_gemv(y_bits, gate, up, qweight, scales, group, rows=None, tensor_cores=None) -> dict:
    """Stated bar plus the elementwise bound of the kernel that ran; by default the
    library is asked which one that was (under the current kernel selection)."""
    M = int(np.prod(np.shape(gate)[:-1])) if np.ndim(gate) > 1 else 1
    K = np.shape(gate)[-1]
    N = np.shape(qweight)[0]
    if tensor_cores is None:
        import memory_bound_decode_fd_gb300 as fd

        tensor_cores = fd.gemv_uses_tensor_cores(M, K, N, group)
    ref, abs_sum, enc_err, tanh_err = gemv_reference(gate, up, qweight, scales, group, rows)
    y = bf16_f64(y_bits)
    if rows is not None:
        y = y[:, rows]
    res = stated_bar(y, ref)
    bound = 2.0**-8 * np.abs(ref) + gemv_sum_error(K, abs_sum, enc_err, tanh_err, tensor_cores)
    res["tensor_cores"] = bool(tensor_cores)
    err = np.abs(y - ref)
    bad = err > bound
    assert not bad.any(), (
        f"{int(bad.sum())} outputs outside the derived bound; worst excess "
        f"{float((err - bound).max())}"
    )
    res["n_checked"] = int(y.size)
    return res


def check_gemv_residual(y_bits, gate, up, qweight, scales, residual, group,
                        tensor_cores=None) -> dict:
    """The residual-add epilogue: y = bf16(f32(residual) + fp32 sum), one rounding, against
    the oracle's float64 residual + sum. Same sum error as check_gemv; the final rounding
    (and the fp32 add) act on |residual + sum|."""
    M = int(np.prod(np.shape(gate)[:-1])) if np.ndim(gate) > 1 else 1
    K = np.shape(gate)[-1]
    N = np.shape(qweight)[0]
    if tensor_cores is None:
        import memory_bound_decode_fd_gb300 as fd

        tensor_cores = fd.gemv_uses_tensor_cores(M, K, N, group)
    ref, eager_bits = oracle.swiglu_w4a16_gemv_residual(gate, up, qweight, scales, residual, group)
    _, abs_sum, enc_err, tanh_err = gemv_reference(gate, up, qweight, scales, group)
    y = bf16_f64(y_bits).reshape(ref.shape)
    res = stated_bar(y, ref)
    bound = 2.0**-8 * np.abs(ref) + gemv_sum_error(K, abs_sum, enc_err, tanh_err, tensor_cores)
    err = np.abs(y - ref)
    bad = err > bound
    assert not bad.any(), (
        f"{int(bad.sum())} outputs outside the derived bound; worst excess "
        f"{float((err - bound).max())}"
    )
    res["tensor_cores"] = bool(tensor_cores)
    res["n_checked"] = int(y.size)
    # how often the unfused chain's two roundings are farther from the unrounded value
    res["eager_farther"] = float(np.mean(np.abs(bf16_f64(eager_bits).reshape(ref.shape) - ref) > err))
    return res


def w4a16_reference(x, qweight, scales, group, rows=None):
    """(ref, abs_sum, enc_err) of the plain GEMV for all or the selected weight rows: the
    float64 result, sum_k |x_k| |W_nk| and sum_k (amax_slice(k) / 65534) |W_nk|."""
    if rows is not None:
        qweight = qweight[rows]
        scales = scales[rows]
    ref = oracle.w4a16_gemv(x, qweight, scales, group)
    M, K = ref.shape[0], np.shape(x)[-1]
    xa = np.abs(bf16_f64(x)).reshape(M, K)
    w = np.abs(oracle.dequant_w4(qweight, scales, group).astype(np.float64))
    amax = xa.reshape(M, K // 32, 32).max(axis=2)
    enc = np.repeat(amax / 65534.0, 32, axis=1)
    return ref, xa @ w.T, enc @ w.T


def check_w4a16(y_bits, x, qweight, scales, group, rows=None) -> dict:
    """Stated bar plus the elementwise bound of the CUDA-core kernels for a plain
    activation (its 16-bit slice encoding and fp32 accumulation; no tanh term)."""
    K = np.shape(x)[-1]
    ref, abs_sum, enc_err = w4a16_reference(x, qweight, scales, group, rows)
    y = bf16_f64(y_bits).reshape(ref.shape[0], -1)
    if rows is not None:
        y = y[:, rows]
    res = stated_bar(y, ref)
    bound = 2.0**-8 * np.abs(ref) + gemv_sum_error(K, abs_sum, enc_err, 0.0, False)
    err = np.abs(y - ref)
    bad = err > bound
    assert not bad.any(), (
        f"{int(bad.sum())} outputs outside the derived bound; worst excess "
        f"{float((err - bound).max())}"
    )
    res["n_checked"] = int(y.size)
    return res


def ordered_key(bits) -> np.ndarray:
    """bf16 bit patterns -> integers whose order is the numeric order (adjacent values
    differ by 1; +0 and -0 both map to 0)."""
    b = np.asarray(bits).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_bf16(v) -> np.ndarray:
    """Spacing of bf16 values at |v| (2^(e-7) for |v| in [2^e, 2^(e+1)))."""
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0**-126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def check_add_rmsnorm(out_bits, res_bits, x, residual, weight, eps) -> dict:
    h_ref, y_ref, y_eager = oracle.add_rmsnorm(x, residual, weight, eps)
    assert np.array_equal(res_bits, h_ref), "residual_out is not bit-exact"
    y = bf16_f64(out_bits)
    res = stated_bar(y, y_ref)
    ye = bf16_f64(y_eager)
    w = np.broadcast_to(bf16_f64(weight), ye.shape)
    t = np.divide(y_ref, w, out=np.zeros_like(y_ref), where=w != 0)
    bound = np.abs(w) * ulp_bf16(t) + ulp_bf16(np.maximum(np.abs(ye), np.abs(y)))
    diff = np.abs(y - ye)
    steps = np.abs(ordered_key(out_bits) - ordered_key(y_eager))
    res["max_bf16_steps"] = int(steps.max(initial=0))
    res["frac_exact"] = float(np.mean(steps == 0))
    res["max_abs_vs_eager"] = float(diff.max(initial=0.0))
    assert np.all(diff <= bound * (1 + 1e-12)), (res, float((diff - bound).max()))
    assert res["frac_exact"] > 0.999, res
    return res


class GuardedBuffer:
    """A device buffer with sentinel-filled guard bands before and after the payload."""

    GUARD = 256  # elements on each side (512 bytes for bf16)

    def __init__(self, shape, dtype=torch.bfloat16, device="cuda", sentinel=-12345):
        n = int(np.prod(shape))
        self.raw = torch.empty(n + 2 * self.GUARD, dtype=dtype, device=device)
        self.raw.view(torch.int16 if dtype == torch.bfloat16 else dtype).fill_(sentinel)
        self.sentinel = sentinel
        self.tensor = self.raw[self.GUARD:self.GUARD + n].view(shape)

    def guards_intact(self) -> bool:
        v = self.raw.view(torch.int16) if self.raw.dtype == torch.bfloat16 else self.raw
        head = v[: self.GUARD]
        tail = v[-self.GUARD:]
        return bool((head == self.sentinel).all() and (tail == self.sentinel).all())
