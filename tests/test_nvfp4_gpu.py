"""GPU parity of fd_nvfp4_scaled_mm (the NVFP4 matmul with its fp32 output multiplier folded
in, on the tensor cores' block-scaled MMA) against the oracle's nvfp4_scaled_mm, called
through the C ABI on seeded synthetic codes.

Tolerance. Every product X[m, k] * W[n, k] (E2M1 x E2M1 x E4M3 x E4M3: at most 2 + 2 + 4 + 4
significant bits) is exact in fp32; the tensor core accumulates in fp32 (allowed one
rounding of 2^-23 of the running magnitude per 16-element block, plus 8 more), alpha
multiplies the fp32 sum (2^-24) and the store rounds once to bf16 (2^-8):
    |y - ref| <= 2^-8 |ref| + |alpha| (K/16 + 8) 2^-23 S + 2^-23 |ref|,  S = sum_k |X||W|,
with ref = alpha * sum_k X W in float64. The stated bar (max |y - ref| <= 2e-2 max |ref|,
mean relative error <= 4e-3) is checked as well.
"""

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
import oracle
from memory_bound_decode_fd_gb300 import inputs
from fd_check import GuardedBuffer, bf16_f64, host_bits, stated_bar

pytestmark = pytest.mark.gpu


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_alpha(v):
    return torch.tensor([float(v)], dtype=torch.float32, device="cuda")


def run(d, out=None, alpha=None):
    a = dev_alpha(d["alpha"]) if alpha is None else alpha
    y = fd.nvfp4_scaled_mm(dev_u8(d["x"]), dev_u8(d["x_sf"]), dev_u8(d["w"]), dev_u8(d["w_sf"]),
                           a, out=out)
    torch.cuda.synchronize()
    return host_bits(y)


def check_nvfp4(y_bits, d) -> dict:
    ref, eager_bits = oracle.nvfp4_scaled_mm(d["x"], d["x_sf"], d["w"], d["w_sf"], d["alpha"])
    y = bf16_f64(y_bits).reshape(ref.shape)
    res = stated_bar(y, ref)
    xa = np.abs(oracle.nvfp4_dequant(d["x"], d["x_sf"]))
    wa = np.abs(oracle.nvfp4_dequant(d["w"], d["w_sf"]))
    S = xa @ wa.T
    K = xa.shape[1]
    alpha = abs(float(np.float32(d["alpha"])))
    bound = 2.0**-8 * np.abs(ref) + alpha * (K / 16 + 8) * 2.0**-23 * S + 2.0**-23 * np.abs(ref)
    err = np.abs(y - ref)
    bad = err > bound
    assert not bad.any(), (f"{int(bad.sum())} outputs outside the derived bound; worst excess "
                           f"{float((err - bound).max())}")
    eager = bf16_f64(eager_bits).reshape(ref.shape)
    res["n_checked"] = int(y.size)
    # the folded result (one rounding) is never farther from the exact value than the
    # unfolded pair's two roundings allow
    res["frac_equal_to_unfolded"] = float(np.mean(y_bits.reshape(ref.shape) == eager_bits))
    res["folded_closer_or_equal"] = float(np.mean(err <= np.abs(eager - ref)))
    return res


def test_qkv_workload_every_output(cuda_device):
    # M=64 K=4096 N=6144, seed 5: the Llama-3.1-8B QKV projection at batch 64.
    d = inputs.nvfp4_inputs()
    res = check_nvfp4(run(d), d)
    assert res["n_checked"] == 64 * 6144
    assert res["folded_closer_or_equal"] > 0.99


SHAPES = [
    # M, K, N: batch paddings 16/32/64/128, every K split (1, 2, 4, 8), ragged weight tiles
    (1, 256, 128),
    (2, 512, 1),
    (16, 768, 200),
    (17, 1024, 129),
    (31, 1536, 300),
    (33, 2048, 256),
    (64, 3072, 384),
    (65, 4096, 130),
    (100, 6144, 256),
    (128, 8192, 128),
    (129, 1024, 64),     # two launches of up to 128 activation rows
    (256, 2048, 200),
]


@pytest.mark.parametrize("M,K,N", SHAPES)
def test_shapes_every_output(cuda_device, M, K, N):
    d = inputs.nvfp4_inputs(M, K, N, seed=600 + M + K + N)
    res = check_nvfp4(run(d), d)
    assert res["n_checked"] == M * N


@pytest.mark.parametrize("n_star,k_star,code", [(0, 0, 0x1), (37, 17, 0x7), (100, 4095, 0xB),
                                                 (127, 2048, 0xE), (6143, 1000, 0x5)])
def test_one_hot_weight_pins_rows_blocks_and_nibbles(cuda_device, n_star, k_star, code):
    # One nonzero weight code at (n*, k*) with its own block scale: column n* of the output
    # is alpha * X[:, k*] * W[n*, k*] (exact products, one rounding), every other output is
    # zero. Rows in every TMEM lane quarter and both nibbles of a byte are covered.
    M, K, N = 64, 4096, 6144
    d = inputs.nvfp4_inputs(M, K, N, seed=71)
    codes = np.zeros((N, K), np.uint8)
    codes[n_star, k_star] = code
    d["w"] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sf = np.full((N, K // 16), 0x38, np.uint8)  # 1.0
    sf[n_star, k_star // 16] = 0x4B             # E4M3 (1 + 3/8) * 2^(9 - 7) = 5.5
    d["w_sf"] = sf
    bits = run(d)
    y = bf16_f64(bits).reshape(M, N)
    mask = np.ones((M, N), bool)
    mask[:, n_star] = False
    assert np.all(y[mask] == 0)
    assert np.count_nonzero(y[:, n_star]) > 0
    check_nvfp4(bits, d)


@pytest.mark.parametrize("m_star,k_star", [(0, 5), (31, 64), (32, 1023), (63, 4094)])
def test_one_hot_activation_pins_batch_rows(cuda_device, m_star, k_star):
    # One nonzero activation code at (m*, k*): row m* of the output is alpha * X * W[:, k*];
    # every other row is zero (the activation scales' TMEM layout, batch rows 0..63).
    M, K, N = 64, 4096, 512
    d = inputs.nvfp4_inputs(M, K, N, seed=72)
    codes = np.zeros((M, K), np.uint8)
    codes[m_star, k_star] = 0x6  # 4.0
    d["x"] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    bits = run(d)
    y = bf16_f64(bits).reshape(M, N)
    mask = np.ones((M, N), bool)
    mask[m_star, :] = False
    assert np.all(y[mask] == 0)
    assert np.count_nonzero(y[m_star]) > 0
    check_nvfp4(bits, d)


def test_alpha_is_read_from_device_memory_at_run_time(cuda_device):
    # The 0-dim multiplier is read by the kernel: a CUDA graph captured once gives the
    # result for the value alpha holds at each replay.
    d = inputs.nvfp4_inputs(16, 1024, 256, seed=73)
    x, xs, w, ws = dev_u8(d["x"]), dev_u8(d["x_sf"]), dev_u8(d["w"]), dev_u8(d["w_sf"])
    alpha = dev_alpha(1.0)
    out = torch.empty((16, 256), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        fd.nvfp4_scaled_mm(x, xs, w, ws, alpha, out=out)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fd.nvfp4_scaled_mm(x, xs, w, ws, alpha, out=out)
    for v in (1.0, 0.75, 1.9375, -0.5):
        alpha.fill_(v)
        g.replay()
        torch.cuda.synchronize()
        check_nvfp4(host_bits(out), dict(d, alpha=np.float32(v)))


def test_graph_and_pdl_match_eager_bitwise(cuda_device):
    d = inputs.nvfp4_inputs(64, 4096, 1024, seed=74)
    eager = run(d)
    x, xs, w, ws = dev_u8(d["x"]), dev_u8(d["x_sf"]), dev_u8(d["w"]), dev_u8(d["w_sf"])
    alpha = dev_alpha(d["alpha"])
    out = torch.empty((64, 1024), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    prev = fd.set_pdl(True)
    try:
        with torch.cuda.stream(stream):
            for _ in range(2):
                fd.nvfp4_scaled_mm(x, xs, w, ws, alpha, out=out)
        stream.synchronize()
        assert np.array_equal(host_bits(out), eager)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(3):
                fd.nvfp4_scaled_mm(x, xs, w, ws, alpha, out=out)
        out.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(out), eager)
    finally:
        fd.set_pdl(prev)


def test_guard_bands_untouched(cuda_device):
    M, K, N = 17, 2048, 129
    d = inputs.nvfp4_inputs(M, K, N, seed=75)
    gb = GuardedBuffer((M, N))
    y = run(d, out=gb.tensor)
    assert gb.guards_intact()
    check_nvfp4(y, d)


def test_zero_scales_give_zero(cuda_device):
    d = inputs.nvfp4_inputs(32, 1024, 256, seed=76)
    d["w_sf"] = np.zeros_like(d["w_sf"])
    y = bf16_f64(run(d))
    assert np.all(y == 0)

