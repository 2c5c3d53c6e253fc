"""Pins for the CPU oracle: each check ties an oracle function to something other than
itself - closed forms, identities, exhaustive tables, library routines on special
cases, brute force on tiny inputs, and the figures the source pages print
(tests/golden/page_figures.json). A plausible slip (dropped term, wrong sign, swapped
index, transposed operand, wrong nibble order or group index) fails at least one."""

import json
import math
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from memory_bound_decode_fd_gb300 import inputs, pack_int4

GOLDEN = json.loads((Path(__file__).parent / "golden" / "page_figures.json").read_text())


def bits_to_torch_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


# ------------------------------------------------------------------------------ bf16

def test_bf16_rne_matches_torch_on_random_and_ties():
    rng = np.random.default_rng(123)
    x = np.concatenate([
        rng.normal(0, 1, 200_000).astype(np.float32),
        (rng.normal(0, 1, 200_000) * 1e30).astype(np.float32),
        (rng.normal(0, 1, 200_000) * 1e-35).astype(np.float32),  # subnormal region
        rng.integers(0, 2**32, 400_000, dtype=np.uint32).view(np.float32),
    ])
    # exact ties: low half == 0x8000 with both parities of the kept LSB
    ties = (rng.integers(0, 2**16, 1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties, np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38], np.float32)])
    finite = ~np.isnan(x)
    ours = oracle.f32_to_bf16_rne(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours[finite], ref[finite])
    # NaN stays NaN
    nan_bits = oracle.f32_to_bf16_rne(np.array([np.nan], np.float32))
    assert np.isnan(oracle.bf16_to_f32(nan_bits))[0]


def test_bf16_widen_is_exact():
    bits = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f32(bits)
    ref = bits_to_torch_bf16(bits).float().numpy()
    same = (f.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(f) & np.isnan(ref))
    assert same.all()


# ------------------------------------------------------------------------------ silu

def test_silu_closed_forms():
    ln3 = math.log(3.0)
    # sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4, sigmoid(0) = 1/2
    got = oracle.silu(np.array([ln3, -ln3, 0.0, 2 * math.log(2.0)]))
    want = np.array([0.75 * ln3, -0.25 * ln3, 0.0, 0.8 * 2 * math.log(2.0)])
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)
    assert oracle.silu(np.array([0.0]))[0] == 0.0


def test_silu_odd_part_and_tails():
    x = np.linspace(-30, 30, 20001)
    # silu(x) - silu(-x) = x * (sigmoid(x) + sigmoid(-x)) = x
    np.testing.assert_allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=1e-13, atol=1e-13)
    assert oracle.silu(np.array([50.0]))[0] == 50.0
    assert abs(oracle.silu(np.array([-50.0]))[0]) < 1e-19
    assert oracle.silu(np.array([-1e4]))[0] == 0.0  # exp overflow -> -0.0, not NaN


def test_swiglu_activation_is_silu_gate_times_up():
    g = inputs.to_bf16_bits(np.array([[0.0, math.log(3.0), -2.5, 1.0]]))
    u = inputs.to_bf16_bits(np.array([[7.0, 2.0, -4.0, 0.0]]))
    a = oracle.swiglu_activation(g, u)
    gf = oracle.bf16_to_f32(g).astype(np.float64)
    assert a[0, 0] == 0.0 and a[0, 3] == 0.0
    np.testing.assert_allclose(a[0, 1], 2.0 * gf[0, 1] * 0.75, rtol=1e-2)  # ln3 rounded to bf16
    np.testing.assert_allclose(a[0, 2], -4.0 * -2.5 / (1 + math.exp(2.5)), rtol=1e-15)


# ------------------------------------------------------------------------------ int4

def test_unpack_nibble_order_and_sign():
    w = np.array([[0x76543210, 0x89ABCDEF - 2**32, 0x0000000F, 0x80000000 - 2**32]], np.int64).astype(np.int32)
    q = oracle.unpack_int4(w)
    assert q[0, 0:8].tolist() == [0, 1, 2, 3, 4, 5, 6, 7]
    assert q[0, 8:16].tolist() == [-1, -2, -3, -4, -5, -6, -7, -8]
    assert q[0, 16:24].tolist() == [-1, 0, 0, 0, 0, 0, 0, 0]
    assert q[0, 24:32].tolist() == [0, 0, 0, 0, 0, 0, 0, -8]


def test_unpack_exhaustive_table():
    # Every nibble value at every position: two's complement table.
    table = [v if v < 8 else v - 16 for v in range(16)]
    words = []
    for j in range(8):
        for v in range(16):
            words.append((v << (4 * j)) & 0xFFFFFFFF)
    w = np.array(words, dtype=np.uint32).view(np.int32).reshape(-1, 1)
    q = oracle.unpack_int4(w)
    for idx, (j, v) in enumerate((j, v) for j in range(8) for v in range(16)):
        expect = [0] * 8
        expect[j] = table[v]
        assert q[idx].tolist() == expect


def test_pack_then_unpack_roundtrip():
    rng = np.random.default_rng(5)
    q = rng.integers(-8, 8, size=(7, 64)).astype(np.int8)
    assert np.array_equal(oracle.unpack_int4(pack_int4(q)), q)


def test_generator_nibbles_are_uniform_on_minus8_to_7():
    rng = np.random.default_rng(0)
    q = oracle.unpack_int4(inputs.int4_words(rng, 64, 4096))
    counts = np.bincount((q.astype(np.int64) + 8).ravel(), minlength=16)
    assert q.min() == -8 and q.max() == 7
    expected = q.size / 16
    assert np.all(np.abs(counts - expected) < 6 * math.sqrt(expected))


def test_dequant_group_indexing_and_exactness():
    N, K, group = 3, 256, 64
    q = np.ones((N, K), np.int8)
    q[1] = -8
    q[2] = 7
    s = np.array([[2.0**-i for i in range(4)], [0.5, 0.25, 0.125, 0.0625], [0.01, 0.02, 0.005, 0.015]])
    sb = inputs.to_bf16_bits(s)
    w = oracle.dequant_w4(pack_int4(q), sb, group)
    sf = oracle.bf16_to_f32(sb)
    for n in range(N):
        for k in (0, 63, 64, 127, 128, 191, 192, 255):
            assert w[n, k] == np.float32(q[n, k]) * sf[n, k // group]
    assert w.dtype == np.float32


# ------------------------------------------------------------------------------ GEMV

def _a(g, u):
    return oracle.swiglu_activation(g, u)


def test_gemv_one_hot_pins_indices():
    rng = np.random.default_rng(7)
    M, K, N, group = 3, 256, 40, 64
    g = inputs.normal_bf16(rng, (M, K))
    u = inputs.normal_bf16(rng, (M, K))
    for (n_star, k_star, qv) in [(0, 0, 3), (39, 255, -8), (17, 129, 7), (5, 64, -1)]:
        q = np.zeros((N, K), np.int8)
        q[n_star, k_star] = qv
        s = np.full((N, K // group), 0.5)
        s[n_star, k_star // group] = 0.25
        y = oracle.swiglu_w4a16_gemv(g, u, pack_int4(q), inputs.to_bf16_bits(s), group)
        a = _a(g, u)
        expect = np.zeros((M, N))
        expect[:, n_star] = a[:, k_star] * qv * 0.25
        assert np.array_equal(y, expect)


def test_gemv_constant_weights_closed_form():
    rng = np.random.default_rng(8)
    M, K, N, group = 2, 512, 6, 128
    g = inputs.normal_bf16(rng, (M, K))
    u = inputs.normal_bf16(rng, (M, K))
    q = np.full((N, K), -3, np.int8)
    s = np.full((N, K // group), 0.015625)
    y = oracle.swiglu_w4a16_gemv(g, u, pack_int4(q), inputs.to_bf16_bits(s), group)
    a_sum = _a(g, u).sum(axis=1)
    for n in range(N):
        np.testing.assert_allclose(y[:, n], -3 * 0.015625 * a_sum, rtol=1e-12)


def test_gemv_group_scales_pin_k_over_group():
    rng = np.random.default_rng(9)
    M, K, N, group = 1, 512, 3, 128
    g = inputs.normal_bf16(rng, (M, K))
    u = inputs.normal_bf16(rng, (M, K))
    q = np.ones((N, K), np.int8)
    s = np.array([[1.0, 2.0, 4.0, 8.0], [8.0, 4.0, 2.0, 1.0], [1.0, 0.0, 0.0, 0.0]])
    y = oracle.swiglu_w4a16_gemv(g, u, pack_int4(q), inputs.to_bf16_bits(s), group)
    a = _a(g, u)[0]
    part = [a[i * group:(i + 1) * group].sum() for i in range(4)]
    np.testing.assert_allclose(y[0, 0], part[0] + 2 * part[1] + 4 * part[2] + 8 * part[3], rtol=1e-12)
    np.testing.assert_allclose(y[0, 1], 8 * part[0] + 4 * part[1] + 2 * part[2] + part[3], rtol=1e-12)
    np.testing.assert_allclose(y[0, 2], part[0], rtol=1e-12)


def test_gemv_brute_force_tiny():
    rng = np.random.default_rng(10)
    M, K, N, group = 2, 64, 5, 32
    d = inputs.gemv_inputs(M, K, N, group, rng=rng)
    y = oracle.swiglu_w4a16_gemv(d["gate"], d["up"], d["qweight"], d["scales"], group)
    g = oracle.bf16_to_f32(d["gate"]).astype(float)
    u = oracle.bf16_to_f32(d["up"]).astype(float)
    s = oracle.bf16_to_f32(d["scales"]).astype(float)
    words = d["qweight"].view(np.uint32)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                nib = (int(words[n, k // 8]) >> (4 * (k % 8))) & 0xF
                qk = nib - 16 if nib & 0x8 else nib
                gk = g[m, k]
                acc += gk / (1.0 + math.exp(-gk)) * u[m, k] * qk * s[n, k // group]
            assert abs(acc - y[m, n]) <= 1e-12 * max(1.0, abs(acc))


def test_gemv_rows_independent_and_linear_in_up():
    rng = np.random.default_rng(11)
    M, K, N, group = 4, 256, 9, 128
    d = inputs.gemv_inputs(M, K, N, group, rng=rng)
    y = oracle.swiglu_w4a16_gemv(d["gate"], d["up"], d["qweight"], d["scales"], group)
    y1 = oracle.swiglu_w4a16_gemv(d["gate"][2:3], d["up"][2:3], d["qweight"], d["scales"], group)
    np.testing.assert_allclose(y[2:3], y1, rtol=1e-13, atol=1e-13)
    # flipping the sign of up flips y exactly (bf16 negation is exact)
    neg_up = d["up"] ^ np.uint16(0x8000)
    yn = oracle.swiglu_w4a16_gemv(d["gate"], neg_up, d["qweight"], d["scales"], group)
    np.testing.assert_allclose(yn, -y, rtol=1e-13, atol=1e-13)
    # a subset of weight rows gives the same outputs for those rows
    ys = oracle.swiglu_w4a16_gemv(d["gate"], d["up"], d["qweight"][[1, 7]], d["scales"][[1, 7]], group)
    np.testing.assert_allclose(ys, y[:, [1, 7]], rtol=1e-13)


def test_gemv_matches_torch_linear_fp64():
    d = inputs.gemv_inputs(3, 1024, 64, 128, seed=12)
    y = oracle.swiglu_w4a16_gemv(d["gate"], d["up"], d["qweight"], d["scales"], 128)
    g = bits_to_torch_bf16(d["gate"]).double()
    u = bits_to_torch_bf16(d["up"]).double()
    a = torch.nn.functional.silu(g) * u
    w32 = torch.from_numpy(d["qweight"].astype(np.int64) & 0xFFFFFFFF)
    shifts = torch.arange(0, 32, 4, dtype=torch.int64)
    nib = (w32.unsqueeze(-1) >> shifts) & 0xF
    q = torch.where(nib >= 8, nib - 16, nib).reshape(64, 1024).double()
    s = bits_to_torch_bf16(d["scales"]).double().repeat_interleave(128, dim=1)
    ref = torch.nn.functional.linear(a, q * s).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------------------------ RMSNorm

def test_gemv_residual_zero_weights_pass_residual_through():
    # q = 0: the epilogue adds exactly nothing, so the new residual is the residual.
    rng = np.random.default_rng(40)
    M, K, N, group = 2, 256, 7, 128
    g = inputs.normal_bf16(rng, (M, K))
    u = inputs.normal_bf16(rng, (M, K))
    r = inputs.normal_bf16(rng, (M, N))
    q = np.zeros((N, K), np.int8)
    s = inputs.scales_bf16(rng, N, K, group)
    ref, eager = oracle.swiglu_w4a16_gemv_residual(g, u, pack_int4(q), s, r, group)
    assert np.array_equal(ref, oracle.bf16_to_f32(r).astype(np.float64))
    assert np.array_equal(eager, r)


def test_gemv_residual_one_hot_published_sigmoid():
    # gate = 1, up = 2 everywhere; one weight q = 5 with scale 0.25 at (n*, k*): the new
    # residual is r + 2 * silu(1) * 5 * 0.25 at n* (sigma(1) = 0.7310585786300049, the
    # tabulated logistic value) and exactly r elsewhere.
    M, K, N, group = 1, 128, 4, 64
    g = inputs.to_bf16_bits(np.ones((M, K)))
    u = inputs.to_bf16_bits(np.full((M, K), 2.0))
    r = inputs.to_bf16_bits(np.array([[0.5, -1.25, 3.0, 0.0]]))
    q = np.zeros((N, K), np.int8)
    q[2, 77] = 5
    s = inputs.to_bf16_bits(np.full((N, K // group), 0.25))
    ref, eager = oracle.swiglu_w4a16_gemv_residual(g, u, pack_int4(q), s, r, group)
    expect = np.array([[0.5, -1.25, 3.0 + 2 * 0.7310585786300049 * 5 * 0.25, 0.0]])
    np.testing.assert_allclose(ref, expect, rtol=1e-15, atol=0)
    # the unfused chain rounds y = 1.8276... to bf16 (1.828125) before the add
    assert oracle.bf16_to_f32(eager)[0, 2] == np.float32(4.8125)
    assert np.array_equal(eager[:, [0, 1, 3]], r[:, [0, 1, 3]])


def test_gemv_residual_shift_by_residual_is_exact():
    # Two residuals that differ by exactly representable amounts shift ref by exactly
    # that difference (the epilogue is an add, nothing else).
    rng = np.random.default_rng(41)
    M, K, N, group = 3, 256, 5, 128
    d = inputs.gemv_inputs(M, K, N, group, rng=rng)
    r1 = inputs.to_bf16_bits(np.full((M, N), 1.0))
    r2 = inputs.to_bf16_bits(np.full((M, N), -2.0))
    a1, _ = oracle.swiglu_w4a16_gemv_residual(d["gate"], d["up"], d["qweight"], d["scales"], r1, group)
    a2, _ = oracle.swiglu_w4a16_gemv_residual(d["gate"], d["up"], d["qweight"], d["scales"], r2, group)
    np.testing.assert_allclose(a1 - a2, 3.0, rtol=0, atol=1e-12)


def test_w4a16_gemv_brute_force_tiny():
    # y[m, n] = sum_k x q s written as loops over the packed words (nothing shared with
    # the oracle's unpack or dequant).
    rng = np.random.default_rng(42)
    M, K, N, group = 2, 64, 5, 32
    x = inputs.normal_bf16(rng, (M, K))
    qw = inputs.int4_words(rng, N, K)
    s = inputs.scales_bf16(rng, N, K, group)
    y = oracle.w4a16_gemv(x, qw, s, group)
    xf = oracle.bf16_to_f32(x).astype(float)
    sf = oracle.bf16_to_f32(s).astype(float)
    words = qw.view(np.uint32)
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                nib = (int(words[n, k // 8]) >> (4 * (k % 8))) & 0xF
                acc += xf[m, k] * (nib - 16 if nib & 0x8 else nib) * sf[n, k // group]
            assert abs(acc - y[m, n]) <= 1e-12 * max(1.0, abs(acc))


def test_gate_up_split_one_hot_pins_halves():
    # A one-hot weight in the up half (row I + j) appears in u[:, j] only; one in the gate
    # half (row j) in g[:, j] only; each is exactly x[k*] * q * s.
    M, K, inter, group = 2, 128, 6, 64
    rng = np.random.default_rng(43)
    x = inputs.normal_bf16(rng, (M, K))
    q = np.zeros((2 * inter, K), np.int8)
    q[inter + 4, 70] = -7
    q[1, 3] = 2
    s = inputs.to_bf16_bits(np.full((2 * inter, K // group), 0.5))
    g, u = oracle.gate_up_gemv(x, pack_int4(q), s, group)
    xf = oracle.bf16_to_f32(x).astype(float)
    expect_u = np.zeros((M, inter))
    expect_u[:, 4] = xf[:, 70] * -7 * 0.5
    expect_g = np.zeros((M, inter))
    expect_g[:, 1] = xf[:, 3] * 2 * 0.5
    assert np.array_equal(u, expect_u) and np.array_equal(g, expect_g)


def test_gate_up_matches_torch_linear_fp64():
    # Each half equals torch's float64 linear with that half's dequantised weights, built
    # here from torch's own bit ops on the packed words.
    rng = np.random.default_rng(44)
    M, K, inter, group = 3, 256, 10, 128
    x = inputs.normal_bf16(rng, (M, K))
    qw = inputs.int4_words(rng, 2 * inter, K)
    s = inputs.scales_bf16(rng, 2 * inter, K, group)
    g, u = oracle.gate_up_gemv(x, qw, s, group)
    words = torch.from_numpy(qw.view(np.uint32).astype(np.int64))
    shifts = torch.arange(8, dtype=torch.int64) * 4
    nib = (words.unsqueeze(-1) >> shifts) & 0xF
    qt = torch.where(nib >= 8, nib - 16, nib).reshape(2 * inter, K).double()
    st = torch.from_numpy(oracle.bf16_to_f32(s).astype(np.float64)).repeat_interleave(group, dim=1)
    xt = torch.from_numpy(oracle.bf16_to_f32(x).astype(np.float64))
    full = torch.nn.functional.linear(xt, qt * st).numpy()
    np.testing.assert_allclose(g, full[:, :inter], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(u, full[:, inter:], rtol=1e-13, atol=1e-13)


def test_add_rmsnorm_residual_matches_torch_bit_exact():
    d = inputs.rmsnorm_inputs(64, 1024, seed=20)
    h, _, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["weight"], 1e-6)
    ref = (bits_to_torch_bf16(d["x"]).float() + bits_to_torch_bf16(d["residual"]).float()).to(torch.bfloat16)
    assert np.array_equal(h, ref.view(torch.int16).numpy().view(np.uint16))


def test_add_rmsnorm_matches_torch_rms_norm_fp64():
    d = inputs.rmsnorm_inputs(32, 512, seed=21)
    h, y, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["weight"], 1e-5)
    hd = bits_to_torch_bf16(h).double()
    wd = bits_to_torch_bf16(d["weight"]).double()
    ref = torch.nn.functional.rms_norm(hd, (512,), wd, eps=1e-5).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_add_rmsnorm_unit_rms_before_weight():
    d = inputs.rmsnorm_inputs(16, 4096, seed=22)
    eps = 1e-6
    ones = inputs.to_bf16_bits(np.ones(4096))
    h, y, _ = oracle.add_rmsnorm(d["x"], d["residual"], ones, eps)
    hf = oracle.bf16_to_f32(h).astype(float)
    ms = np.mean(hf * hf, axis=1)
    np.testing.assert_allclose(np.mean(y * y, axis=1), ms / (ms + eps), rtol=1e-12)


def test_add_rmsnorm_constant_row_closed_form():
    hidden, eps = 256, 1e-5
    x = inputs.to_bf16_bits(np.full((2, hidden), 0.5))
    r = inputs.to_bf16_bits(np.stack([np.full(hidden, 1.0), np.full(hidden, -2.5)]))
    w = inputs.to_bf16_bits(np.linspace(0.5, 1.5, hidden))
    h, y, _ = oracle.add_rmsnorm(x, r, w, eps)
    wf = oracle.bf16_to_f32(w).astype(float)
    for i, c in enumerate([1.5, -2.0]):
        np.testing.assert_allclose(y[i], c / math.sqrt(c * c + eps) * wf, rtol=1e-14)


def test_add_rmsnorm_eager_variant_matches_torch_eager_chain():
    # The eager chain written with torch ops (fp32 variance and rsqrt; round to bf16;
    # multiply by the bf16 weight) agrees with the oracle's two-rounding variant to one
    # bf16 step everywhere, and exactly almost everywhere.
    d = inputs.rmsnorm_inputs(256, 1024, seed=23)
    eps = 1e-6
    h, _, ye = oracle.add_rmsnorm(d["x"], d["residual"], d["weight"], eps)
    ht = bits_to_torch_bf16(h).float()
    var = ht.pow(2).mean(-1, keepdim=True)
    t = (ht * torch.rsqrt(var + eps)).to(torch.bfloat16)
    ref = (bits_to_torch_bf16(d["weight"]) * t).view(torch.int16).numpy().view(np.uint16)
    a = oracle.bf16_to_f32(ye).astype(float)
    b = oracle.bf16_to_f32(ref).astype(float)
    step = np.abs(oracle.bf16_to_f32(oracle.f32_to_bf16_rne(np.abs(b) * (1 + 2.0**-7))) - np.abs(b))
    assert np.all(np.abs(a - b) <= np.maximum(step, 1e-30) * 1.0001)
    assert np.mean(ye == ref) > 0.99


def test_rmsnorm_output_step_matches_page_0031():
    # The page's "one BF16 rounding step (0.031)" is the bf16 spacing 2^-5 of values in
    # [4, 8): the largest normalised outputs of the 8192 x 4096 workload land there.
    d = inputs.rmsnorm_inputs(1024, 4096, seed=1)
    _, y, _ = oracle.add_rmsnorm(d["x"], d["residual"], d["weight"], 1e-6)
    top = np.max(np.abs(y))
    assert 4.0 <= top < 8.0
    assert abs(2.0 ** (math.floor(math.log2(top)) - 7) - GOLDEN["add_rmsnorm_parity"]["y_step_value"]) < 5e-4


# ------------------------------------------------------------------------------ decode step

def test_decode_step_zero_weights_pass_residual_through():
    hidden, inter, group = 64, 128, 32
    rng = np.random.default_rng(30)
    x0 = inputs.normal_bf16(rng, (1, hidden))
    r0 = inputs.normal_bf16(rng, (1, hidden))
    layers = []
    for _ in range(2):
        layers.append({
            "rms_weight": inputs.normal_bf16(rng, (hidden,), 1.0, 0.1),
            "gate": inputs.normal_bf16(rng, (1, inter)),
            "up": inputs.normal_bf16(rng, (1, inter)),
            "qweight": np.zeros((hidden, inter // 8), np.int32),
            "scales": inputs.to_bf16_bits(np.full((hidden, inter // group), 0.01)),
        })
    rec, x_last, res = oracle.decode_mlp_step(x0, r0, layers, 1e-5, group)
    h1 = oracle.f32_to_bf16_rne(oracle.bf16_to_f32(x0) + oracle.bf16_to_f32(r0))
    assert np.array_equal(rec[0][0], h1)
    assert np.array_equal(rec[1][0], h1)  # x_1 = 0, so h_2 = h_1
    assert np.all(rec[0][3] == 0) and np.all(oracle.bf16_to_f32(x_last) == 0)
    assert np.array_equal(res, h1)


def _torch_bf16(v: float) -> float:
    """A float rounded to bf16 by torch (independent of the oracle's rounding)."""
    return float(torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).float())


def _torch_bf16_bits(v) -> np.ndarray:
    t = torch.as_tensor(np.asarray(v, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# The two-layer chain of the pin below (hidden 64, MLP width 128, group 32, eps 1e-5):
#   x0 = r0 = 0.5 everywhere, so h1 = 1.0 everywhere;
#   layer 1: rms_weight 1.0; gate 1, up 2, one int4 weight q = -8 at (n1, k1) with scale
#            3/32: y1[n1] = silu(1) * 2 * (-8) * 3/32, every other output 0;
#   x1 = bf16(y1): bf16(y1[n1]) = -1.09375, so h2 = bf16(-1.09375 + 1.0) = -0.09375 at
#            n1 (with x1 left unrounded the same add gives -0.0966796875) and 1.0 elsewhere;
#   layer 2: rms_weight 0.5; gate -1, up 1, one weight q = 5 at (n2, k2) with scale 1/4:
#            y2[n2] = silu(-1) * 5 / 4.
PIN_HIDDEN, PIN_INTER, PIN_GROUP, PIN_EPS = 64, 128, 32, 1e-5
PIN_N1, PIN_K1, PIN_N2, PIN_K2 = 17, 37, 40, 100
SIGMOID_1 = 0.7310585786300049  # 1 / (1 + e^-1), published value (also in the GEMV pins)


def _pin_layers():
    def one_hot(n, k, q, s):
        qq = np.zeros((PIN_HIDDEN, PIN_INTER), np.int8)
        qq[n, k] = q
        ss = np.full((PIN_HIDDEN, PIN_INTER // PIN_GROUP), 0.5)
        ss[n, k // PIN_GROUP] = s
        return pack_int4(qq), inputs.to_bf16_bits(ss)

    q1, s1 = one_hot(PIN_N1, PIN_K1, -8, 3 / 32)
    q2, s2 = one_hot(PIN_N2, PIN_K2, 5, 0.25)
    full = lambda v, shape: inputs.to_bf16_bits(np.full(shape, v))  # noqa: E731
    return [
        {"rms_weight": full(1.0, (PIN_HIDDEN,)), "gate": full(1.0, (1, PIN_INTER)),
         "up": full(2.0, (1, PIN_INTER)), "qweight": q1, "scales": s1},
        {"rms_weight": full(0.5, (PIN_HIDDEN,)), "gate": full(-1.0, (1, PIN_INTER)),
         "up": full(1.0, (1, PIN_INTER)), "qweight": q2, "scales": s2},
    ]


def _check_two_layer_pin(step_fn):
    """Run `step_fn` (decode_mlp_step or a planted mutant) on the two-layer chain and
    assert every field of every layer against the values worked out by hand above."""
    H = PIN_HIDDEN
    x0 = inputs.to_bf16_bits(np.full((1, H), 0.5))
    r0 = inputs.to_bf16_bits(np.full((1, H), 0.5))
    rec, x_last, res = step_fn(x0, r0, _pin_layers(), PIN_EPS, PIN_GROUP)
    assert len(rec) == 2

    # layer 1: h = 1 everywhere; unit mean square; weight 1
    y1 = SIGMOID_1 * 2.0 * -8 * (3 / 32)
    rstd1 = 1.0 / math.sqrt(1.0 + PIN_EPS)
    h1 = np.full((1, H), 1.0)
    assert np.array_equal(rec[0][0], _torch_bf16_bits(h1))
    np.testing.assert_allclose(rec[0][1], np.full((1, H), rstd1), rtol=1e-14)
    assert np.array_equal(rec[0][2], _torch_bf16_bits(np.full((1, H), _torch_bf16(_torch_bf16(rstd1) * 1.0))))
    y1_ref = np.zeros((1, H))
    y1_ref[0, PIN_N1] = y1
    np.testing.assert_allclose(rec[0][3], y1_ref, rtol=1e-15, atol=0)

    # layer 2: x1 = bf16(y1) joins the residual h1
    x1_hot = _torch_bf16(y1)
    assert x1_hot == -1.09375
    h2_hot = _torch_bf16(x1_hot + 1.0)
    assert h2_hot == -0.09375
    h2 = np.full((1, H), 1.0)
    h2[0, PIN_N1] = h2_hot
    ms2 = ((H - 1) * 1.0 + h2_hot * h2_hot) / H
    rstd2 = 1.0 / math.sqrt(ms2 + PIN_EPS)
    assert np.array_equal(rec[1][0], _torch_bf16_bits(h2))
    np.testing.assert_allclose(rec[1][1], h2 * rstd2 * 0.5, rtol=1e-14)
    eager2 = np.array([[_torch_bf16(_torch_bf16(v * rstd2) * 0.5) for v in h2[0]]])
    assert np.array_equal(rec[1][2], _torch_bf16_bits(eager2))
    y2 = -(1.0 - SIGMOID_1) * 5 * 0.25  # silu(-1) = -sigmoid(-1) = -(1 - sigmoid(1))
    y2_ref = np.zeros((1, H))
    y2_ref[0, PIN_N2] = y2
    np.testing.assert_allclose(rec[1][3], y2_ref, rtol=1e-14, atol=0)

    # after the chain: x_2 = bf16(y2), the residual stream is h2
    x2 = np.zeros((1, H))
    x2[0, PIN_N2] = _torch_bf16(y2)
    assert np.array_equal(np.asarray(x_last).reshape(1, H), _torch_bf16_bits(x2))
    assert np.array_equal(np.asarray(res).reshape(1, H), _torch_bf16_bits(h2))


def test_decode_step_two_layer_closed_form():
    # Every field of every layer's record, the handed-on x and the final residual.
    # [FUSE] "The fusion boundary problem" (add_rmsnorm writes the residual and the
    # normalised row; the down projection's output joins the stream at the next add);
    # [KFM] Step 2 (h rounded to bf16, then normalised; two roundings of the output).
    _check_two_layer_pin(oracle.decode_mlp_step)


def _mutant_step(slip):
    """decode_mlp_step with one planted mistake, built from the oracle's own pieces."""
    def step(x_bits, residual_bits, layers, eps, group):
        x = np.asarray(x_bits, dtype=np.uint16)
        xf = None  # the unrounded x of the "unrounded x_next" slip
        res = np.asarray(residual_bits, dtype=np.uint16)
        record = []
        for i, layer in enumerate(layers):
            w = layers[(i + 1) % len(layers)]["rms_weight"] if slip == "wrong_weight" else layer["rms_weight"]
            if xf is not None:
                h_bits = oracle.f32_to_bf16_rne(xf + oracle.bf16_to_f32(res))
                _, y_norm, y_eager = oracle.add_rmsnorm(np.zeros_like(res), h_bits, w, eps)
            else:
                h_bits, y_norm, y_eager = oracle.add_rmsnorm(x, res, w, eps)
            if slip == "no_rstd":
                y_norm = oracle.bf16_to_f32(h_bits).astype(np.float64) * oracle.bf16_to_f32(w)
            y = oracle.swiglu_w4a16_gemv(layer["gate"], layer["up"], layer["qweight"], layer["scales"], group)
            record.append((h_bits, y_norm, y_eager, y))
            y_bits = oracle.f32_to_bf16_rne(y.astype(np.float32)).reshape(x.shape)
            if slip == "swap_roles":
                res, x = y_bits, h_bits
            else:
                res, x = h_bits, y_bits
            if slip == "unrounded_x":
                xf = y.astype(np.float32).reshape(x.shape)
        return record, x, res
    return step


@pytest.mark.parametrize("slip", ["wrong_weight", "unrounded_x", "swap_roles", "no_rstd"])
def test_decode_step_pin_catches_planted_slips(slip):
    # Each plausible mistake in the chain (the next layer's norm weight, x handed on
    # without its bf16 rounding, residual and x exchanged, the rstd factor dropped) fails
    # the closed-form pin.
    with pytest.raises(AssertionError):
        _check_two_layer_pin(_mutant_step(slip))


def test_decode_step_pin_mutant_harness_is_faithful():
    # With no slip planted the mutant harness passes the pin, so the failures above come
    # from the planted mistakes alone.
    _check_two_layer_pin(_mutant_step(None))


def test_contract_is_the_plain_triple_loop():
    rng = np.random.default_rng(77)
    a = rng.normal(size=(3, 20))
    w = rng.normal(size=(5, 20))
    ref = np.zeros((3, 5))
    for m in range(3):
        for n in range(5):
            acc = 0.0
            for k in range(20):
                acc += float(a[m, k]) * float(w[n, k])
            ref[m, n] = acc
    np.testing.assert_allclose(oracle.contract(a, w), ref, rtol=1e-13, atol=1e-13)
    t = torch.nn.functional.linear(torch.from_numpy(a), torch.from_numpy(w)).numpy()
    np.testing.assert_allclose(oracle.contract(a, w), t, rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------------------ NVFP4

# The FP4 E2M1 code points (sign, 2 exponent bits, 1 mantissa bit), written out as values:
# the eight magnitudes 0, 1/2, 1, 3/2, 2, 3, 4, 6, then the same with the sign set.
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
               -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def torch_e4m3(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e2m1_codes_are_the_fp4_values():
    v = oracle.e2m1_to_f64(np.arange(16))
    assert v.tolist() == E2M1_VALUES
    assert np.signbit(v[8]) and not np.signbit(v[0])


def test_e4m3_matches_torch_float8_e4m3fn_on_every_code():
    codes = np.arange(256)
    v, t = oracle.e4m3_to_f64(codes), torch_e4m3(codes)
    nan = np.isnan(t)
    assert np.array_equal(np.isnan(v), nan) and np.nonzero(nan)[0].tolist() == [0x7F, 0xFF]
    assert np.array_equal(v[~nan], t[~nan])
    assert np.array_equal(np.signbit(v[~nan]), np.signbit(t[~nan]))  # -0.0 at 0x80
    assert v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9 and v[0x38] == 1.0


def test_unpack_fp4_even_k_in_low_nibble():
    codes = oracle.unpack_fp4(np.array([[0x21, 0xF0]], dtype=np.uint8))
    assert codes.tolist() == [[1, 2, 0, 15]]


def nvfp4_brute(x, x_sf, w, w_sf, alpha):
    """Element by element: nibbles by integer division, values from the code table,
    scales from torch's float8_e4m3fn."""
    sx, sw = torch_e4m3(x_sf), torch_e4m3(w_sf)
    M, N, K = x.shape[0], w.shape[0], 2 * x.shape[1]

    def elem(b, r, k):
        byte = int(b[r, k // 2])
        return E2M1_VALUES[byte % 16 if k % 2 == 0 else byte // 16]

    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += elem(x, m, k) * sx[m, k // 16] * elem(w, n, k) * sw[n, k // 16]
            out[m, n] = float(alpha) * acc
    return out


def test_nvfp4_brute_force_tiny():
    # With these scale codes every product is a multiple of 2^-16 below 2^11, so the
    # sums are exact in float64 in any order and the two sides agree bit for bit.
    d = inputs.nvfp4_inputs(M=3, K=48, N=5, rng=np.random.default_rng(40))
    ref, _ = oracle.nvfp4_scaled_mm(d["x"], d["x_sf"], d["w"], d["w_sf"], d["alpha"])
    assert np.array_equal(ref, nvfp4_brute(d["x"], d["x_sf"], d["w"], d["w_sf"], d["alpha"]))


def test_nvfp4_one_hot_pins_block_index_and_packing():
    # one nonzero element at k = 17 (high nibble of byte 8, block 1) in x row 0 and in
    # w row 3; distinct scales per block, so k // 8 or k // 32 picks another scale
    M, N, K = 2, 4, 64
    x = np.zeros((M, K // 2), np.uint8)
    w = np.zeros((N, K // 2), np.uint8)
    x[0, 8] = 0x20          # code 2 = 1.0 at k = 17
    w[3, 8] = 0x50          # code 5 = 3.0 at k = 17
    x_sf = np.tile(np.array([0x38, 0x40, 0x48, 0x50], np.uint8), (M, 1))   # 1, 2, 4, 8
    w_sf = np.tile(np.array([0x30, 0x28, 0x20, 0x18], np.uint8), (N, 1))   # 1/2, 1/4, 1/8, 1/16
    ref, eager = oracle.nvfp4_scaled_mm(x, x_sf, w, w_sf, np.float32(1.5))
    want = np.zeros((M, N))
    want[0, 3] = 1.5 * (1.0 * 2.0) * (3.0 * 0.25)
    assert np.array_equal(ref, want)
    assert np.array_equal(eager, oracle.f32_to_bf16_rne(want.astype(np.float32)))


def test_nvfp4_output_scale_fold_against_the_unfolded_pair():
    d = inputs.nvfp4_inputs(M=16, K=256, N=64, rng=np.random.default_rng(41))
    args = (d["x"], d["x_sf"], d["w"], d["w_sf"])
    ref1, eager1 = oracle.nvfp4_scaled_mm(*args, np.float32(1.0))
    # alpha = 1: the separate multiplication changes nothing
    assert np.array_equal(eager1, oracle.f32_to_bf16_rne(ref1.astype(np.float32)))
    # a power of two commutes with rounding: folded and unfolded agree exactly
    ref4, eager4 = oracle.nvfp4_scaled_mm(*args, np.float32(0.25))
    assert np.array_equal(ref4, 0.25 * ref1)
    assert np.array_equal(eager4, oracle.f32_to_bf16_rne(ref4.astype(np.float32)))
    # any other alpha scales the exact sum; the unfolded pair rounds twice, stays within
    # one bf16 step of the once-rounded folded result and differs from it somewhere
    ref, eager = oracle.nvfp4_scaled_mm(*args, np.float32(0.7))
    assert np.array_equal(ref, float(np.float32(0.7)) * ref1)
    fused = oracle.bf16_to_f32(oracle.f32_to_bf16_rne(ref.astype(np.float32))).astype(np.float64)
    e = oracle.bf16_to_f32(eager).astype(np.float64)
    assert np.all(np.abs(e - fused) <= np.abs(fused) * 2.0 ** -7)
    assert np.any(e != fused)


def test_nvfp4_zero_scale_and_negative_zero_contribute_nothing():
    d = inputs.nvfp4_inputs(M=2, K=64, N=3, rng=np.random.default_rng(42))
    ref, _ = oracle.nvfp4_scaled_mm(d["x"], d["x_sf"], d["w"], d["w_sf"], d["alpha"])
    x_sf = d["x_sf"].copy()
    x_sf[0, :] = 0x00                                         # row 0: every block scale 0
    x = d["x"].copy()
    x[1, :] = 0x88                                            # row 1: every element -0.0
    ref0, _ = oracle.nvfp4_scaled_mm(x, x_sf, d["w"], d["w_sf"], d["alpha"])
    assert np.all(ref0 == 0.0)
    assert np.any(ref != 0.0)


def test_nvfp4_fold_removes_one_launch_per_layer():
    # the page's figures agree with one folded output multiplication (one launch) per
    # decoder layer, the QKV projection's, over Llama-3's 32 layers; the default NVFP4
    # workload is that projection at the page's batch
    f = GOLDEN["nvfp4_output_scale_fold"]
    assert f["graph_nodes_before"] - f["graph_nodes_after"] == f["fewer_launches_per_step"]
    layers = GOLDEN["silu_traffic_llama3_8b"]["layers"]
    assert f["fewer_launches_per_step"] == f["scaling_launches_removed_per_layer"] * layers
    d = inputs.nvfp4_inputs(K=64, N=8)
    assert d["M"] == f["batch"]


def test_nvfp4_generator_draws_valid_codes():
    d = inputs.nvfp4_inputs(M=64, K=512, N=128, seed=5)
    for key in ("x_sf", "w_sf"):
        sf = d[key]
        assert sf.dtype == np.uint8 and np.all(sf >> 7 == 0)
        e = sf >> 3
        assert e.min() == 3 and e.max() == 9
        assert set(np.unique(sf & 7).tolist()) == set(range(8))
    codes = oracle.unpack_fp4(d["w"])
    assert set(np.unique(codes).tolist()) == set(range(16))
    assert d["x"].shape == (64, 256) and d["w"].shape == (128, 256)
    assert d["x_sf"].shape == (64, 32) and 0.5 <= d["alpha"] < 2.0


# ------------------------------------------------------------------------------ page figures

def test_byte_model_unfused_product_is_94mb():
    f = GOLDEN["unfused_product"]
    b = oracle.unfused_product_bytes(f["M"], f["K"], f["N"], f["dtype_bytes"])
    assert b == 94_371_840
    assert round(b / 1e6) == f["approx_MB"]


def test_byte_model_silu_traffic_llama3():
    f = GOLDEN["silu_traffic_llama3_8b"]
    per = f["inter"] * f["dtype_bytes"]
    assert round(per / 1024) == f["silu_output_KB_per_token_per_layer"]
    assert round(2 * per / 1024) == f["saved_KB_per_token_per_layer"]
    assert round(2 * per * f["layers"] / 1e6, 1) == f["saved_MB_per_token"]


def test_byte_model_eager_rmsnorm_42_vs_8():
    f = GOLDEN["add_rmsnorm_eager_vs_fused"]
    assert len(oracle.eager_add_rmsnorm_kernels()) == f["eager_kernels"]
    assert oracle.eager_add_rmsnorm_bytes_per_elem() == f["eager_bytes_per_elem"]
    elems = f["rows"] * f["hidden"]
    bw = f["mixed_rw_GBps"] * 1e9
    assert round(elems * f["eager_bytes_per_elem"] / bw * 1e3, 1) == f["eager_ms"]
    assert round(elems * f["fused_bytes_per_elem"] / bw * 1e3, 2) == f["fused_ms"]
    assert round(f["eager_ms"] / f["fused_ms"], 1) == f["speedup"]


def test_byte_model_swiglu_10_vs_6():
    f = GOLDEN["swiglu_eager_vs_fused"]
    assert oracle.eager_swiglu_bytes_per_elem() == f["eager_bytes_per_elem"]
    assert oracle.fused_swiglu_bytes_per_elem() == f["fused_bytes_per_elem"]
    assert round(f["flops_per_elem"] / oracle.fused_swiglu_bytes_per_elem(), 1) == f["flops_per_byte"]
    assert round(100 * (1 - 6 / 10)) == f["time_cut_pct"]
