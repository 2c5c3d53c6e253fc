"""GPU parity of fd_swiglu_w4a16_gemv_residual (the down projection with a residual-add
epilogue, new_residual = x + out) against the CPU oracle, through the C ABI: every kernel
(bulk-copy M=1 and small M, CUDA-core ring, tensor cores), in place, the exact
pass-through with zero weights, agreement with the plain GEMV, graph capture with
programmatic dependent launch, and no stray writes."""

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
import oracle  # noqa: F401
from memory_bound_decode_fd_gb300 import inputs, pack_int4
from fd_check import GuardedBuffer, bf16_f64, check_gemv_residual, dev_bf16, dev_i32, host_bits, ulp_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["auto", "cuda_core", "tensor"])
def gemv_path(request, cuda_device):
    prev = fd.set_gemv_path(request.param)
    yield request.param
    fd.set_gemv_path(prev)


def residual_inputs(M, K, N, group, seed):
    d = inputs.gemv_inputs(M, K, N, group, seed=seed)
    d["residual"] = inputs.normal_bf16(np.random.default_rng(seed + 100), (M, N))
    return d


def run(d, out=None, residual_dev=None):
    g, u = dev_bf16(d["gate"]), dev_bf16(d["up"])
    q, s = dev_i32(d["qweight"]), dev_bf16(d["scales"])
    r = residual_dev if residual_dev is not None else dev_bf16(d["residual"])
    y = fd.swiglu_w4a16_gemv_residual(g, u, q, s, r, out=out, group=d["group"])
    torch.cuda.synchronize()
    return host_bits(y)


SHAPES = [
    # M, K, N, group
    (1, 14336, 4096, 128),   # the decode-step down projection
    (1, 9216, 2560, 128),
    (1, 1024, 256, 128),
    (1, 4096, 1000, 64),     # ragged rows per CTA
    (3, 4096, 1000, 128),    # two activation rows per pass + one
    (16, 2048, 384, 128),    # tensor cores from M = 16 (default choice)
    (64, 14336, 4096, 128),  # batched decode
    (1, 96, 7, 32),          # CUDA-core kernel only (K % 1024 != 0)
]


@pytest.mark.parametrize("M,K,N,group", SHAPES)
def test_residual_epilogue_every_output(gemv_path, M, K, N, group):
    d = residual_inputs(M, K, N, group, seed=500 + M + K + N)
    y = run(d)
    res = check_gemv_residual(y, d["gate"], d["up"], d["qweight"], d["scales"], d["residual"], group)
    assert res["n_checked"] == M * N


@pytest.mark.parametrize("M,K,N,group", [(1, 14336, 4096, 128), (3, 4096, 1000, 128), (64, 2048, 384, 128)])
def test_residual_in_place_matches_out_of_place(gemv_path, M, K, N, group):
    d = residual_inputs(M, K, N, group, seed=600 + M)
    apart = run(d)
    r = dev_bf16(d["residual"])
    inplace = run(d, out=r, residual_dev=r)
    assert np.array_equal(inplace, apart)


@pytest.mark.parametrize("M,K,N,group", [(1, 14336, 4096, 128), (2, 2048, 300, 128), (32, 2048, 256, 128)])
def test_zero_weights_pass_residual_through_exactly(gemv_path, M, K, N, group):
    rng = np.random.default_rng(700 + M)
    d = {"gate": inputs.normal_bf16(rng, (M, K)), "up": inputs.normal_bf16(rng, (M, K)),
         "qweight": pack_int4(np.zeros((N, K), np.int8)),
         "scales": inputs.scales_bf16(rng, N, K, group), "group": group,
         "residual": inputs.normal_bf16(rng, (M, N))}
    assert np.array_equal(run(d), d["residual"])


def test_one_hot_weight_adds_one_product(cuda_device):
    # A single nonzero weight: every other output is the residual bit for bit; the hot
    # column is bf16(r + a[k*] q s) within the kernel's bound.
    M, K, N, group = 1, 14336, 4096, 128
    rng = np.random.default_rng(9)
    gate = inputs.normal_bf16(rng, (M, K))
    up = inputs.normal_bf16(rng, (M, K))
    q = np.zeros((N, K), np.int8)
    q[3001, 12345] = -6
    s = inputs.scales_bf16(rng, N, K, group)
    d = {"gate": gate, "up": up, "qweight": pack_int4(q), "scales": s, "group": group,
         "residual": inputs.normal_bf16(rng, (M, N))}
    y = run(d)
    mask = np.ones((M, N), bool)
    mask[:, 3001] = False
    assert np.array_equal(y[mask], d["residual"][mask])
    check_gemv_residual(y, gate, up, d["qweight"], s, d["residual"], group)


def test_agrees_with_plain_gemv_plus_residual(cuda_device):
    # The fused epilogue and the unfused chain (GEMV rounded to bf16, then the add) differ
    # only by the rounding of y: within one bf16 step of the sum plus half a step of y.
    d = residual_inputs(1, 14336, 4096, 128, seed=13)
    fused = bf16_f64(run(d))
    g, u = dev_bf16(d["gate"]), dev_bf16(d["up"])
    q, s = dev_i32(d["qweight"]), dev_bf16(d["scales"])
    plain = fd.swiglu_w4a16_gemv(g, u, q, s, group=128)
    torch.cuda.synchronize()
    yb = bf16_f64(host_bits(plain))
    chain = yb + bf16_f64(d["residual"])
    assert np.all(np.abs(fused - chain) <= ulp_bf16(chain) + 0.5 * ulp_bf16(yb))


def test_guard_bands_untouched(gemv_path):
    d = residual_inputs(3, 2048, 300, 128, seed=14)
    buf = GuardedBuffer((3, 300))
    run(d, out=buf.tensor)
    assert buf.guards_intact()
    check_gemv_residual(host_bits(buf.tensor), d["gate"], d["up"], d["qweight"], d["scales"],
                        d["residual"], 128)


def test_graph_with_pdl_after_add_rmsnorm(cuda_device):
    # The decode layer of a fused model: add_rmsnorm writes the residual stream h, the down
    # projection adds its output to h in place. Captured in a CUDA graph with programmatic
    # dependent launch; the GEMV must read h only after add_rmsnorm has written it.
    hidden, inter, group = 4096, 14336, 128
    rng = np.random.default_rng(15)
    x = inputs.normal_bf16(rng, (1, hidden))
    r = inputs.normal_bf16(rng, (1, hidden))
    w = inputs.to_bf16_bits(1.0 + 0.1 * rng.standard_normal(hidden))
    d = inputs.gemv_inputs(1, inter, hidden, group, seed=16)
    h_bits, _, _ = oracle.add_rmsnorm(x, r, w, 1e-5)
    xd, rd, wd = dev_bf16(x), dev_bf16(r), dev_bf16(w)
    g, u = dev_bf16(d["gate"]), dev_bf16(d["up"])
    q, s = dev_i32(d["qweight"]), dev_bf16(d["scales"])
    normed = torch.empty_like(xd)
    h = torch.empty_like(xd)
    prev = fd.set_pdl(True)
    try:
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            fd.add_rmsnorm(xd, rd, wd, 1e-5, out=normed, residual_out=h)
            fd.swiglu_w4a16_gemv_residual(g, u, q, s, h, out=h, group=group)
        stream.synchronize()
        eager = host_bits(h)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            fd.add_rmsnorm(xd, rd, wd, 1e-5, out=normed, residual_out=h)
            fd.swiglu_w4a16_gemv_residual(g, u, q, s, h, out=h, group=group)
        for _ in range(3):
            h.fill_(0)
            graph.replay()
            torch.cuda.synchronize()
            assert np.array_equal(host_bits(h), eager)
    finally:
        fd.set_pdl(prev)
    check_gemv_residual(eager, d["gate"], d["up"], d["qweight"], d["scales"], h_bits, group)
