"""GPU parity of fd_w4a16_gate_up_gemv (the gate and up projections as one horizontally
fused W4A16 GEMV) against the CPU oracle, through the C ABI: the Llama-3-8B-shaped
projection (K=4096, I=14336) on sampled rows, ragged and small shapes on every output,
the split of the stacked weight into its two halves, both kernels, no stray writes, and
the whole fused MLP (gate/up GEMV, then the SwiGLU-prologue down projection with its
residual epilogue) after add_rmsnorm in a CUDA graph with programmatic dependent launch."""

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
import oracle
from memory_bound_decode_fd_gb300 import inputs, pack_int4
from fd_check import GuardedBuffer, check_gemv_residual, check_w4a16, dev_bf16, dev_i32, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["auto", "cuda_core"])
def gemv_path(request, cuda_device):
    """The default kernel choice (the bulk-copy kernel where its layout rules hold) and
    the CUDA-core ring kernel forced."""
    prev = fd.set_gemv_path(request.param)
    yield request.param
    fd.set_gemv_path(prev)


def gate_up_inputs(M, K, inter, group, seed):
    rng = np.random.default_rng(seed)
    return {"x": inputs.normal_bf16(rng, (M, K)), "qweight": inputs.int4_words(rng, 2 * inter, K),
            "scales": inputs.scales_bf16(rng, 2 * inter, K, group), "group": group}


def run(d, gate_out=None, up_out=None):
    g, u = fd.w4a16_gate_up_gemv(dev_bf16(d["x"]), dev_i32(d["qweight"]), dev_bf16(d["scales"]),
                                 gate_out=gate_out, up_out=up_out, group=d["group"])
    torch.cuda.synchronize()
    return host_bits(g), host_bits(u)


SHAPES = [
    # M, K, I, group
    (1, 4096, 1024, 128),    # the model width, fewer rows
    (1, 8192, 256, 128),     # x of 16 KB: still read by the lanes directly
    (1, 9216, 256, 128),     # x of 18 KB: bulk-copied into shared memory first
    (1, 1024, 300, 128),     # ragged rows per CTA
    (1, 4096, 2500, 64),
    (3, 4096, 500, 128),     # two activation rows per pass + one
    (2, 2048, 1000, 128),
    (16, 1024, 256, 128),
    (1, 96, 7, 32),          # CUDA-core kernel only (K % 1024 != 0)
    (5, 160, 33, 32),
]


@pytest.mark.parametrize("M,K,inter,group", SHAPES)
def test_gate_up_every_output(gemv_path, M, K, inter, group):
    d = gate_up_inputs(M, K, inter, group, seed=800 + M + K + inter)
    g, u = run(d)
    res = check_w4a16(np.concatenate([g, u], axis=1), d["x"], d["qweight"], d["scales"], group)
    assert res["n_checked"] == M * 2 * inter


def test_gate_up_llama_shape_every_output(gemv_path):
    # K=4096 (model width), I=14336 (MLP width): all 28672 stacked rows.
    M, K, inter, group = 1, 4096, 14336, 128
    d = gate_up_inputs(M, K, inter, group, seed=17)
    g, u = run(d)
    res = check_w4a16(np.concatenate([g, u], axis=1), d["x"], d["qweight"], d["scales"], group)
    assert res["n_checked"] == 2 * inter


def test_gate_up_one_hot_lands_in_its_half(gemv_path):
    # One weight in the gate half and one in the up half: every other output is exactly
    # zero, and the two hot ones are within the kernel's bound of x[k*] q s.
    M, K, inter, group = 1, 4096, 14336, 128
    rng = np.random.default_rng(18)
    x = inputs.normal_bf16(rng, (M, K))
    q = np.zeros((2 * inter, K), np.int8)
    q[77, 4000] = 5
    q[inter + 13000, 129] = -8
    s = inputs.to_bf16_bits(np.full((2 * inter, K // group), 0.25))
    d = {"x": x, "qweight": pack_int4(q), "scales": s, "group": group}
    g, u = run(d)
    gf, uf = oracle.bf16_to_f32(g), oracle.bf16_to_f32(u)
    gmask = np.ones_like(gf, bool)
    gmask[0, 77] = False
    umask = np.ones_like(uf, bool)
    umask[0, 13000] = False
    assert np.all(gf[gmask] == 0) and np.all(uf[umask] == 0)
    rows = np.array([77, inter + 13000])
    check_w4a16(np.concatenate([g, u], axis=1), x, d["qweight"], s, group, rows=rows)


def test_gate_up_guard_bands_untouched(gemv_path):
    M, K, inter, group = 3, 2048, 300, 128
    d = gate_up_inputs(M, K, inter, group, seed=19)
    gb, ub = GuardedBuffer((M, inter)), GuardedBuffer((M, inter))
    run(d, gate_out=gb.tensor, up_out=ub.tensor)
    assert gb.guards_intact() and ub.guards_intact()
    check_w4a16(np.concatenate([host_bits(gb.tensor), host_bits(ub.tensor)], axis=1), d["x"],
                d["qweight"], d["scales"], group)


def test_gate_up_back_to_back_identical(cuda_device):
    d = gate_up_inputs(1, 4096, 14336, 128, seed=20)
    x, q, s = dev_bf16(d["x"]), dev_i32(d["qweight"]), dev_bf16(d["scales"])
    outs = [fd.w4a16_gate_up_gemv(x, q, s) for _ in range(4)]
    torch.cuda.synchronize()
    for g, u in outs[1:]:
        assert np.array_equal(host_bits(g), host_bits(outs[0][0]))
        assert np.array_equal(host_bits(u), host_bits(outs[0][1]))


def test_fused_mlp_layer_in_a_graph_with_pdl(cuda_device):
    # The decode layer of the pages' fully fused form: add_rmsnorm -> (normed, h);
    # gate/up GEMV on normed -> g, u; down projection with the SwiGLU prologue and the
    # residual epilogue -> h + down(silu(g) u), in place in h. Eager and graph replays
    # (programmatic dependent launch) agree bit for bit; each kernel is checked against
    # the oracle on the bytes it read.
    hidden, inter, group, eps = 4096, 14336, 128, 1e-5
    rng = np.random.default_rng(21)
    x = inputs.normal_bf16(rng, (1, hidden))
    r = inputs.normal_bf16(rng, (1, hidden))
    w = inputs.to_bf16_bits(1.0 + 0.1 * rng.standard_normal(hidden))
    qgu = inputs.int4_words(rng, 2 * inter, hidden)
    sgu = inputs.scales_bf16(rng, 2 * inter, hidden, group)
    qd = inputs.int4_words(rng, hidden, inter)
    sd = inputs.scales_bf16(rng, hidden, inter, group)
    xd, rd, wd = dev_bf16(x), dev_bf16(r), dev_bf16(w)
    qgu_d, sgu_d, qd_d, sd_d = dev_i32(qgu), dev_bf16(sgu), dev_i32(qd), dev_bf16(sd)
    normed = torch.empty_like(xd)
    h = torch.empty_like(xd)
    g = torch.empty((1, inter), dtype=torch.bfloat16, device="cuda")
    u = torch.empty_like(g)

    def layer():
        fd.add_rmsnorm(xd, rd, wd, eps, out=normed, residual_out=h)
        fd.w4a16_gate_up_gemv(normed, qgu_d, sgu_d, gate_out=g, up_out=u, group=group)
        fd.swiglu_w4a16_gemv_residual(g, u, qd_d, sd_d, h, out=h, group=group)

    prev = fd.set_pdl(True)
    try:
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            fd.add_rmsnorm(xd, rd, wd, eps, out=normed, residual_out=h)
            stream.synchronize()
            normed_bits, h_bits = host_bits(normed), host_bits(h)
            layer()
        stream.synchronize()
        eager = [host_bits(t) for t in (g, u, h)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            layer()
        for _ in range(3):
            for t in (g, u, h):
                t.fill_(0)
            graph.replay()
            torch.cuda.synchronize()
            for t, e in zip((g, u, h), eager):
                assert np.array_equal(host_bits(t), e)
    finally:
        fd.set_pdl(prev)
    g_bits, u_bits, out_bits = eager
    check_w4a16(np.concatenate([g_bits, u_bits], axis=1), normed_bits, qgu, sgu, group)
    check_gemv_residual(out_bits, g_bits, u_bits, qd, sd, h_bits, group)
