"""GPU parity of the tensor-core (tcgen05) kernel of fd_swiglu_w4a16_gemv against the CPU
oracle, through the C ABI: the batched-decode workload (M=64, K=14336, N=4096, seed 4)
in full, ragged M around the MMA tile sizes, K and N at the kernel's divisibility rules,
the layout (one-hot weights), agreement with the CUDA-core kernel, and the call
properties (deterministic, graph-capturable, no allocation, no stray writes)."""

import gc

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
import oracle
from memory_bound_decode_fd_gb300 import inputs
from fd_check import GuardedBuffer, check_gemv, dev_bf16, dev_i32, host_bits, bf16_f64, stated_bar

pytestmark = pytest.mark.gpu


@pytest.fixture
def tensor_path(cuda_device):
    prev = fd.set_gemv_path("tensor")
    yield
    fd.set_gemv_path(prev)


def run_gemv(d, out=None):
    g, u = dev_bf16(d["gate"]), dev_bf16(d["up"])
    q, s = dev_i32(d["qweight"]), dev_bf16(d["scales"])
    y = fd.swiglu_w4a16_gemv(g, u, q, s, out=out, group=d["group"])
    torch.cuda.synchronize()
    return host_bits(y)


def test_tc_batched_m64_every_output(tensor_path):
    # Batched decode M=64, K=14336, N=4096, group 128, seed 4: all 262144 outputs.
    d = inputs.batched_inputs()["gemv"]
    assert fd.gemv_uses_tensor_cores(64, 14336, 4096, 128)
    y = run_gemv(d)
    res = check_gemv(y, d["gate"], d["up"], d["qweight"], d["scales"], 128)
    assert res["tensor_cores"] and res["n_checked"] == 64 * 4096


def test_auto_selects_tensor_cores_from_m16(cuda_device):
    prev = fd.set_gemv_path("auto")
    try:
        assert fd.gemv_uses_tensor_cores(64, 14336, 4096, 128)
        assert fd.gemv_uses_tensor_cores(16, 1024, 128, 128)
        assert not fd.gemv_uses_tensor_cores(15, 1024, 128, 128)
        assert not fd.gemv_uses_tensor_cores(1, 14336, 4096, 128)
        assert not fd.gemv_uses_tensor_cores(64, 14336, 4000, 128)  # N % 128
        assert not fd.gemv_uses_tensor_cores(64, 14336 + 32, 4096, 32)  # K % 1024
        assert not fd.gemv_uses_tensor_cores(64, 2048, 256, 32)  # group % 64
    finally:
        fd.set_gemv_path(prev)


TC_SHAPES = [
    # M, K, N, group
    (1, 1024, 128, 128),      # one activation row, padded to the MMA's N = 16
    (16, 1024, 128, 128),     # smallest K and N
    (17, 1024, 256, 64),      # N = 32 tile, 15 padded rows
    (31, 2048, 128, 128),
    (32, 4096, 384, 128),
    (33, 2048, 128, 256),     # two groups per K quarter
    (48, 2048, 256, 128),
    (63, 1024, 128, 128),
    (64, 9216, 2560, 128),    # the K=9216 N=2560 shape at M=64
    (65, 1024, 128, 128),     # N = 128 tile
    (100, 2048, 256, 128),
    (128, 1024, 128, 128),
    (129, 1024, 128, 128),    # two row blocks: 128 + 1
    (200, 2048, 128, 64),
    (256, 1024, 256, 128),    # largest M
    (16, 16384, 128, 512),
    (20, 32768, 128, 64),     # largest K; 136-column scale window
    (33, 32768, 128, 64),     # the same at 64 rows: 64-k steps (128-k stages do not fit)
    (64, 32768, 256, 64),
]


@pytest.mark.parametrize("M,K,N,group", TC_SHAPES)
def test_tc_shapes(tensor_path, M, K, N, group):
    assert fd.gemv_uses_tensor_cores(M, K, N, group)
    d = inputs.gemv_inputs(M, K, N, group, seed=2000 + M + K + N + group)
    y = run_gemv(d)
    res = check_gemv(y, d["gate"], d["up"], d["qweight"], d["scales"], group)
    assert res["tensor_cores"]


@pytest.mark.parametrize("n_star,k_star,qv", [(0, 0, 3), (2559, 9215, -8), (1234, 4097, 7),
                                              (77, 31, -1), (128, 2304, 5), (255, 6911, -7)])
def test_tc_one_hot_layout(tensor_path, n_star, k_star, qv):
    # A single nonzero weight: every other output is exactly zero (index mapping, nibble
    # pairing, k order inside the core matrices, scale index, K quarter and n tile).
    M, K, N, group = 20, 9216, 2560, 128
    rng = np.random.default_rng(6)
    gate = inputs.normal_bf16(rng, (M, K))
    up = inputs.normal_bf16(rng, (M, K))
    q = np.zeros((N, K), np.int8)
    q[n_star, k_star] = qv
    s = np.full((N, K // group), 0.5)
    s[n_star, k_star // group] = 0.75
    d = {"gate": gate, "up": up, "qweight": fd.pack_int4(q), "scales": inputs.to_bf16_bits(s),
         "group": group}
    y = run_gemv(d)
    yf = oracle.bf16_to_f32(y)
    mask = np.ones((M, N), bool)
    mask[:, n_star] = False
    assert np.all(yf[mask] == 0.0)
    # the hot column: one product of two bf16 operands, rounded once
    a = oracle.swiglu_activation(gate, up)[:, k_star]
    expect = a * qv * 0.75
    got = yf[:, n_star].astype(np.float64)
    assert np.all(np.abs(got - expect) <= 2.0**-7 * np.abs(expect) + 2.0**-10.5 * 0.5 * np.abs(
        bf16_f64(gate)[:, k_star] * bf16_f64(up)[:, k_star]) * abs(qv) * 0.75 + 1e-30)


def test_tc_agrees_with_cuda_core_m64(cuda_device):
    # The two kernels of the batched workload (M=64, K=14336, N=4096, seed 4) agree with
    # each other within the stated bar, and each meets its own bound.
    d = inputs.batched_inputs()["gemv"]
    outs = {}
    for p in ("tensor", "cuda_core"):
        prev = fd.set_gemv_path(p)
        try:
            outs[p] = run_gemv(d)
        finally:
            fd.set_gemv_path(prev)
    stated_bar(bf16_f64(outs["tensor"]), bf16_f64(outs["cuda_core"]))
    stated_bar(bf16_f64(outs["cuda_core"]), bf16_f64(outs["tensor"]))


def test_tc_back_to_back_calls_identical(tensor_path):
    d = inputs.gemv_inputs(64, 14336, 4096, 128, seed=12)
    g, u = dev_bf16(d["gate"]), dev_bf16(d["up"])
    q, s = dev_i32(d["qweight"]), dev_bf16(d["scales"])
    outs = torch.empty((16, 64, 4096), dtype=torch.bfloat16, device="cuda")
    for i in range(16):
        fd.swiglu_w4a16_gemv(g, u, q, s, out=outs[i])
    torch.cuda.synchronize()
    bits = host_bits(outs)
    assert all(np.array_equal(bits[i], bits[0]) for i in range(1, 16))
    check_gemv(bits[0], d["gate"], d["up"], d["qweight"], d["scales"], 128)


def test_tc_graph_replay_matches_eager(tensor_path):
    d = inputs.gemv_inputs(64, 14336, 4096, 128, seed=13)
    g, u = dev_bf16(d["gate"]), dev_bf16(d["up"])
    q, s = dev_i32(d["qweight"]), dev_bf16(d["scales"])
    eager = fd.swiglu_w4a16_gemv(g, u, q, s)
    out = torch.empty_like(eager)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fd.swiglu_w4a16_gemv(g, u, q, s, out=out)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(graph):
        fd.swiglu_w4a16_gemv(g, u, q, s, out=out)
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out), host_bits(eager))


def test_tc_guard_bands_untouched(tensor_path):
    d = inputs.gemv_inputs(20, 2048, 384, 128, seed=14)
    buf = GuardedBuffer((20, 384))
    run_gemv(d, out=buf.tensor)
    assert buf.guards_intact()
    check_gemv(host_bits(buf.tensor), d["gate"], d["up"], d["qweight"], d["scales"], 128)


def test_tc_allocates_nothing(tensor_path):
    d = inputs.gemv_inputs(64, 9216, 2560, 128, seed=15)
    g, u = dev_bf16(d["gate"]), dev_bf16(d["up"])
    q, s = dev_i32(d["qweight"]), dev_bf16(d["scales"])
    out = torch.empty((64, 2560), dtype=torch.bfloat16, device="cuda")
    fd.swiglu_w4a16_gemv(g, u, q, s, out=out)
    gc.collect()
    gc.disable()
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    torch.cuda.reset_peak_memory_stats()
    for _ in range(5):
        fd.swiglu_w4a16_gemv(g, u, q, s, out=out)
    torch.cuda.synchronize()
    gc.enable()
    assert torch.cuda.memory_allocated() == before
    assert torch.cuda.max_memory_allocated() == before
    assert torch.cuda.mem_get_info()[0] == free_before


def test_tc_with_pdl_matches_plain(tensor_path):
    # Programmatic dependent launch: gate/up written by the previous kernel in the stream
    # (a copy) must be read only after it completes.
    d = inputs.gemv_inputs(64, 4096, 1024, 128, seed=16)
    g_src, u_src = dev_bf16(d["gate"]), dev_bf16(d["up"])
    q, s = dev_i32(d["qweight"]), dev_bf16(d["scales"])
    g, u = torch.zeros_like(g_src), torch.zeros_like(u_src)
    plain = fd.swiglu_w4a16_gemv(g_src, u_src, q, s)
    prev = fd.set_pdl(True)
    try:
        outs = []
        for _ in range(4):
            g.zero_()
            u.zero_()
            g.copy_(g_src)
            u.copy_(u_src)
            outs.append(fd.swiglu_w4a16_gemv(g, u, q, s))
        torch.cuda.synchronize()
    finally:
        fd.set_pdl(prev)
    for o in outs:
        assert np.array_equal(host_bits(o), host_bits(plain))
