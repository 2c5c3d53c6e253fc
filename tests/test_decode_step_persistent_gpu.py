"""The decode step as one persistent launch (fd_decode_mlp_step): every layer's normalised
row and GEMV output, and the final residual, equal bit for bit the chain of separate calls
(add_rmsnorm, then swiglu_w4a16_gemv, per layer) on the same inputs; that chain's every
layer is itself checked against the oracle in test_decode_step_gpu.py. Also: single-layer
and short chains, two calls in a row, another hidden size, the step captured in a CUDA
graph and run end to end through pinned host memory, and a clean device status."""

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
from memory_bound_decode_fd_gb300 import inputs
from fd_check import dev_bf16, dev_i32, host_bits

pytestmark = pytest.mark.gpu

EPS = 1e-5


def device_layers(d):
    return [{
        "rms_weight": dev_bf16(L["rms_weight"]),
        "gate": dev_bf16(L["gate"]),
        "up": dev_bf16(L["up"]),
        "qweight": dev_i32(L["qweight"]),
        "scales": dev_bf16(L["scales"]),
    } for L in d["layers"]]


def separate_chain(d, layers):
    """The chain of separate calls: per layer (normed, residual after, y) as host bits."""
    x = dev_bf16(d["x"])
    res = dev_bf16(d["residual"])
    rec = []
    for L in layers:
        normed, _ = fd.add_rmsnorm(x, res, L["rms_weight"], EPS, residual_out=res)
        y = fd.swiglu_w4a16_gemv(L["gate"], L["up"], L["qweight"], L["scales"], group=d["group"])
        torch.cuda.synchronize()
        rec.append((host_bits(normed), host_bits(res), host_bits(y)))
        x = y
    return rec


def persistent(d, layers):
    """One fd_decode_mlp_step call over `layers`: (normed list, y list, residual) bits."""
    x = dev_bf16(d["x"])
    res = dev_bf16(d["residual"])
    normed = [torch.full((1, d["hidden"]), float("nan"), dtype=torch.bfloat16, device="cuda")
              for _ in layers]
    ys = [torch.full((1, d["hidden"]), float("nan"), dtype=torch.bfloat16, device="cuda")
          for _ in layers]
    table = fd.step_layer_table(layers, normed, ys)
    scratch = fd.step_scratch(len(layers), d["hidden"])
    fd.decode_mlp_step_persistent(x, res, table, EPS, d["inter"], d["group"], scratch)
    torch.cuda.synchronize()
    return [host_bits(t) for t in normed], [host_bits(t) for t in ys], host_bits(res)


def assert_same(got, rec):
    normed, ys, res = got
    assert len(normed) == len(rec)
    for l, (n_ref, _, y_ref) in enumerate(rec):
        assert np.array_equal(normed[l].reshape(-1), n_ref.reshape(-1)), f"normed of layer {l}"
        assert np.array_equal(ys[l].reshape(-1), y_ref.reshape(-1)), f"y of layer {l}"
    assert np.array_equal(res.reshape(-1), rec[-1][1].reshape(-1)), "final residual"


@pytest.fixture(scope="module")
def step_data():
    return inputs.decode_step_inputs(layers=32, seed=3)


@pytest.fixture(scope="module")
def dev_layers(cuda_device, step_data):
    return device_layers(step_data)


@pytest.fixture(scope="module")
def chain(cuda_device, step_data, dev_layers):
    return separate_chain(step_data, dev_layers)


def test_persistent_step_equals_the_separate_calls(step_data, dev_layers, chain):
    assert_same(persistent(step_data, dev_layers), chain)


@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_persistent_short_chains(step_data, dev_layers, chain, n):
    # one layer: no count between layers, the residual is written after the exit count
    assert_same(persistent(step_data, dev_layers[:n]), chain[:n])


def test_persistent_twice_in_a_row(step_data, dev_layers):
    # the second call starts from zeroed counters again (the call zeroes its scratch)
    a = persistent(step_data, dev_layers[:4])
    b = persistent(step_data, dev_layers[:4])
    for ta, tb in zip(a[0] + a[1] + [a[2]], b[0] + b[1] + [b[2]]):
        assert np.array_equal(ta, tb)


def test_persistent_other_hidden(cuda_device):
    # hidden 2048: 13 or 14 rows per CTA (two chunks), the same partition as the GEMV
    d = inputs.decode_step_inputs(layers=3, hidden=2048, seed=11)
    layers = device_layers(d)
    assert_same(persistent(d, layers), separate_chain(d, layers))


@pytest.mark.parametrize("hidden", [8, 64, 1216, 4104, 4408])
def test_persistent_edge_hidden(cuda_device, hidden):
    # 1 CTA of 8 rows; 8 CTAs; 8 rows on every SM; 27 rows on every SM (a last chunk of
    # 3 rows); 29 rows on every SM, the most whose weights fit one CTA's shared memory
    d = inputs.decode_step_inputs(layers=2, hidden=hidden, seed=13)
    layers = device_layers(d)
    assert_same(persistent(d, layers), separate_chain(d, layers))


def test_persistent_long_chain(cuda_device):
    # 48 layers (the two h rows alternate 24 times each; 48 counters) at 8 rows per SM
    d = inputs.decode_step_inputs(layers=48, hidden=1216, seed=15)
    layers = device_layers(d)
    assert_same(persistent(d, layers), separate_chain(d, layers))


def test_persistent_rows_beyond_shared_memory_are_unsupported(cuda_device):
    # hidden 8192: 54 rows per CTA do not fit one CTA's shared memory; nothing is launched
    from memory_bound_decode_fd_gb300 import _lib

    d = inputs.decode_step_inputs(layers=1, hidden=8192, seed=14)
    layers = device_layers(d)
    x = dev_bf16(d["x"])
    res = dev_bf16(d["residual"])
    res0 = res.clone()
    normed = [torch.zeros((1, 8192), dtype=torch.bfloat16, device="cuda")]
    ys = [torch.zeros((1, 8192), dtype=torch.bfloat16, device="cuda")]
    table = fd.step_layer_table(layers, normed, ys)
    with pytest.raises(_lib.FdError) as e:
        fd.decode_mlp_step_persistent(x, res, table, EPS, d["inter"], d["group"],
                                      fd.step_scratch(1, 8192))
    assert e.value.status == _lib.FD_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.equal(res.view(torch.int16), res0.view(torch.int16))
    assert not normed[0].view(torch.int16).any() and not ys[0].view(torch.int16).any()


def _decode_step(d, layers, persistent_mode):
    from memory_bound_decode_fd_gb300.step import DecodeStep

    st = DecodeStep([{k: L[k] for k in ("rms_weight", "qweight", "scales")} for L in layers],
                    d["hidden"], d["inter"], d["group"], EPS, pdl=True, persistent=persistent_mode)
    st.x.copy_(dev_bf16(d["x"]))
    st.residual.copy_(dev_bf16(d["residual"]))
    for i, L in enumerate(layers):
        st.gate[i].copy_(L["gate"])
        st.up[i].copy_(L["up"])
    return st


def test_persistent_step_in_a_graph(step_data, dev_layers, chain):
    st = _decode_step(step_data, dev_layers, True)
    x0, r0 = st.x.clone(), st.residual.clone()
    st.capture()
    for _ in range(2):  # two replays from the same inputs
        st.x.copy_(x0)
        st.residual.copy_(r0)
        st.replay()
        torch.cuda.synchronize()
        got = ([host_bits(t) for t in st.normed], [host_bits(t) for t in st.y], host_bits(st.residual))
        assert_same(got, chain)


def test_persistent_run_pinned_equals_the_kernel_graph(step_data, dev_layers):
    # end to end through pinned host memory, two consecutive tokens: the persistent step
    # and the graph of separate kernels give the same host outputs
    steps = [_decode_step(step_data, dev_layers, m) for m in (False, True)]
    ios = []
    for st in steps:
        io = st.pinned_io()
        st.capture_pinned(io)
        io.x.copy_(st.x.cpu())
        io.residual.copy_(st.residual.cpu())
        io.gate.copy_(st.gate.cpu())
        io.up.copy_(st.up.cpu())
        ios.append(io)
    for _ in range(2):
        for st, io in zip(steps, ios):
            st.run_pinned(io)
            st.stream.synchronize()
        assert torch.equal(ios[0].out_x.view(torch.int16), ios[1].out_x.view(torch.int16))
        assert torch.equal(ios[0].residual.view(torch.int16), ios[1].residual.view(torch.int16))
        for io in ios:  # the next token's input: the output and the new residual
            io.x.copy_(io.out_x)


@pytest.mark.parametrize("n", [1, 3])
def test_persistent_wait_timeout_is_reported(step_data, dev_layers, chain, n):
    # FD_LAUNCH_TEST_WAIT_TIMEOUT: one CTA withholds its first count, every CTA's wait for it
    # runs out on the short limit; layer 0 stays correct, everything after it is NaN, the
    # status is reported once, and the next call is bit-identical again
    import time

    from memory_bound_decode_fd_gb300 import _lib

    lib = _lib.load()
    persistent(step_data, dev_layers[:n])  # the kernel's launch facts, outside the flag
    assert fd.device_status(clear=True) == 0
    flags = lib.fd_get_launch_flags()
    assert lib.fd_set_launch_flags(flags | _lib.FD_LAUNCH_TEST_WAIT_TIMEOUT) == _lib.FD_OK
    try:
        t0 = time.perf_counter()
        normed, ys, res = persistent(step_data, dev_layers[:n])
        elapsed = time.perf_counter() - t0
    finally:
        lib.fd_set_launch_flags(flags)
    assert elapsed < 5.0, elapsed
    n_ref, _, y_ref = chain[0]
    assert np.array_equal(normed[0].reshape(-1), n_ref.reshape(-1))
    assert np.array_equal(ys[0].reshape(-1), y_ref.reshape(-1))
    nan = lambda bits: np.all(np.isnan(bf16_float(bits)))  # noqa: E731
    for l in range(1, n):
        assert nan(normed[l]) and nan(ys[l]), l
    assert nan(res)
    assert fd.device_status(clear=True) & _lib.FD_DEVICE_STATUS_WAIT_TIMEOUT
    assert fd.device_status(clear=True) == 0
    assert_same(persistent(step_data, dev_layers[:n]), chain[:n])
    assert fd.device_status(clear=True) == 0


def bf16_float(bits):
    b = np.asarray(bits).reshape(-1).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def test_layer_table_rejects_misaligned_tensors(cuda_device):
    # the table's pointers are checked on the host (the C ABI cannot read device memory);
    # nothing is launched
    hidden, inter, group = 64, 256, 128
    bf = torch.bfloat16
    base = torch.zeros(inter + 8, dtype=bf, device="cuda")
    layer = {"gate": base[:inter], "up": torch.zeros(inter, dtype=bf, device="cuda"),
             "qweight": torch.zeros((hidden, inter // 8), dtype=torch.int32, device="cuda"),
             "scales": torch.zeros((hidden, inter // group), dtype=bf, device="cuda"),
             "rms_weight": torch.zeros(hidden, dtype=bf, device="cuda")}
    normed = [torch.zeros((1, hidden), dtype=bf, device="cuda")]
    y = [torch.zeros((1, hidden), dtype=bf, device="cuda")]
    assert tuple(fd.step_layer_table([layer], normed, y).shape) == (1, 7)
    layer["gate"] = base[1:inter + 1]  # 2 bytes past an aligned start
    with pytest.raises(ValueError, match="16-byte aligned"):
        fd.step_layer_table([layer], normed, y)


def test_device_status_clean_after_the_persistent_steps(cuda_device):
    assert fd.device_status(clear=True) == 0
