"""The whole hot path on the GPU: the 32-layer decode step (add-RMSNorm on [1, 4096],
then the SwiGLU-W4A16 down projection K=14336 N=4096, per layer, seed 3), eagerly and
captured in a CUDA graph as the benchmark runs it, against the oracle's chain."""

import numpy as np
import pytest
import torch

import memory_bound_decode_fd_gb300 as fd
import oracle
from memory_bound_decode_fd_gb300 import inputs
from fd_check import check_add_rmsnorm, check_gemv, dev_bf16, dev_i32, host_bits, stated_bar, bf16_f64

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


@pytest.fixture(scope="module")
def step_data():
    return inputs.decode_step_inputs(layers=32, seed=3)


@pytest.fixture(scope="module")
def oracle_chain(step_data):
    d = step_data
    return oracle.decode_mlp_step(d["x"], d["residual"], d["layers"], EPS, d["group"])


def run_step(d, graph: bool):
    layers = device_layers(d)
    x = dev_bf16(d["x"])
    res = dev_bf16(d["residual"])
    normed = [torch.empty((1, d["hidden"]), dtype=torch.bfloat16, device="cuda") for _ in layers]
    ys = [torch.empty((1, d["hidden"]), dtype=torch.bfloat16, device="cuda") for _ in layers]
    if not graph:
        fd.decode_mlp_step(x, res, layers, EPS, normed=normed, y=ys)
    else:
        x_static, res_static = x.clone(), res.clone()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):  # warm-up outside capture (loads the modules)
            fd.decode_mlp_step(x_static.clone(), res_static.clone(), layers, EPS,
                               normed=normed, y=ys)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fd.decode_mlp_step(x_static, res_static, layers, EPS, normed=normed, y=ys)
        res_static.copy_(res)
        x_static.copy_(x)
        g.replay()
        res = res_static
    torch.cuda.synchronize()
    return [host_bits(t) for t in normed], [host_bits(t) for t in ys], host_bits(res)


@pytest.mark.parametrize("graph", [False, True])
def test_decode_step_32_layers_matches_oracle_chain(cuda_device, step_data, oracle_chain, graph):
    normed, ys, res_final = run_step(step_data, graph)
    record, x_last, res_ref = oracle_chain
    for layer, (h_ref, yn_ref, yn_eager, y_ref) in enumerate(record):
        stated_bar(bf16_f64(normed[layer]), yn_ref)
        stated_bar(bf16_f64(ys[layer]), y_ref)
    # residual after the last layer: bit-exact where the chain's inputs agree bit for bit;
    # the GEMV outputs feeding it differ from the oracle only by rounding, so compare with
    # the stated bar.
    stated_bar(bf16_f64(res_final), bf16_f64(res_ref))


@pytest.fixture(scope="module")
def eager_layers(cuda_device, step_data):
    """The chain run layer by layer through the C ABI, with every layer's own inputs
    kept: (x_l, residual before, normed_l, residual after, y_l) as host bits."""
    d = step_data
    layers = device_layers(d)
    x = dev_bf16(d["x"])
    res = dev_bf16(d["residual"])
    rec = []
    for L in layers:
        x_in, res_in = host_bits(x), host_bits(res)
        normed, _ = fd.add_rmsnorm(x, res, L["rms_weight"], EPS, residual_out=res)
        y = fd.swiglu_w4a16_gemv(L["gate"], L["up"], L["qweight"], L["scales"], group=d["group"])
        torch.cuda.synchronize()
        rec.append((x_in, res_in, host_bits(normed), host_bits(res), host_bits(y)))
        x = y
    return rec


@pytest.fixture(scope="module")
def folded_layers(cuda_device, step_data):
    """The chain with each later layer's add-RMSNorm folded into the previous layer's GEMV
    (swiglu_w4a16_gemv_add_rmsnorm), run call by call with every layer's own inputs kept:
    (x_l, residual before, normed_l, residual after, y_l) as host bits."""
    d = step_data
    layers = device_layers(d)
    x = dev_bf16(d["x"])
    res = dev_bf16(d["residual"])
    scratch = fd.fold_scratch()
    x_in, res_in = host_bits(x), host_bits(res)
    normed, _ = fd.add_rmsnorm(x, res, layers[0]["rms_weight"], EPS, residual_out=res)
    torch.cuda.synchronize()
    rec = []
    normed_bits, res_after = host_bits(normed), host_bits(res)
    for i, L in enumerate(layers):
        if i + 1 < len(layers):
            y, nxt, _ = fd.swiglu_w4a16_gemv_add_rmsnorm(
                L["gate"], L["up"], L["qweight"], L["scales"], res, layers[i + 1]["rms_weight"],
                EPS, scratch, residual_out=res, group=d["group"])
        else:
            y = fd.swiglu_w4a16_gemv(L["gate"], L["up"], L["qweight"], L["scales"], group=d["group"])
            nxt = None
        torch.cuda.synchronize()
        y_bits = host_bits(y)
        rec.append((x_in, res_in, normed_bits, res_after, y_bits))
        if nxt is not None:
            x_in, res_in = y_bits, res_after
            normed_bits, res_after = host_bits(nxt), host_bits(res)
    return rec


def test_folded_decode_step_every_layer_exact_on_its_own_inputs(cuda_device, step_data, folded_layers):
    # The folded chain: every layer's add-RMSNorm (computed in the previous GEMV's tail)
    # checked on its own inputs, every GEMV output within its bound, the links intact.
    d = step_data
    for l, (x_in, res_in, normed, res_out, y) in enumerate(folded_layers):
        L = d["layers"][l]
        check_add_rmsnorm(normed, res_out, x_in, res_in, L["rms_weight"], EPS)
        check_gemv(y, L["gate"], L["up"], L["qweight"], L["scales"], d["group"])
    for a, b in zip(folded_layers, folded_layers[1:]):
        assert np.array_equal(b[0], a[4]) and np.array_equal(b[1], a[3])


def test_decode_step_every_layer_exact_on_its_own_inputs(cuda_device, step_data, eager_layers):
    # Each layer checked against the oracle on the bf16 x and residual the GPU handed it:
    # residual_out bit-exact, the normalised row within the add-RMSNorm element bound, and
    # every GEMV output within the GEMV's derived element-wise bound.
    d = step_data
    for l, (x_in, res_in, normed, res_out, y) in enumerate(eager_layers):
        L = d["layers"][l]
        check_add_rmsnorm(normed, res_out, x_in, res_in, L["rms_weight"], EPS)
        res = check_gemv(y, L["gate"], L["up"], L["qweight"], L["scales"], d["group"])
        assert res["n_checked"] == d["hidden"]
    # the chain's links: layer l + 1 starts from layer l's y and residual
    for a, b in zip(eager_layers, eager_layers[1:]):
        assert np.array_equal(b[0], a[4]) and np.array_equal(b[1], a[3])


@pytest.mark.parametrize("graph", [False, True])
def test_decode_step_equals_the_per_layer_checked_chain(cuda_device, step_data, eager_layers, graph):
    # decode_mlp_step (eager, and captured in a CUDA graph) reproduces, bit for bit, the
    # layer-by-layer chain whose every layer is checked above.
    normed, ys, res_final = run_step(step_data, graph)
    for l, rec in enumerate(eager_layers):
        assert np.array_equal(normed[l], rec[2]) and np.array_equal(ys[l], rec[4])
    assert np.array_equal(res_final, eager_layers[-1][3])


def test_decode_step_graph_and_eager_agree_bitwise(cuda_device, step_data):
    a = run_step(step_data, graph=False)
    b = run_step(step_data, graph=True)
    for ta, tb in zip(a[0] + a[1] + [a[2]], b[0] + b[1] + [b[2]]):
        assert np.array_equal(ta, tb)


def _step_outputs(d, pdl: bool, fold: bool = False):
    from memory_bound_decode_fd_gb300.step import DecodeStep

    layers = device_layers(d)
    step = DecodeStep([{k: L[k] for k in ("rms_weight", "qweight", "scales")} for L in layers],
                      d["hidden"], d["layers"][0]["gate"].shape[1], d["group"], EPS, pdl=pdl,
                      fold=fold)
    step.x.copy_(dev_bf16(d["x"]))
    step.residual.copy_(dev_bf16(d["residual"]))
    for i, L in enumerate(layers):
        step.gate[i].copy_(L["gate"])
        step.up[i].copy_(L["up"])
    step.capture()
    step.replay()
    torch.cuda.synchronize()
    return [host_bits(t) for t in step.normed] + [host_bits(t) for t in step.y] + [host_bits(step.residual)]


@pytest.mark.parametrize("fold", [True, False])
def test_decode_step_graph_equals_the_checked_chain(cuda_device, step_data, eager_layers,
                                                    folded_layers, fold):
    # The captured DecodeStep (programmatic dependent launch) reproduces, bit for bit, the
    # call-by-call chain whose every layer is checked: the folded chain (L + 1 launches) or
    # the plain one (2L launches).
    ref = folded_layers if fold else eager_layers
    out = _step_outputs(step_data, pdl=True, fold=fold)
    L = len(ref)
    for l, rec in enumerate(ref):
        assert np.array_equal(out[l].reshape(-1), rec[2].reshape(-1))
        assert np.array_equal(out[L + l].reshape(-1), rec[4].reshape(-1))
    assert np.array_equal(out[-1].reshape(-1), ref[-1][3].reshape(-1))


def test_decode_step_with_pdl_matches_plain_launches(cuda_device, step_data, oracle_chain):
    # Programmatic dependent launch lets each kernel start while the previous one runs;
    # the results must be identical to ordinary stream-ordered launches, and match the
    # oracle's chain.
    plain = _step_outputs(step_data, pdl=False)
    pdl = _step_outputs(step_data, pdl=True)
    for a, b in zip(plain, pdl):
        assert np.array_equal(a, b)
    record, _, res_ref = oracle_chain
    L = len(record)
    for layer, (h_ref, yn_ref, yn_eager, y_ref) in enumerate(record):
        stated_bar(bf16_f64(pdl[layer]), yn_ref)
        stated_bar(bf16_f64(pdl[L + layer]), y_ref)
    stated_bar(bf16_f64(pdl[-1]), bf16_f64(res_ref))


def test_pdl_flag_roundtrip(cuda_device):
    prev = fd.set_pdl(True)
    assert fd.load_library().fd_get_launch_flags() == 1
    fd.set_pdl(False)
    assert fd.load_library().fd_get_launch_flags() == 0
    fd.set_pdl(prev)
    assert fd.load_library().fd_set_launch_flags(4) == fd.FD_ERR_UNSUPPORTED


@pytest.mark.parametrize("captured", [False, True])
def test_decode_step_pinned_io_matches_call(cuda_device, step_data, oracle_chain, eager_layers, captured):
    # One host->device and one device->host copy per step (StepIO, the end-to-end path the
    # benchmark times) give the same outputs as the four-input __call__ path, for two
    # consecutive tokens (the new residual is the next token's input residual); the first
    # token's host outputs are checked against the oracle.
    from memory_bound_decode_fd_gb300.step import DecodeStep

    d = step_data
    layers = device_layers(d)
    inter = d["layers"][0]["gate"].shape[1]

    def make():
        st = DecodeStep([{k: L[k] for k in ("rms_weight", "qweight", "scales")} for L in layers],
                        d["hidden"], inter, d["group"], EPS, pdl=True)
        return st.capture()

    a, b = make(), make()
    gate = torch.from_numpy(np.stack([L["gate"] for L in d["layers"]]).view(np.int16)).view(torch.bfloat16)
    up = torch.from_numpy(np.stack([L["up"] for L in d["layers"]]).view(np.int16)).view(torch.bfloat16)
    x = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).reshape(1, -1)
    res = torch.from_numpy(d["residual"].view(np.int16)).view(torch.bfloat16).reshape(1, -1)
    pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
    xh, rh, gh, uh = pin(x), pin(res), pin(gate), pin(up)
    ox, orr = torch.empty_like(xh).pin_memory(), torch.empty_like(rh).pin_memory()
    io = b.pinned_io()
    if captured:
        b.capture_pinned(io)
    io.x.copy_(x)
    io.residual.copy_(res)
    io.gate.copy_(gate)
    io.up.copy_(up)
    for token in range(2):
        a(xh, rh, gh, uh, ox, orr)
        a.stream.synchronize()
        b.run_pinned(io)
        b.stream.synchronize()
        assert torch.equal(io.out_x.view(torch.int16), ox.view(torch.int16))
        assert torch.equal(io.residual.view(torch.int16), orr.view(torch.int16))
        if token == 0:
            # the first token's host outputs against the oracle's chain
            out_x = io.out_x.view(torch.int16).numpy().view(np.uint16).copy()
            out_res = io.residual.view(torch.int16).numpy().view(np.uint16).copy()
            record, x_last, res_ref = oracle_chain
            stated_bar(bf16_f64(out_x), record[-1][3])
            stated_bar(bf16_f64(out_res), bf16_f64(res_ref))
            # and bit for bit the chain checked layer by layer above
            assert np.array_equal(out_x.reshape(-1), eager_layers[-1][4].reshape(-1))
            assert np.array_equal(out_res.reshape(-1), eager_layers[-1][3].reshape(-1))
        rh.copy_(orr)  # the next token starts from the new residual on both paths
    assert io.h2d_bytes == (2 * d["hidden"] + 2 * len(layers) * inter) * 2
