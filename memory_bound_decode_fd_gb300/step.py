"""A decode step captured once in a CUDA graph and replayed per token.

"Kernel Fusion, torch.compile and CUDA Graphs, Measured", Step 4: in decode the launch
cost exceeds the kernels' own time, so the whole step is recorded once and replayed with
one launch; every replay reads and writes the same addresses, so new inputs are copied
into the captured buffers. ``DecodeStep`` owns those static buffers; the kernel launches
inside (L + 1 with the add-RMSNorm folded into the GEMVs, else 2 x L) are the fd C-ABI
calls of ``kernels.decode_mlp_step``.
"""

from __future__ import annotations

import torch

from .kernels import (add_rmsnorm, copy, copy_rows, decode_mlp_step, decode_mlp_step_persistent,
                      fold_scratch, set_pdl, step_layer_table, step_scratch, swiglu_w4a16_gemv)

# Layers whose gate/up the graph step copies in with x and the residual before its first
# kernel; the rest arrive on a side stream while those layers run (capture_pinned).
_EARLY_LAYERS = 4


class DecodeStep:
    """L layers of (add_rmsnorm on [1, hidden]; SwiGLU-W4A16 down projection).

    ``layers``: per-layer dicts of device tensors ``rms_weight`` [hidden], ``qweight``
    [hidden, inter/8] int32, ``scales`` [hidden, inter/group] bf16 (the model weights,
    resident in HBM). Per-token inputs: x, residual [1, hidden] and per-layer gate, up
    [1, inter], copied into static device buffers on each call.
    """

    def __init__(self, layers, hidden: int, inter: int, group: int, eps: float,
                 device="cuda", stream: torch.cuda.Stream | None = None, pdl: bool = True,
                 fold: bool = False, persistent: bool = False):
        self.device = torch.device(device)
        self.eps = eps
        self.group = group
        self.stream = stream if stream is not None else torch.cuda.Stream(self.device)
        bf16 = dict(dtype=torch.bfloat16, device=self.device)
        L = len(layers)
        if hidden % 8 or inter % 8:
            raise ValueError("hidden and inter must be multiples of 8 (16-byte aligned views)")
        # The per-token tensors share one device block,
        #     [x | residual | gate_0 up_0 | gate_1 up_1 | ... | y_last],
        # so that every prefix of the inputs is contiguous: run_pinned moves the first
        # layers' inputs with one host->device copy and the rest with a second one that
        # overlaps those layers; the outputs are the residual and the last layer's y.
        self.hidden, self.inter, self.n_layers = hidden, inter, L
        self._n_in = 2 * hidden + 2 * L * inter
        self._io = torch.zeros(self._n_in + hidden, **bf16)
        self.x = self._io[0:hidden].view(1, hidden)
        self.residual = self._io[hidden:2 * hidden].view(1, hidden)
        gu = self._io[2 * hidden:self._n_in].view(L, 2, inter)
        self.gate = gu[:, 0:1, :]  # [L, 1, inter], each layer's row contiguous
        self.up = gu[:, 1:2, :]
        self.normed = [torch.empty((1, hidden), **bf16) for _ in range(L)]
        self.y = [torch.empty((1, hidden), **bf16) for _ in range(L - 1)]
        self.y.append(self._io[self._n_in:self._n_in + hidden].view(1, hidden))
        self.layers = [dict(rms_weight=l["rms_weight"], qweight=l["qweight"], scales=l["scales"],
                            gate=self.gate[i], up=self.up[i]) for i, l in enumerate(layers)]
        self.graph = None
        self.io_graph = None  # the step with its pinned-host transfers (capture_pinned)
        self._io_host = None
        # Programmatic dependent launch between the step's kernels: each kernel's CTAs
        # launch and set up while the previous kernel finishes.
        self.pdl = pdl
        # fold=True: each layer's add-RMSNorm after the first folded into the previous
        # layer's GEMV (L + 1 launches instead of 2L), with the fold's scratch buffer. In a
        # CUDA graph with programmatic dependent launch the separate kernels measured faster
        # on GB300 (the fold's last CTA adds about 3 us of dependent L2 round trips per
        # layer, the separate add-RMSNorm about 1.35 us), so it is off by default.
        self.scratch = fold_scratch(self.device) if fold else None
        # persistent=True: the whole step as one cooperative launch (fd_decode_mlp_step), with
        # the same outputs bit for bit; the layer table points at this object's buffers.
        self.persistent = persistent
        if persistent:
            self.table = step_layer_table(self.layers, self.normed, self.y, self.device)
            self.step_sync = step_scratch(L, self.hidden, self.device)

    def _launch(self):
        if self.persistent:
            decode_mlp_step_persistent(self.x, self.residual, self.table, self.eps, self.inter,
                                       self.group, self.step_sync, stream=self.stream)
            return self.y[-1], self.residual
        return decode_mlp_step(self.x, self.residual, self.layers, self.eps, self.group,
                               normed=self.normed, y=self.y, stream=self.stream,
                               scratch=self.scratch)

    def capture(self):
        """Warm up once outside capture (module load, cached launch facts), then record."""
        saved = (self.x.clone(), self.residual.clone())
        self.stream.wait_stream(torch.cuda.current_stream(self.device))
        prev = set_pdl(self.pdl)
        try:
            with torch.cuda.stream(self.stream):
                self._launch()
            self.stream.synchronize()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph, stream=self.stream):
                self._launch()
        finally:
            set_pdl(prev)
        self.x.copy_(saved[0])
        self.residual.copy_(saved[1])
        torch.cuda.synchronize(self.device)
        return self

    def replay(self):
        """One step on the static buffers (inputs already in place)."""
        with torch.cuda.stream(self.stream):
            self.graph.replay()

    def output(self) -> torch.Tensor:
        """x_L, the last layer's down-projection output."""
        return self.y[-1]

    def pinned_io(self) -> "StepIO":
        """Pinned host buffers laid out like the device block, for run_pinned."""
        return StepIO(self)

    def _transfer_in(self, io: "StepIO"):
        copy(self._io[:self._n_in], io.host[:self._n_in], stream=self.stream)

    def _transfer_out(self, io: "StepIO"):
        h = self.hidden
        copy(io.host[h:2 * h], self._io[h:2 * h], stream=self.stream)  # the new residual
        copy(io.host[self._n_in:], self._io[self._n_in:], stream=self.stream)  # y of the last layer

    def _launch_pinned(self, io: "StepIO"):
        """The step with its transfers. The graph of separate kernels copies x, the residual
        and the first _EARLY_LAYERS layers' gate/up before its first kernel, and the other
        layers' gate/up with the copy engine on a side stream, which the first of those
        layers' GEMV waits for; the folded and persistent steps copy all inputs first."""
        L = self.n_layers
        if self.persistent or self.scratch is not None or L <= _EARLY_LAYERS:
            self._transfer_in(io)
            self._launch()
            self._transfer_out(io)
            return
        n0 = 2 * self.hidden + 2 * _EARLY_LAYERS * self.inter
        copy(self._io[:n0], io.host[:n0], stream=self.stream)
        side = self._side_stream
        side.wait_stream(self.stream)
        with torch.cuda.stream(side):
            self._io[n0:self._n_in].copy_(io.host[n0:self._n_in], non_blocking=True)
        late = torch.cuda.Event()
        late.record(side)
        cur = self.x
        for i, layer in enumerate(self.layers):
            add_rmsnorm(cur, self.residual, layer["rms_weight"], self.eps, out=self.normed[i],
                        residual_out=self.residual, stream=self.stream)
            if i == _EARLY_LAYERS:
                self.stream.wait_event(late)
            cur = swiglu_w4a16_gemv(layer["gate"], layer["up"], layer["qweight"], layer["scales"],
                                    out=self.y[i], group=self.group, stream=self.stream)
        self._transfer_out(io)

    def capture_pinned(self, io: "StepIO") -> "DecodeStep":
        """Record the step together with its two transfers to and from `io` (fixed host
        addresses) in one graph, so that run_pinned(io) is a single graph launch and the
        copy kernels overlap the first and last layer's kernels under programmatic
        dependent launch."""
        if self.graph is None:
            self.capture()
        saved = (self.x.clone(), self.residual.clone())
        prev = set_pdl(self.pdl)
        try:
            # load the copy kernel outside the capture (16 bytes into a scratch output)
            with torch.cuda.stream(self.stream):
                copy(self.normed[0].view(-1)[:8], self._io[:8], stream=self.stream)
            self.stream.synchronize()
            self._side_stream = torch.cuda.Stream(self.device)
            self.io_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.io_graph, stream=self.stream):
                self._launch_pinned(io)
        finally:
            set_pdl(prev)
        self._io_host = io.host
        self.x.copy_(saved[0])
        self.residual.copy_(saved[1])
        torch.cuda.synchronize(self.device)
        return self

    def run_pinned(self, io: "StepIO"):
        """End to end: the step's inputs (x, residual, every layer's gate and up) from the
        pinned host block and its outputs (new residual, last layer's y) back to it, on the
        step's stream: after the stream is synchronised, io.residual holds the new residual
        and io.out_x the output."""
        # The transfers are fd_copy kernels, which read and write the pinned host block
        # over NVLink-C2C and overlap the neighbouring kernels (the step measured 321 us end
        # to end with them against 335 us with copy-engine transfers on GB300). The graph of
        # separate kernels copies only the first layers' inputs before its first kernel and
        # the rest with the copy engine behind them (_launch_pinned). With capture_pinned(io)
        # all of it is one graph launch.
        with torch.cuda.stream(self.stream):
            if self.io_graph is not None and io.host is self._io_host:
                self.io_graph.replay()
            else:
                self._transfer_in(io)
                self.graph.replay()
                self._transfer_out(io)

    def __call__(self, x_host, residual_host, gate_host, up_host, out_x_host, out_res_host):
        """End to end on host (ideally pinned) tensors: H2D copies, replay, D2H copies,
        all on the step's stream (asynchronous; synchronize the stream to read results)."""
        L, i = self.n_layers, self.inter
        with torch.cuda.stream(self.stream):
            self.x.copy_(x_host, non_blocking=True)
            self.residual.copy_(residual_host, non_blocking=True)
            # the layers' gate and up rows are interleaved on the device: one strided copy each
            copy_rows(self.gate.view(L, i), gate_host.reshape(L, i), stream=self.stream)
            copy_rows(self.up.view(L, i), up_host.reshape(L, i), stream=self.stream)
            self.graph.replay()
            out_x_host.copy_(self.y[-1], non_blocking=True)
            out_res_host.copy_(self.residual, non_blocking=True)


class StepIO:
    """Pinned host twin of a DecodeStep's device block: write the inputs into ``x``,
    ``gate`` [L, 1, inter], ``up`` and ``residual`` (views), call ``step.run_pinned(io)``,
    synchronise the step's stream, then read ``out_x`` and ``residual`` (the residual view
    is overwritten with the new residual, the next token's input)."""

    def __init__(self, step: DecodeStep):
        h, i, L = step.hidden, step.inter, step.n_layers
        self.host = torch.zeros(step._io.numel(), dtype=torch.bfloat16, pin_memory=True)
        self.x = self.host[0:h].view(1, h)
        self.residual = self.host[h:2 * h].view(1, h)
        gu = self.host[2 * h:step._n_in].view(L, 2, i)
        self.gate = gu[:, 0:1, :]  # [L, 1, inter] views, as on the device
        self.up = gu[:, 1:2, :]
        self.out_x = self.host[step._n_in:step._n_in + h].view(1, h)
        self.h2d_bytes = step._n_in * 2
        self.d2h_bytes = 2 * h * 2
