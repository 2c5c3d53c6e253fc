"""A decode step captured once in a CUDA graph and replayed per token.

"Kernel Fusion, torch.compile and CUDA Graphs, Measured", Step 4: in decode the launch
cost exceeds the kernels' own time, so the whole step is recorded once and replayed with
one launch; every replay reads and writes the same addresses, so new inputs are copied
into the captured buffers. ``DecodeStep`` owns those static buffers; the 2 x L kernel
launches inside are the fd C-ABI calls of ``kernels.decode_mlp_step``.
"""

from __future__ import annotations

import torch

from .kernels import decode_mlp_step, set_pdl


class DecodeStep:
    """L layers of (add_rmsnorm on [1, hidden]; SwiGLU-W4A16 down projection).

    ``layers``: per-layer dicts of device tensors ``rms_weight`` [hidden], ``qweight``
    [hidden, inter/8] int32, ``scales`` [hidden, inter/group] bf16 (the model weights,
    resident in HBM). Per-token inputs: x, residual [1, hidden] and per-layer gate, up
    [1, inter], copied into static device buffers on each call.
    """

    def __init__(self, layers, hidden: int, inter: int, group: int, eps: float,
                 device="cuda", stream: torch.cuda.Stream | None = None, pdl: bool = True):
        self.device = torch.device(device)
        self.eps = eps
        self.group = group
        self.stream = stream if stream is not None else torch.cuda.Stream(self.device)
        bf16 = dict(dtype=torch.bfloat16, device=self.device)
        L = len(layers)
        self.x = torch.zeros((1, hidden), **bf16)
        self.residual = torch.zeros((1, hidden), **bf16)
        self.gate = torch.zeros((L, 1, inter), **bf16)
        self.up = torch.zeros((L, 1, inter), **bf16)
        self.normed = [torch.empty((1, hidden), **bf16) for _ in range(L)]
        self.y = [torch.empty((1, hidden), **bf16) for _ in range(L)]
        self.layers = [dict(rms_weight=l["rms_weight"], qweight=l["qweight"], scales=l["scales"],
                            gate=self.gate[i], up=self.up[i]) for i, l in enumerate(layers)]
        self.graph = None
        # Programmatic dependent launch between the step's kernels: each GEMV starts
        # streaming its (constant) weights while the add-RMSNorm before it runs.
        self.pdl = pdl

    def _launch(self):
        return decode_mlp_step(self.x, self.residual, self.layers, self.eps, self.group,
                               normed=self.normed, y=self.y, stream=self.stream)

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

    def __call__(self, x_host, residual_host, gate_host, up_host, out_x_host, out_res_host):
        """End to end on host (ideally pinned) tensors: H2D copies, replay, D2H copies,
        all on the step's stream (asynchronous; synchronize the stream to read results)."""
        with torch.cuda.stream(self.stream):
            self.x.copy_(x_host, non_blocking=True)
            self.residual.copy_(residual_host, non_blocking=True)
            self.gate.copy_(gate_host, non_blocking=True)
            self.up.copy_(up_host, non_blocking=True)
            self.graph.replay()
            out_x_host.copy_(self.y[-1], non_blocking=True)
            out_res_host.copy_(self.residual, non_blocking=True)
