"""Run one fd kernel a few times on seeded inputs, nothing else (for ncu captures).

    python -m memory_bound_decode_fd_gb300.profile_case gemv --M 1 --K 14336 --N 4096
    python -m memory_bound_decode_fd_gb300.profile_case gemv --M 64 --path tensor
    python -m memory_bound_decode_fd_gb300.profile_case gemv_residual --M 1 --K 14336 --N 4096
    python -m memory_bound_decode_fd_gb300.profile_case rmsnorm --rows 8192 --hidden 4096
    python -m memory_bound_decode_fd_gb300.profile_case gate_up --K 4096 --N 14336
    python -m memory_bound_decode_fd_gb300.profile_case nvfp4 --M 64 --K 4096 --N 6144

Each iteration uses the next of --sets input sets, so that consecutive launches do not
find their weights in L2. Exits 0 after a final synchronize.
"""

from __future__ import annotations

import argparse

import numpy as np
import torch


def _dev(a, device):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def main(argv=None) -> int:
    import memory_bound_decode_fd_gb300 as fd
    from memory_bound_decode_fd_gb300 import build, inputs

    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["gemv", "gemv_residual", "rmsnorm", "gate_up", "nvfp4"])
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--K", type=int, default=14336)
    ap.add_argument("--N", type=int, default=4096, help="rows (gate_up: I, the stacked weight has 2I)")
    ap.add_argument("--group", type=int, default=128)
    ap.add_argument("--rows", type=int, default=8192)
    ap.add_argument("--hidden", type=int, default=4096)
    ap.add_argument("--eps", type=float, default=1e-6)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--sets", type=int, default=2)
    ap.add_argument("--path", choices=sorted(["auto", "cuda_core", "bulk", "tensor"]), default="auto")
    args = ap.parse_args(argv)

    build.build()
    fd.set_gemv_path(args.path)
    dev = torch.device("cuda:0")
    if args.case in ("gemv", "gemv_residual"):
        rng = np.random.default_rng(0)
        d = inputs.gemv_inputs(args.M, args.K, args.N, args.group, rng=rng)
        g, u = _dev(d["gate"], dev), _dev(d["up"], dev)
        sets = [(_dev(inputs.int4_words(rng, args.N, args.K), dev),
                 _dev(inputs.scales_bf16(rng, args.N, args.K, args.group), dev))
                for _ in range(args.sets)]
        out = torch.empty((args.M, args.N), dtype=torch.bfloat16, device=dev)
        res = _dev(inputs.normal_bf16(rng, (args.M, args.N)), dev)
        for i in range(args.iters):
            q, s = sets[i % len(sets)]
            if args.case == "gemv":
                fd.swiglu_w4a16_gemv(g, u, q, s, out=out, group=args.group)
            else:
                fd.swiglu_w4a16_gemv_residual(g, u, q, s, res, out=out, group=args.group)
    elif args.case == "gate_up":
        rng = np.random.default_rng(0)
        x = _dev(inputs.normal_bf16(rng, (args.M, args.K)), dev)
        sets = [(_dev(inputs.int4_words(rng, 2 * args.N, args.K), dev),
                 _dev(inputs.scales_bf16(rng, 2 * args.N, args.K, args.group), dev))
                for _ in range(args.sets)]
        g = torch.empty((args.M, args.N), dtype=torch.bfloat16, device=dev)
        u = torch.empty_like(g)
        for i in range(args.iters):
            q, s = sets[i % len(sets)]
            fd.w4a16_gate_up_gemv(x, q, s, gate_out=g, up_out=u, group=args.group)
    elif args.case == "nvfp4":
        sets = []
        for i in range(args.sets):
            d = inputs.nvfp4_inputs(args.M, args.K, args.N, seed=5 + i)
            sets.append(tuple(torch.from_numpy(np.ascontiguousarray(d[k])).to(dev)
                              for k in ("x", "x_sf", "w", "w_sf")))
        alpha = torch.tensor([1.25], dtype=torch.float32, device=dev)
        out = torch.empty((args.M, args.N), dtype=torch.bfloat16, device=dev)
        for i in range(args.iters):
            x, xs, w, ws = sets[i % len(sets)]
            fd.nvfp4_scaled_mm(x, xs, w, ws, alpha, out=out)
    else:
        sets = []
        for i in range(args.sets):
            d = inputs.rmsnorm_inputs(args.rows, args.hidden, seed=i)
            sets.append((_dev(d["x"], dev), _dev(d["residual"], dev), _dev(d["weight"], dev)))
        y = torch.empty((args.rows, args.hidden), dtype=torch.bfloat16, device=dev)
        h = torch.empty_like(y)
        for i in range(args.iters):
            x, r, w = sets[i % len(sets)]
            fd.add_rmsnorm(x, r, w, args.eps, out=y, residual_out=h)
    torch.cuda.synchronize()
    print("profile_case done", flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
