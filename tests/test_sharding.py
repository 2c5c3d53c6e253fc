"""How the path would shard over P GPUs, checked on the CPU with two gloo ranks and the
oracle (the build itself runs replicas only: one GPU per box, no collective).

* GEMV column-parallel: each rank owns N/P output rows; an all-gather of the rank outputs
  equals the unsharded result exactly.
* GEMV row-parallel: K split group-aligned; the all-reduced float64 partial sums equal the
  unsharded result up to summation order.
* add-RMSNorm with hidden split: the residual add is elementwise (bit-exact per shard); one
  all-reduce of the per-row sums of squares gives every rank the row's rstd.
"""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from memory_bound_decode_fd_gb300 import inputs


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        M, K, N, group = 2, 1024, 256, 128
        d = inputs.gemv_inputs(M, K, N, group, seed=17)
        g, u, q, s = d["gate"], d["up"], d["qweight"], d["scales"]
        full = oracle.swiglu_w4a16_gemv(g, u, q, s, group)

        # column-parallel: rows [lo, hi) of the weights, then an all-gather
        lo, hi = rank * N // world, (rank + 1) * N // world
        part = torch.from_numpy(np.ascontiguousarray(oracle.swiglu_w4a16_gemv(g, u, q[lo:hi], s[lo:hi], group)))
        pieces = [torch.empty_like(part) for _ in range(world)]
        dist.all_gather(pieces, part)
        col = torch.cat(pieces, dim=1).numpy()

        # row-parallel: k in [k0, k1), whole scale groups, then an all-reduce of the sums
        k0, k1 = rank * K // world, (rank + 1) * K // world
        assert k0 % group == 0 and k1 % group == 0
        partial = oracle.swiglu_w4a16_gemv(g[:, k0:k1], u[:, k0:k1], q[:, k0 // 8:k1 // 8],
                                           s[:, k0 // group:k1 // group], group)
        t = torch.from_numpy(np.ascontiguousarray(partial))
        dist.all_reduce(t)
        row = t.numpy()

        # add-RMSNorm with the hidden dimension split
        rows, hidden, eps = 3, 4096, 1e-6
        r = inputs.rmsnorm_inputs(rows, hidden, seed=18)
        h_full, y_full, _ = oracle.add_rmsnorm(r["x"], r["residual"], r["weight"], eps)
        j0, j1 = rank * hidden // world, (rank + 1) * hidden // world
        h_bits, _, _ = oracle.add_rmsnorm(r["x"][:, j0:j1], r["residual"][:, j0:j1],
                                          r["weight"][j0:j1], eps)
        h = oracle.bf16_to_f32(h_bits).astype(np.float64)
        ss = torch.from_numpy(np.ascontiguousarray((h * h).sum(axis=1)))
        dist.all_reduce(ss)
        rstd = 1.0 / np.sqrt(ss.numpy()[:, None] / hidden + eps)
        y = torch.from_numpy(h * rstd * oracle.bf16_to_f32(r["weight"][j0:j1]).astype(np.float64))
        ys = [torch.empty_like(y) for _ in range(world)]
        dist.all_gather(ys, y)
        hs = [torch.empty(h_bits.shape, dtype=torch.int32) for _ in range(world)]
        dist.all_gather(hs, torch.from_numpy(h_bits.astype(np.int32)))

        out[rank] = {
            "col_exact": bool(np.array_equal(col, full)),
            "row_err": float(np.max(np.abs(row - full)) / np.max(np.abs(full))),
            "h_exact": bool(np.array_equal(torch.cat(hs, dim=1).numpy().astype(np.uint16), h_full)),
            "y_err": float(np.max(np.abs(torch.cat(ys, dim=1).numpy() - y_full)) / np.max(np.abs(y_full))),
        }
    finally:
        dist.destroy_process_group()


def test_two_rank_sharding_matches_unsharded_oracle():
    world = 2
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        res = out[rank]
        assert res["col_exact"]
        assert res["row_err"] <= 1e-12
        assert res["h_exact"]
        assert res["y_err"] <= 1e-12
