"""Times the CPU oracle, as it stands, on each workload configuration: single-threaded
and on all cores (numpy's BLAS threads; everything else in the oracle is plain numpy),
median of three runs. Test infrastructure like the rest of ``oracle/``.

    python -m oracle.time_configs            # prints one JSON line per config and thread count

Each measurement runs in a fresh subprocess so that the BLAS thread count is set before
numpy loads. The 32-layer decode step is timed on a two-layer sample and scaled by 16.
"""

from __future__ import annotations

import json
import os
import subprocess
import sys

CONFIGS = ["gemv_small", "rmsnorm_big", "gemv_94mb", "decode_step", "batched_m64"]


def _measure(name: str) -> dict:
    import time

    import numpy as np

    import oracle
    from memory_bound_decode_fd_gb300 import inputs

    def median3(fn):
        times = []
        for _ in range(3):
            t0 = time.perf_counter()
            fn()
            times.append(time.perf_counter() - t0)
        return float(np.median(times))

    if name in ("gemv_small", "gemv_94mb"):
        spec = inputs.WORKLOADS[name]
        d = inputs.gemv_inputs(spec["M"], spec["K"], spec["N"], spec["group"], seed=spec["seed"])
        s = median3(lambda: oracle.swiglu_w4a16_gemv(d["gate"], d["up"], d["qweight"], d["scales"], spec["group"]))
        return {"seconds_per_call": s, "sample": "one call"}
    if name == "rmsnorm_big":
        spec = inputs.WORKLOADS[name]
        d = inputs.rmsnorm_inputs(spec["rows"], spec["hidden"], seed=spec["seed"])
        s = median3(lambda: oracle.add_rmsnorm(d["x"], d["residual"], d["weight"], spec["eps"]))
        return {"seconds_per_call": s, "sample": "one call"}
    if name == "decode_step":
        d = inputs.decode_step_inputs(layers=32, seed=3)
        two = d["layers"][:2]
        s = median3(lambda: oracle.decode_mlp_step(d["x"], d["residual"], two, 1e-5, d["group"]))
        return {"seconds_per_call": 16 * s, "sample": "2 of 32 layers, scaled by 16"}
    if name == "batched_m64":
        b = inputs.batched_inputs()
        g, r = b["gemv"], b["rmsnorm"]
        eps = inputs.WORKLOADS[name]["eps"]
        s = median3(lambda: (oracle.swiglu_w4a16_gemv(g["gate"], g["up"], g["qweight"], g["scales"], g["group"]),
                             oracle.add_rmsnorm(r["x"], r["residual"], r["weight"], eps)))
        return {"seconds_per_call": s, "sample": "GEMV M=64 + add-RMSNorm 64x4096, one call each"}
    raise ValueError(name)


def main() -> int:
    if len(sys.argv) == 3 and sys.argv[1] == "--one":
        print(json.dumps(_measure(sys.argv[2])), flush=True)
        return 0
    cores = os.cpu_count() or 1
    for name in CONFIGS:
        for threads in (1, cores):
            env = dict(os.environ)
            for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
                env[v] = str(threads)
            out = subprocess.run([sys.executable, "-m", "oracle.time_configs", "--one", name],
                                 capture_output=True, text=True, env=env, check=True)
            r = json.loads(out.stdout.strip().splitlines()[-1])
            r.update({"config": name, "threads": threads})
            print(json.dumps(r), flush=True)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
