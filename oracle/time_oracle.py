"""Time the CPU oracle on a bounded sample of a workload (TEST/BENCH INFRASTRUCTURE).

Run as a module by bench.py in a fresh process whose BLAS/OpenMP threads are pinned, so
the core count it reports is the one it used.  Prints one JSON object.

  python -m oracle.time_oracle --workload highconc --tier medium --blocks 2 \
      --steps 3 --warmup 1
"""
import argparse
import json
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import lilicorr_oracle as O  # noqa: E402
from synth import bf16_bits_to_f32, make_workload  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="highconc")
    ap.add_argument("--tier", default=None)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--blocks", type=int, default=2, help="blocks per step")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=1)
    a = ap.parse_args()

    # Only the sampled blocks are needed: generate the workload once, keep its first rows.
    wl = make_workload(a.workload, tier=a.tier, batch=a.batch)
    f64 = lambda x: None if x is None else bf16_bits_to_f32(x).reshape(x.shape).astype(np.float64)
    w = {k: f64(v) for k, v in wl.weights.items()}
    tgt = f64(wl.target_state)
    nblk = a.blocks * (a.steps + a.warmup)
    idx = [i % wl.batch for i in range(nblk)]
    logits = {i: wl.logits_f32(slice(i, i + 1))[0].astype(np.float64) for i in set(idx)}
    del wl.logits

    def step(k):
        for j in range(a.blocks):
            b = idx[k * a.blocks + j]
            O.rerank_block(logits[b], wl.K, w, wl.dims, tgt[b], None,
                           None if wl.anchor_ids is None else int(wl.anchor_ids[b]))

    for k in range(a.warmup):
        step(k)
    times = []
    for k in range(a.warmup, a.warmup + a.steps):
        t0 = time.perf_counter()
        step(k)
        times.append(time.perf_counter() - t0)
    threads = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                                "MKL_NUM_THREADS")}
    print(json.dumps({"blocks_per_step": a.blocks, "steps": a.steps, "step_s": times,
                      "blocks_per_s": a.blocks * a.steps / sum(times), "threads": threads,
                      "workload": wl.name, "batch": wl.batch}))


if __name__ == "__main__":
    main()
