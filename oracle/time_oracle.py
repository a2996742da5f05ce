"""Time the CPU oracle on a bounded sample of a workload (TEST/BENCH INFRASTRUCTURE).

Run as a module by bench.py in a fresh process, so the cores it reports are the ones it
used.  Prints one JSON object.

  one thread:  python -m oracle.time_oracle --workload highconc --tier medium --blocks 2 \
                   --steps 3 --warmup 1
  all cores:   python -m oracle.time_oracle --workload highconc --tier medium --blocks 2 \
                   --procs 16

With --procs N the blocks are spread over N spawned processes (the oracle is serial per
block and blocks are independent), each running numpy on one thread: every process
widens the weights once, reranks one warm-up block, waits at a common barrier and then
reranks --steps blocks, cycling over --blocks blocks of its own.  Throughput = all timed
blocks / (last finish - first start).  The sample is a fresh draw of the same workload
with only the distinct blocks needed (blocks per process x processes), so generating it
stays cheap.
"""
import argparse
import json
import multiprocessing as mp
import os
import shutil
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import lilicorr_oracle as O  # noqa: E402
from synth import bf16_bits_to_f32, make_workload  # noqa: E402

THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _f64(x):
    return None if x is None else bf16_bits_to_f32(x).reshape(x.shape).astype(np.float64)


def _logits_f64(logits, ldtype, b):
    x = np.asarray(logits[b])
    return (bf16_bits_to_f32(x).reshape(x.shape) if ldtype == "bf16" else x).astype(np.float64)


def _one_block(x, meta, w, tgt, anc, b):
    O.rerank_block(x, meta["K"], w, meta["dims"], None if tgt is None else tgt[b], None,
                   None if anc is None else int(anc[b]))


def _proc_main(path, ids, warm, reps, barrier, queue):
    meta = json.load(open(os.path.join(path, "meta.json")))
    wz = np.load(os.path.join(path, "weights.npz"))
    w = {k: _f64(wz[k]) for k in wz.files}
    logits = np.load(os.path.join(path, "logits.npy"), mmap_mode="r")
    tgt = _f64(np.load(os.path.join(path, "target_state.npy"))) \
        if os.path.exists(os.path.join(path, "target_state.npy")) else None
    anc = np.load(os.path.join(path, "anchor_ids.npy")) \
        if os.path.exists(os.path.join(path, "anchor_ids.npy")) else None
    xs = {b: _logits_f64(logits, meta["ldtype"], b) for b in list(ids) + [warm]}
    _one_block(xs[warm], meta, w, tgt, anc, warm)
    barrier.wait()
    t0 = time.time()
    for i in range(reps):
        b = ids[i % len(ids)]
        _one_block(xs[b], meta, w, tgt, anc, b)
    queue.put((t0, time.time(), reps))


def time_all_cores(a):
    """--procs N: N processes, each timing --steps reranks over its own --blocks blocks
    (cycled) after one warm-up block; a step is one block per process."""
    n = a.procs
    wl = make_workload(a.workload, tier=a.tier, batch=n * a.blocks)
    tmp = tempfile.mkdtemp(prefix="lilicorr_oracle_time_")
    saved = {v: os.environ.get(v) for v in THREAD_VARS}
    try:
        np.save(os.path.join(tmp, "logits.npy"), wl.logits)
        np.savez(os.path.join(tmp, "weights.npz"), **wl.weights)
        if wl.target_state is not None:
            np.save(os.path.join(tmp, "target_state.npy"), wl.target_state)
        if wl.anchor_ids is not None:
            np.save(os.path.join(tmp, "anchor_ids.npy"), wl.anchor_ids)
        json.dump({"K": wl.K, "dims": wl.dims, "ldtype": wl.ldtype},
                  open(os.path.join(tmp, "meta.json"), "w"))
        for v in THREAD_VARS:
            os.environ[v] = "1"
        ctx = mp.get_context("spawn")
        barrier, queue = ctx.Barrier(n), ctx.Queue()
        procs = []
        for i in range(n):
            ids = list(range(i * a.blocks, (i + 1) * a.blocks))
            p = ctx.Process(target=_proc_main,
                            args=(tmp, ids, ids[0], a.steps, barrier, queue))
            p.start()
            procs.append(p)
        res = [queue.get() for _ in range(n)]
        for p in procs:
            p.join()
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
        shutil.rmtree(tmp, ignore_errors=True)
    t0 = min(r[0] for r in res)
    t1 = max(r[1] for r in res)
    blocks = sum(r[2] for r in res)
    return {"blocks": blocks, "procs": n, "steps": a.steps, "wall_s": t1 - t0,
            "blocks_per_s": blocks / (t1 - t0), "ms_per_step": 1e3 * (t1 - t0) / a.steps,
            "threads_per_proc": 1, "workload": wl.name, "distinct_blocks": wl.batch}


def time_one_thread(a):
    # Only the sampled blocks are needed: generate the workload once, keep its first rows.
    wl = make_workload(a.workload, tier=a.tier, batch=a.batch)
    w = {k: _f64(v) for k, v in wl.weights.items()}
    tgt = _f64(wl.target_state)
    nblk = a.blocks * (a.steps + a.warmup)
    idx = [i % wl.batch for i in range(nblk)]
    logits = {i: _logits_f64(wl.logits, wl.ldtype, i) for i in set(idx)}
    meta = {"K": wl.K, "dims": wl.dims}
    del wl.logits

    def step(k):
        for j in range(a.blocks):
            b = idx[k * a.blocks + j]
            _one_block(logits[b], meta, w, tgt, wl.anchor_ids, b)

    for k in range(a.warmup):
        step(k)
    times = []
    for k in range(a.warmup, a.warmup + a.steps):
        t0 = time.perf_counter()
        step(k)
        times.append(time.perf_counter() - t0)
    threads = {v: os.environ.get(v) for v in THREAD_VARS}
    return {"blocks_per_step": a.blocks, "steps": a.steps, "step_s": times,
            "blocks_per_s": a.blocks * a.steps / sum(times), "threads": threads,
            "workload": wl.name, "batch": wl.batch}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="highconc")
    ap.add_argument("--tier", default=None)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--blocks", type=int, default=2, help="blocks per step (per process)")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--procs", type=int, default=0, help="processes (0: one thread)")
    a = ap.parse_args()
    res = time_all_cores(a) if a.procs > 0 else time_one_thread(a)
    print(json.dumps(res))


if __name__ == "__main__":
    main()
