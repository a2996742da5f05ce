"""The CPU oracle over many blocks at once, in a pool of host processes (test infrastructure).

Full-size parity runs check every block of a workload against the float64 oracle, which
takes about a fifth of a second per block on one core.  Blocks are independent, so they
are spread over processes: the workload's arrays are written once to a scratch
directory, every worker maps the logits read-only and widens the weights once, and each
task is one block index.

Workers are started with the "spawn" method, so this works after the parent process has
initialised CUDA, and each worker runs numpy on one thread.  This module imports no
torch and nothing from the CUDA package.
"""
from __future__ import annotations

import json
import multiprocessing as mp
import os
import shutil
import tempfile
from typing import Dict, List, Optional, Sequence

import numpy as np

# what a parity check reads from one oracle block (the large intermediates stay behind)
KEEP = ("cand_id", "cand_logit", "lse", "pair_scores", "tokens", "margin", "path_score",
        "choice")

_STATE: Dict[str, object] = {}


def _init(path: str) -> None:
    from synth import bf16_bits_to_f32
    meta = json.load(open(os.path.join(path, "meta.json")))
    f64 = lambda a: bf16_bits_to_f32(a).reshape(a.shape).astype(np.float64)
    wz = np.load(os.path.join(path, "weights.npz"))
    _STATE["w"] = {k: f64(wz[k]) for k in wz.files}
    _STATE["meta"] = meta
    _STATE["logits"] = np.load(os.path.join(path, "logits.npy"), mmap_mode="r")
    for name in ("target_state", "slot_hidden", "anchor_ids"):
        p = os.path.join(path, name + ".npy")
        a = np.load(p) if os.path.exists(p) else None
        if a is not None and name != "anchor_ids":
            a = f64(a)
        _STATE[name] = a


def _block(b: int) -> Dict[str, np.ndarray]:
    from oracle import lilicorr_oracle as O
    from synth import bf16_bits_to_f32
    meta = _STATE["meta"]
    x = np.asarray(_STATE["logits"][b])
    x = (bf16_bits_to_f32(x).reshape(x.shape) if meta["ldtype"] == "bf16" else x)
    tgt, sh, anc = _STATE["target_state"], _STATE["slot_hidden"], _STATE["anchor_ids"]
    r = O.rerank_block(x.astype(np.float64), meta["K"], _STATE["w"], meta["dims"],
                       None if tgt is None else tgt[b], None if sh is None else sh[b],
                       None if anc is None else int(anc[b]))
    return {k: r[k] for k in KEEP}


def oracle_blocks(wl, blocks: Optional[Sequence[int]] = None,
                  workers: Optional[int] = None) -> List[Dict[str, np.ndarray]]:
    """The oracle's results for the given blocks of synth Workload `wl` (all by default),
    in order, computed by `workers` spawned processes (default: the host's cores)."""
    blocks = list(range(wl.batch) if blocks is None else blocks)
    workers = max(1, min(workers or os.cpu_count() or 1, len(blocks)))
    tmp = tempfile.mkdtemp(prefix="lilicorr_oracle_")
    saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                             "MKL_NUM_THREADS")}
    try:
        np.save(os.path.join(tmp, "logits.npy"), wl.logits)
        np.savez(os.path.join(tmp, "weights.npz"), **wl.weights)
        for name in ("target_state", "slot_hidden", "anchor_ids"):
            a = getattr(wl, name)
            if a is not None:
                np.save(os.path.join(tmp, name + ".npy"), a)
        json.dump({"K": wl.K, "dims": wl.dims, "ldtype": wl.ldtype},
                  open(os.path.join(tmp, "meta.json"), "w"))
        for v in saved:
            os.environ[v] = "1"
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers, initializer=_init, initargs=(tmp,)) as pool:
            return pool.map(_block, blocks, chunksize=max(1, len(blocks) // (4 * workers)))
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
        shutil.rmtree(tmp, ignore_errors=True)
