"""Several host threads calling the library at once.

The library keeps per-device launch state (kernel shared-memory limits, SM counts) behind
one mutex and its error message per thread; everything else a call touches is the
caller's: workspace, outputs and stream.  Two threads, each with its own workspace and
stream, rerank different workloads at the same time (ctypes releases the interpreter
lock during the call) and must get exactly what one thread gets alone.
"""
import threading

import numpy as np
import pytest
import torch

from synth import make_workload
from tests.gpu_util import dev_bf16, dev_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as m
    return m


def _inputs(lc, wl):
    w = lc.Weights(wl.dims, wl.weights)
    return dict(w=w, logits=dev_logits(wl), tgt=dev_bf16(wl.target_state),
                anc=torch.from_numpy(wl.anchor_ids).cuda(),
                ws=w.workspace(wl.batch, wl.B, wl.K), K=wl.K)


def _call(lc, a, stream, reps=1):
    out = None
    for _ in range(reps):
        out = lc.rerank(a["w"], a["logits"], a["K"], target_state=a["tgt"], anchor_ids=a["anc"],
                        workspace=a["ws"], taps=("pair_scores", "lse"), stream=stream)
    stream.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_two_host_threads_match_one(lc):
    wls = [make_workload("highconc", V=8192, batch=16, tier="low"),
           make_workload("widepool", V=4096, batch=4)]
    args = [_inputs(lc, wl) for wl in wls]
    alone = [_call(lc, a, torch.cuda.Stream()) for a in args]
    got = [None, None]
    errs = []

    def run(i):
        try:
            got[i] = _call(lc, args[i], torch.cuda.Stream(), reps=5)
        except Exception as e:  # reported below
            errs.append(e)

    ts = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    for a, g in zip(alone, got):
        for k in a:
            assert np.array_equal(a[k], g[k]), k
    for a in args:
        a["w"].close()
