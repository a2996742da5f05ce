import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case")


def weights_f64(weights):
    """bf16 bit-pattern tensors -> exact float64 arrays (oracle input)."""
    from synth import bf16_bits_to_f32
    return {k: bf16_bits_to_f32(v).reshape(v.shape).astype(np.float64) for k, v in weights.items()}


def oracle_inputs(wl):
    """A synth Workload -> the oracle's float64 inputs."""
    from synth import bf16_bits_to_f32
    f64 = lambda a: None if a is None else bf16_bits_to_f32(a).reshape(a.shape).astype(np.float64)
    logits = wl.logits_f32().astype(np.float64)
    return dict(logits=logits, w=weights_f64(wl.weights), target=f64(wl.target_state),
                hidden=f64(wl.slot_hidden), anchor=wl.anchor_ids)


@pytest.fixture(scope="session")
def rng():
    return np.random.default_rng(1234)


def pytest_sessionfinish(session, exitstatus):
    """Write the GPU parity record (tests/gpu_util.REPORT) when GPU parity tests ran:
    per workload the blocks compared, the smallest oracle decision margin, the largest
    score and lse differences and every token divergence.  Path: $LILICORR_PARITY_REPORT,
    else tests/parity_report.json."""
    gu = sys.modules.get("tests.gpu_util")
    if gu is None or not getattr(gu, "REPORT", None):
        return
    import json
    path = os.environ.get("LILICORR_PARITY_REPORT",
                          os.path.join(ROOT, "tests", "parity_report.json"))
    rep = {}
    for label, r in sorted(gu.REPORT.items()):
        r = dict(r)
        if r.get("min_margin") == float("inf"):
            r["min_margin"] = None
        rep[label] = r
    total = {"blocks": sum(r["blocks"] for r in rep.values()),
             "decisions": sum(r.get("decisions", 0) for r in rep.values()),
             "tie_ambiguous": sum(r.get("tie_ambiguous", 0) for r in rep.values()),
             "pytest_exit_status": int(exitstatus)}
    with open(path, "w") as f:
        json.dump({"total": total, "workloads": rep}, f, indent=1, sort_keys=True)
        f.write("\n")
