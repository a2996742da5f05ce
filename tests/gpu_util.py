"""Helpers shared by the GPU parity tests (imported only by tests marked gpu)."""
import numpy as np
import torch

from synth import bf16_bits_to_f32

# Tolerances (the parity contract): ids and tokens bit-exact; lse abs 1e-5 (f32 result of
# a log-partition over up to 151,936 terms); scores abs 1e-3 (sigma-scaled cosines).
LSE_ATOL = 1e-5
SCORE_ATOL = 1e-3


def dev_logits(wl) -> torch.Tensor:
    if wl.ldtype == "bf16":
        return torch.from_numpy(wl.logits.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(wl.logits).cuda()


def dev_bf16(bits):
    if bits is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def f64(bits):
    return None if bits is None else bf16_bits_to_f32(bits).reshape(bits.shape).astype(np.float64)


def oracle_block(wl, b, mirror=False):
    from oracle import lilicorr_oracle as O
    w = {k: f64(v) for k, v in wl.weights.items()}
    logits = wl.logits_f32(slice(b, b + 1))[0].astype(np.float64)
    return O.rerank_block(logits, wl.K, w, wl.dims,
                          None if wl.target_state is None else f64(wl.target_state)[b],
                          None if wl.slot_hidden is None else f64(wl.slot_hidden)[b],
                          None if wl.anchor_ids is None else int(wl.anchor_ids[b]), mirror)


def check_block(gpu, ref, b, report):
    """Compare one block: ids exact, lse and scores within tolerance, tokens exact or
    tie-ambiguous under the near-tie protocol.  Updates `report`."""
    assert np.array_equal(gpu["cand_id"][b], ref["cand_id"]), f"block {b}: candidate ids differ"
    assert np.array_equal(gpu["cand_logit"][b], ref["cand_logit"].astype(np.float32))
    dl = np.abs(gpu["lse"][b].astype(np.float64) - ref["lse"]).max()
    assert dl <= LSE_ATOL, f"block {b}: |dlse| {dl}"
    ps, rs = gpu["pair_scores"][b].astype(np.float64), ref["pair_scores"]
    fin = np.isfinite(rs)
    assert np.array_equal(np.isfinite(ps), fin)
    ds = np.abs(ps[fin] - rs[fin]).max()
    assert ds <= SCORE_ATOL, f"block {b}: |dscore| {ds}"
    report["max_dlse"] = max(report.get("max_dlse", 0.0), dl)
    report["max_dscore"] = max(report.get("max_dscore", 0.0), ds)
    tg, tr = gpu["tokens"][b], ref["tokens"]
    assert tg[0] == tr[0]
    diff = np.flatnonzero(tg[1:] != tr[1:])
    report["blocks"] = report.get("blocks", 0) + 1
    report["min_margin"] = min(report.get("min_margin", np.inf), float(ref["margin"].min()))
    if diff.size:
        s = int(diff[0])
        margin = float(ref["margin"][s])
        assert margin < 2 * ds, (f"block {b}: token differs at slot {s + 1} with oracle margin "
                                 f"{margin:.3e} >= 2 x max|dscore| {ds:.3e}")
        report["tie_ambiguous"] = report.get("tie_ambiguous", 0) + 1
    else:
        # path scores of an identical path agree within the score tolerance
        assert np.abs(gpu["path_score"][b] - ref["path_score"]).max() <= SCORE_ATOL
