"""The whole path on the GPU against the oracle.

Walk (a5) fed the oracle's own scores: choices bit-exact.  End to end: candidate ids
bit-exact, lse within 1e-5, pair scores within 1e-3, committed tokens bit-identical to the
oracle on every block (a divergence at a float32 tie of the oracle's own scores is listed
in the parity record and still fails these seeded cases)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import lilicorr_oracle as O
from synth import make_workload
from tests.gpu_util import (SCORE_ATOL, assert_no_divergence, check_block, dev_bf16, dev_logits,
                            oracle_block, report_for)

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as m
    return m


# ------------------------------------------------------------------ walk on given scores

def test_walk_golden(lc):
    gd = json.load(open(os.path.join(GOLDEN, "greedy_vs_exact_path.json")))
    sc = np.array([[[float(v) for v in r] for r in p] for p in gd["scores"]], np.float32)
    cid = torch.tensor(gd["cand_id"], dtype=torch.int32).cuda()[None]
    tok, ch, path = lc.greedy_walk(torch.from_numpy(sc).cuda()[None], cid,
                                   torch.tensor([gd["anchor_id"]], dtype=torch.int32).cuda())
    assert ch.cpu().numpy()[0].tolist() == gd["greedy_choice"]
    assert tok.cpu().numpy()[0].tolist() == gd["greedy_tokens"]
    assert path.cpu().numpy()[0].tolist() == gd["greedy_path_score"]


@pytest.mark.parametrize("K", [1, 2, 3, 8, 16, 31, 32])
def test_walk_matches_oracle_on_oracle_scores(lc, K):
    rng = np.random.default_rng(K)
    batch, B = 37, 16
    sc = (np.round(rng.standard_normal((batch, B - 1, K, K)) * 3) / 4).astype(np.float32)  # ties
    sc[:, 0, 1:] = -np.inf
    cid = rng.integers(0, 151936, size=(batch, B - 1, K)).astype(np.int32)
    tok, ch, path = lc.greedy_walk(torch.from_numpy(sc).cuda(), torch.from_numpy(cid).cuda())
    tok, ch, path = tok.cpu().numpy(), ch.cpu().numpy(), path.cpu().numpy()
    for b in range(batch):
        rc, rp, _ = O.greedy_walk(sc[b].astype(np.float64))
        assert ch[b].tolist() == rc.tolist()
        assert np.array_equal(path[b], rp.astype(np.float32))
        assert tok[b, 0] == -1 and tok[b, 1:].tolist() == cid[b, np.arange(B - 1), rc].tolist()


# ------------------------------------------------------------------ end to end

def _gpu_run(lc, wl, weights=None, taps=True, blocks=None):
    w = weights or lc.Weights(wl.dims, wl.weights)
    out = lc.rerank(w, dev_logits(wl), wl.K, slot_hidden=dev_bf16(wl.slot_hidden),
                    target_state=dev_bf16(wl.target_state),
                    anchor_ids=None if wl.anchor_ids is None else torch.from_numpy(wl.anchor_ids).cuda(),
                    taps=taps)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    if weights is None:
        w.close()
    return res


def _label(name, kw):
    return name + "".join(f" {k}={v}" for k, v in sorted(kw.items()))


def _compare(lc, wl, blocks=None, label=None):
    gpu = _gpu_run(lc, wl)
    label = label or wl.name
    report = report_for(label)
    for b in (range(wl.batch) if blocks is None else blocks):
        ref = oracle_block(wl, b)
        check_block(gpu, ref, b, report)
    assert_no_divergence(report, label)
    return gpu, report


SMALL = [  # name, overrides
    ("tiny", {}),
    ("tiny", dict(batch=3, seed=11)),
    ("single", dict(V=4096, batch=3)),
    ("sweep", dict(V=4096, batch=4)),
    ("highconc", dict(V=4096, batch=2, tier="low")),
    ("highconc", dict(V=4096, batch=2, tier="high")),
    ("widepool", dict(V=4096, batch=2)),
    ("single", dict(V=3001, batch=2, B=9)),          # shorter block than B_max, odd V
    ("single", dict(V=4096, batch=2, with_slot_hidden=True)),
    ("single", dict(V=4096, batch=1, with_target=False, with_anchor=False)),
    ("highconc", dict(V=2048, batch=5, K=1)),
    ("single", dict(V=2048, batch=2, B=26)),         # 25 query slots: the largest bias
                                                     # table of the tcgen05 attention
    ("single", dict(V=2048, batch=2, B=27)),         # 26: the mma.sync attention instead
    # lattices of 257..512 tokens: the chunked tcgen05 attention (keys in chunks of 128)
    ("single", dict(V=2048, batch=3, K=20)),         # 300 tokens: 3 chunks, ragged last
    ("single", dict(V=2048, batch=2, K=24, B=12)),   # 264 tokens, 11 slots
    ("widepool", dict(V=2048, batch=2, B=12)),       # 352 tokens at hidden 512
    ("single", dict(V=2048, batch=2, K=32, B=17)),   # 512 tokens: 4 full chunks
    ("single", dict(V=2048, batch=1, K=32, B=18)),   # 544 tokens: the mma.sync attention
    # head dim 32 on the tcgen05 attention (zero-filled 64-wide tiles): two query tiles
    # with the K / V tiles reused, and a 3-slot lattice
    ("single", dict(V=2048, batch=3, heads=8, K=16)),  # hidden 256, 8 heads, 240 tokens
    ("tiny", dict(batch=2, seed=5)),
]


@pytest.mark.parametrize("name,kw", SMALL)
def test_rerank_small(lc, name, kw):
    wl = make_workload(name, **kw)
    gpu, rep = _compare(lc, wl, label="small: " + _label(name, kw))
    if kw.get("K") == 1:      # K = 1 reproduces the per-slot argmax block
        x = wl.logits_f32()
        for b in range(wl.batch):
            assert gpu["tokens"][b, 1:].tolist() == [int(np.argmax(x[b, s])) for s in range(1, wl.B)]


def test_rerank_taps_match_oracle_intermediates(lc):
    wl = make_workload("single", V=4096, batch=2, with_slot_hidden=True)
    gpu = _gpu_run(lc, wl)
    for b in range(wl.batch):
        ref = oracle_block(wl, b)
        for name, atol in (("nodes", 1e-5), ("hidden", 1e-4), ("out_vec", 1e-5), ("in_vec", 1e-5)):
            g = gpu[name][b].reshape(ref[name].shape)
            assert np.abs(g - ref[name]).max() <= atol, (name, np.abs(g - ref[name]).max())
        assert np.abs(gpu["anchor_vec"][b] - ref["anchor_vec"]).max() <= 1e-6


def test_rerank_is_deterministic(lc):
    wl = make_workload("highconc", V=8192, batch=8)
    a = _gpu_run(lc, wl)
    b = _gpu_run(lc, wl)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


def test_permuted_vocabulary_commits_same_tokens(lc):
    """Relabelling the vocabulary (logits columns and embedding rows permuted together)
    relabels the committed tokens and changes nothing else: the path sees a token only
    through its logit and its embedding.  f32 logits, so no two candidates tie and the
    id tie-break never comes into play."""
    wl = make_workload("tiny", batch=3, seed=21)
    gpu_a = _gpu_run(lc, wl, taps=False)
    perm = np.random.default_rng(5).permutation(wl.V)
    wl2 = make_workload("tiny", batch=3, seed=21)
    wl2.logits = np.ascontiguousarray(wl.logits[:, :, perm])
    wl2.weights = dict(wl.weights)
    wl2.weights["embed"] = np.ascontiguousarray(wl.weights["embed"][perm])
    gpu_b = _gpu_run(lc, wl2, taps=False)
    assert np.array_equal(perm[gpu_b["tokens"][:, 1:]], gpu_a["tokens"][:, 1:])
    # the log-partition sums the row in a different order: scores agree to rounding
    assert np.abs(gpu_b["path_score"] - gpu_a["path_score"]).max() <= SCORE_ATOL


@pytest.mark.parametrize("name,kw,nblocks", [
    ("single", {}, 1),
    ("highconc", dict(tier="medium"), 3),
    ("widepool", {}, 3),
    ("sweep", dict(batch=128), 2),
])
def test_rerank_full_size_sampled_blocks(lc, name, kw, nblocks):
    wl = make_workload(name, **kw)
    rng = np.random.default_rng(1)
    blocks = sorted(rng.choice(wl.batch, nblocks, replace=False).tolist())
    _compare(lc, wl, blocks, label="sampled: " + _label(name, kw))


def test_rerank_captures_in_a_cuda_graph(lc):
    """The entry point allocates nothing and never synchronises: one call captures into a
    CUDA graph whose replays reproduce the eager outputs bit for bit."""
    wl = make_workload("highconc", batch=8, tier="medium")
    w = lc.Weights(wl.dims, wl.weights)
    logits = dev_logits(wl)
    tgt = dev_bf16(wl.target_state)
    anc = torch.from_numpy(wl.anchor_ids).cuda()
    B, K = logits.shape[1], wl.K
    ws = w.workspace(logits.shape[0], B, K)
    eager = lc.rerank(w, logits, K, target_state=tgt, anchor_ids=anc, workspace=ws)
    torch.cuda.synchronize()
    out = {"tokens": torch.zeros_like(eager["tokens"]),
           "path_score": torch.zeros_like(eager["path_score"])}
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        lc.rerank(w, logits, K, target_state=tgt, anchor_ids=anc, workspace=ws, out=out,
                  stream=cap)
    for _ in range(2):
        out["tokens"].zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out["tokens"], eager["tokens"])
        assert torch.equal(out["path_score"], eager["path_score"])


def test_attention_rebase_when_far_keys_dominate(lc):
    """Slot-distance biases of +14 for keys eight or more slots ahead make the second key
    half (keys 128-239) dominate the first slots' queries by more than 2^16: the
    tcgen05 attention re-bases those rows on the second half's maximum and rescales the
    first half's partial output.  Encoder output and tokens still match the oracle."""
    wl = make_workload("highconc", V=4096, batch=2, tier="medium")
    Bm = wl.dims["B_max"]
    from synth.inputs import bf16_bits_to_f32, f32_to_bf16_bits
    for l in range(wl.dims["layers"]):
        bits = wl.weights[f"layers.{l}.dist_bias"]
        f = bf16_bits_to_f32(bits).reshape(bits.shape)
        f[:, Bm - 2 + 8:] += 14.0
        wl.weights[f"layers.{l}.dist_bias"] = f32_to_bf16_bits(f).reshape(bits.shape)
    gpu, rep = _compare(lc, wl, label="attention re-base case")
    for b in range(wl.batch):
        ref = oracle_block(wl, b)
        g = gpu["hidden"][b].reshape(ref["hidden"].shape)
        assert np.abs(g - ref["hidden"]).max() <= 1e-4


def test_long_attention_rebase_when_far_chunks_dominate(lc):
    """Wide pool (480 tokens, keys in four chunks of 128): slot-distance biases of +14 for
    keys five or more slots ahead make the later key chunks dominate the first slots'
    queries by more than 2^16, so the chunked attention re-bases those rows on a later
    chunk and rescales the output accumulated so far.  Encoder output and tokens still
    match the oracle."""
    wl = make_workload("widepool", V=2048, batch=2)
    Bm = wl.dims["B_max"]
    from synth.inputs import bf16_bits_to_f32, f32_to_bf16_bits
    for l in range(wl.dims["layers"]):
        bits = wl.weights[f"layers.{l}.dist_bias"]
        f = bf16_bits_to_f32(bits).reshape(bits.shape)
        f[:, Bm - 2 + 5:] += 14.0
        f[:, Bm - 2 + 10:] += 14.0
        wl.weights[f"layers.{l}.dist_bias"] = f32_to_bf16_bits(f).reshape(bits.shape)
    gpu, rep = _compare(lc, wl, label="long attention re-base case")
    for b in range(wl.batch):
        ref = oracle_block(wl, b)
        g = gpu["hidden"][b].reshape(ref["hidden"].shape)
        assert np.abs(g - ref["hidden"]).max() <= 1e-4


@pytest.mark.parametrize("name,kw", [("highconc", dict(V=4096, batch=11)),
                                     ("single", dict(V=3001, batch=3, B=9, with_slot_hidden=True)),
                                     ("tiny", dict(batch=1)),
                                     # full vocabulary, 8 blocks = 120 rows: chunks of
                                     # fewer rows would split the rows' logit pass
                                     ("sweep", dict(batch=8))])
def test_rerank_host_matches_device_entry(lc, name, kw):
    """The host-memory entry point (chunked copies of rows 1..B-1 overlapped with the
    per-chunk reranks) returns exactly what the device entry point returns."""
    wl = make_workload(name, **kw)
    w = lc.Weights(wl.dims, wl.weights)
    dev = _gpu_run(lc, wl, weights=w, taps=False)
    x = torch.from_numpy(wl.logits.view(np.int16)).view(torch.bfloat16) if wl.ldtype == "bf16" \
        else torch.from_numpy(wl.logits)
    pin = lambda t: None if t is None else t.pin_memory()
    tgt = None if wl.target_state is None else torch.from_numpy(wl.target_state.view(np.int16)).view(torch.bfloat16)
    sh = None if wl.slot_hidden is None else torch.from_numpy(wl.slot_hidden.view(np.int16)).view(torch.bfloat16)
    anc = None if wl.anchor_ids is None else torch.from_numpy(wl.anchor_ids)
    for _ in range(2):  # the second call reuses the staging
        tok, ps = lc.rerank_host(w, pin(x.contiguous()), wl.K, target_state=pin(tgt),
                                 slot_hidden=pin(sh), anchor_ids=pin(anc))
        assert np.array_equal(tok.numpy(), dev["tokens"])
        assert np.array_equal(ps.numpy(), dev["path_score"])
    w.close()
