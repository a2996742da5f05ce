"""Exact best path (LiLiCorr App. E, Eq. 12) on the GPU against the oracle's dynamic
programme, which is pinned to brute force and to a hand-made lattice in the oracle
tests.  Both sides form path sums in double from the same f32 scores, so choices,
tokens, per-pair scores and the total are compared exactly."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import lilicorr_oracle as O

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as m
    return m


def test_viterbi_golden(lc):
    gd = json.load(open(os.path.join(GOLDEN, "greedy_vs_exact_path.json")))
    sc = np.array([[[float(v) for v in r] for r in p] for p in gd["scores"]], np.float32)
    cid = torch.tensor(gd["cand_id"], dtype=torch.int32).cuda()[None]
    tok, ch, path, tot = lc.viterbi(torch.from_numpy(sc).cuda()[None], cid,
                                    torch.tensor([gd["anchor_id"]], dtype=torch.int32).cuda())
    assert ch.cpu().numpy()[0].tolist() == gd["exact_choice"]
    assert tot.cpu().item() == gd["exact_g"]
    cidn = np.array(gd["cand_id"])
    assert tok.cpu().numpy()[0].tolist() == [gd["anchor_id"]] + [
        int(cidn[s, c]) for s, c in enumerate(gd["exact_choice"])]


@pytest.mark.parametrize("B,K", [(2, 1), (3, 2), (16, 1), (16, 4), (16, 16), (16, 31), (16, 32),
                                 (40, 32), (64, 32)])
def test_viterbi_matches_oracle(lc, B, K):
    rng = np.random.default_rng(1000 * B + K)
    batch = 23
    sc = (np.round(rng.standard_normal((batch, B - 1, K, K)) * 3) / 4).astype(np.float32)  # ties
    sc[:, 0, 1:] = -np.inf
    if K > 2:
        sc[0, 3 % (B - 1)] = -np.inf  # a whole pair without a finite score
    cid = rng.integers(0, 151936, size=(batch, B - 1, K)).astype(np.int32)
    anchor = rng.integers(0, 151936, size=batch).astype(np.int32)
    tok, ch, path, tot = lc.viterbi(torch.from_numpy(sc).cuda(), torch.from_numpy(cid).cuda(),
                                    torch.from_numpy(anchor).cuda())
    tok, ch, path, tot = tok.cpu().numpy(), ch.cpu().numpy(), path.cpu().numpy(), tot.cpu().numpy()
    for b in range(batch):
        rc, g = O.viterbi(sc[b].astype(np.float64))
        assert ch[b].tolist() == rc.tolist(), f"block {b}"
        assert tot[b] == g or (np.isneginf(tot[b]) and np.isneginf(g))
        prev = np.concatenate([[0], rc[:-1]])
        assert np.array_equal(path[b], sc[b, np.arange(B - 1), prev, rc])
        assert tok[b, 0] == anchor[b]
        assert tok[b, 1:].tolist() == cid[b, np.arange(B - 1), rc].tolist()


def test_viterbi_at_least_greedy_on_rerank_scores(lc):
    """On scores from the whole path the exact path's g is at least the greedy path's."""
    rng = np.random.default_rng(5)
    batch, B, K = 64, 16, 16
    sc = rng.standard_normal((batch, B - 1, K, K)).astype(np.float32) * 8
    sc[:, 0, 1:] = -np.inf
    cid = torch.zeros(batch, B - 1, K, dtype=torch.int32, device="cuda")
    t = torch.from_numpy(sc).cuda()
    _, _, gpath = lc.greedy_walk(t, cid)
    _, _, _, tot = lc.viterbi(t, cid)
    g_greedy = gpath.double().sum(1).cpu().numpy()
    assert np.all(tot.cpu().numpy() >= g_greedy - 1e-9)
