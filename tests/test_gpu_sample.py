"""Sampled commit on the GPU against the oracle's sample_walk (pinned on the CPU to
softmax, to draw frequencies and to the greedy walk).  Greedy rows are bit-identical to
the greedy walk; sampled rows draw the same candidates as the oracle from the same
uniforms (both form the weights and running sums in double from the same f32 scores;
a draw may differ only if its uniform lies within 1e-12 of a CDF step, counted as
tie-ambiguous), and publish the same proposal within 1e-6."""
import numpy as np
import pytest
import scipy.special
import torch

from oracle import lilicorr_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as m
    return m


def _scores(rng, batch, B, K, ties=True):
    sc = rng.standard_normal((batch, B - 1, K, K)) * 3
    if ties:
        sc = np.round(sc * 4) / 4
    sc = sc.astype(np.float32)
    sc[:, 0, 1:] = -np.inf
    return sc


def test_greedy_rows_match_the_greedy_walk(lc):
    rng = np.random.default_rng(11)
    batch, B, K = 40, 16, 16
    sc = torch.from_numpy(_scores(rng, batch, B, K)).cuda()
    cid = torch.from_numpy(rng.integers(0, 151936, (batch, B - 1, K)).astype(np.int32)).cuda()
    g = lc.greedy_walk(sc, cid)
    for temp in (None, torch.zeros(batch, device="cuda"), -torch.ones(batch, device="cuda")):
        u = None if temp is None else torch.rand(batch, B - 1, device="cuda")
        tok, ch, path, prop = lc.sample_walk(sc, cid, temp, u)
        assert torch.equal(tok, g[0]) and torch.equal(ch, g[1]) and torch.equal(path, g[2])
        onehot = torch.nn.functional.one_hot(ch.long(), K).float()
        assert torch.equal(prop, onehot)


@pytest.mark.parametrize("K", [1, 2, 5, 16, 32])
def test_sampled_rows_match_the_oracle(lc, K):
    rng = np.random.default_rng(100 + K)
    batch, B = 48, 16
    sc = _scores(rng, batch, B, K, ties=K % 2 == 0)
    temps = np.array([[0.0, 0.5, 1.0, 2.0][b % 4] for b in range(batch)], np.float32)
    u = rng.random((batch, B - 1)).astype(np.float32)
    cid = rng.integers(0, 151936, (batch, B - 1, K)).astype(np.int32)
    tok, ch, path, prop = lc.sample_walk(torch.from_numpy(sc).cuda(), torch.from_numpy(cid).cuda(),
                                         torch.from_numpy(temps).cuda(),
                                         torch.from_numpy(u).cuda())
    tok, ch, path, prop = tok.cpu().numpy(), ch.cpu().numpy(), path.cpu().numpy(), prop.cpu().numpy()
    ambiguous = 0
    for b in range(batch):
        rc, rp, rprop = O.sample_walk(sc[b].astype(np.float64), float(temps[b]), u[b])
        if ch[b].tolist() != rc.tolist():
            s = int(np.flatnonzero(ch[b] != rc)[0])
            prev = 0 if s == 0 else rc[s - 1]
            z = sc[b, s, prev].astype(np.float64)
            w = np.exp((z - z.max()) / temps[b])
            cdf = np.cumsum(w) / w.sum()
            assert np.min(np.abs(cdf - float(u[b, s]))) < 1e-12, f"block {b} slot {s}"
            ambiguous += 1
            continue
        assert np.array_equal(path[b], rp.astype(np.float32))
        assert np.abs(prop[b] - rprop).max() <= 1e-6
        assert tok[b, 1:].tolist() == cid[b, np.arange(B - 1), rc].tolist()
    assert ambiguous == 0


def test_first_slot_draw_frequencies(lc):
    """20,000 blocks share one score row; their first-slot draws follow softmax(z / T)."""
    rng = np.random.default_rng(3)
    batch, B, K, T = 20000, 2, 8, 0.8
    row = (rng.standard_normal(K) * 2).astype(np.float32)
    sc = np.full((batch, 1, K, K), -np.inf, np.float32)
    sc[:, 0, 0] = row
    temps = torch.full((batch,), T, device="cuda")
    u = torch.rand(batch, 1, device="cuda", generator=torch.Generator("cuda").manual_seed(7))
    cid = torch.zeros(batch, 1, K, dtype=torch.int32, device="cuda")
    _, ch, _, prop = lc.sample_walk(torch.from_numpy(sc).cuda(), cid, temps, u)
    counts = np.bincount(ch.cpu().numpy()[:, 0], minlength=K)
    p = scipy.special.softmax(row.astype(np.float64) / T)
    sd = np.sqrt(batch * p * (1 - p))
    assert np.all(np.abs(counts - batch * p) <= 5 * sd + 1)
    assert np.abs(prop[0, 0].cpu().numpy() - p).max() <= 1e-6
