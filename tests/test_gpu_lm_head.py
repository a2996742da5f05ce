"""The drafter's vocabulary projection fused with step a1 (lilicorr_lm_head_topk_lse)
against the oracle.  The GPU logits are f32 sums of exact bf16 products in the tensor
cores' order, so the comparison is: every returned logit within 1e-4 of the float64
logit of its id; the returned ids a valid top-K of the float64 logits up to near-ties
(every id at or above the oracle's K-th value less 1e-4, every id strictly above it
plus 1e-4 returned); values sorted by (value desc, id asc); lse within 1e-5."""
import numpy as np
import pytest
import torch

from oracle import lilicorr_oracle as O
from synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as m
    return m


def _bf16(x):
    bits = f32_to_bf16_bits(np.ascontiguousarray(x, np.float32))
    exact = np.frombuffer((bits.astype(np.uint32) << 16).tobytes(), np.float32).reshape(x.shape)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda(), exact


def _check(cid, cv, lse, L, K):
    rows = L.shape[0]
    srt = -np.sort(-L, axis=1)
    for r in range(rows):
        g = cid[r]
        assert len(set(g.tolist())) == K
        assert np.all(np.abs(cv[r] - L[r, g]) <= TOL), r
        kth = srt[r, K - 1]
        assert np.all(L[r, g] >= kth - TOL), r
        must = np.nonzero(L[r] > kth + TOL)[0]
        assert set(must.tolist()) <= set(g.tolist()), r
        for k in range(K - 1):  # (value desc, id asc) among the returned values
            assert cv[r, k] > cv[r, k + 1] or (cv[r, k] == cv[r, k + 1] and g[k] < g[k + 1])
    assert np.abs(lse - O.logsumexp_rows(L)).max() <= 1e-5


@pytest.mark.parametrize("rows,V,D,K", [
    (60, 10000, 256, 1),
    (60, 10000, 256, 8),
    (60, 10000, 256, 16),
    (60, 10000, 256, 32),
    (5, 300, 64, 5),          # one partial vocabulary tile after a full one
    (300, 151_936, 512, 16),  # full vocabulary, three row tiles
])
def test_lm_head_topk_lse_matches_oracle(lc, rows, V, D, K):
    rng = np.random.default_rng(rows * 7 + V + K)
    h, h_ex = _bf16(rng.standard_normal((rows, D)))
    w, w_ex = _bf16(rng.standard_normal((V, D)) * (1.5 / np.sqrt(D)))
    cid, cv, lse = lc.lm_head_topk_lse(h, w, K)
    torch.cuda.synchronize()
    L = O.lm_head_logits(h_ex, w_ex)
    _check(cid.cpu().numpy(), cv.cpu().numpy(), lse.cpu().numpy(), L, K)


def test_lm_head_planted_winners_and_determinism(lc):
    """Rows whose top logits are planted far above the rest: the returned ids are exactly
    the planted ones, in order, and two calls agree bit for bit."""
    rng = np.random.default_rng(3)
    rows, V, D, K = 40, 5000, 128, 4
    hx = rng.standard_normal((rows, D))
    wx = rng.standard_normal((V, D)) * 0.05
    planted = rng.choice(V, rows * K, replace=False).reshape(rows, K)  # distinct ids
    # each planted vocabulary row aligned with its row's hidden state, decreasing scale
    for r in range(rows):
        for k, v in enumerate(planted[r]):
            wx[v] = hx[r] * (0.5 - 0.1 * k) / np.linalg.norm(hx[r]) ** 2 * 40
    h, h_ex = _bf16(hx)
    w, w_ex = _bf16(wx)
    a = lc.lm_head_topk_lse(h, w, K)
    b = lc.lm_head_topk_lse(h, w, K)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    L = O.lm_head_logits(h_ex, w_ex)
    ids_o = O.topk_rows(L, K)
    assert np.array_equal(a[0].cpu().numpy(), ids_o)
    _check(a[0].cpu().numpy(), a[1].cpu().numpy(), a[2].cpu().numpy(), L, K)
