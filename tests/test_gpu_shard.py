"""Vocabulary-sharded logit pass + packed merge (the tensor-parallel shape, emulated on
one GPU by column slices of one logits tensor): merged ids and logits bit-identical to
the whole-row pass and to the oracle, lse within 1e-5 of the oracle."""
import numpy as np
import pytest
import torch

from oracle import lilicorr_oracle as O
from synth import make_workload
from tests.gpu_util import LSE_ATOL, dev_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as m
    return m


def _sharded(lc, x, K, bounds):
    recs = [lc.topk_lse_shard(x[:, :, a:b], a, K) for a, b in zip(bounds[:-1], bounds[1:])]
    return lc.topk_lse_merge(torch.stack(recs), K)


@pytest.mark.parametrize("bounds", [[0, 75968, 151936], [0, 50001, 100003, 151936],
                                    [0, 7, 19003, 38000, 57001, 76000, 95003, 131071, 151936]])
def test_sharded_equals_whole_row_pass(lc, bounds):
    wl = make_workload("highconc", batch=4, tier="medium")
    x = dev_logits(wl)
    K = wl.K
    cid, cv, lse = lc.topk_lse(x, K)
    mid, mv, mlse = _sharded(lc, x, K, bounds)
    batch, B = x.shape[0], x.shape[1]
    assert torch.equal(mid.view(batch, B - 1, K), cid)
    assert torch.equal(mv.view(batch, B - 1, K), cv)
    assert (mlse.view(batch, B - 1) - lse).abs().max().item() <= 2e-6


@pytest.mark.parametrize("ldtype", ["bf16", "f32"])
def test_sharded_against_oracle_with_ties_and_small_shards(lc, ldtype):
    rng = np.random.default_rng(9)
    batch, B, V, K = 3, 6, 5003, 8
    x = np.round(rng.standard_normal((batch, B, V)) * 2) / 2  # heavy ties
    x[0, 2, rng.choice(V, 40, replace=False)] = 7.0            # ties at the top
    t = torch.from_numpy(x.astype(np.float32)).cuda()
    if ldtype == "bf16":
        t = t.to(torch.bfloat16)
    exact = t.float().cpu().numpy().astype(np.float64)
    bounds = [0, 3, 5, 1001, 2500, 2503, V]  # shards of 3 and 2 columns: padded records
    mid, mv, mlse = _sharded(lc, t, K, bounds)
    mid, mv, mlse = mid.cpu().numpy(), mv.cpu().numpy(), mlse.cpu().numpy()
    for b in range(batch):
        ids, vals, l = O.logit_pass(exact[b], K)
        r = slice(b * (B - 1), (b + 1) * (B - 1))
        assert np.array_equal(mid[r], ids)
        assert np.array_equal(mv[r], vals.astype(np.float32))
        assert np.abs(mlse[r] - l).max() <= LSE_ATOL
