"""Step a1 on the GPU against the oracle: candidate ids and logits bit-exact, lse within
1e-5, over sizes that span several 16 KB stages, ragged tails, unaligned rows, split rows
(few rows -> P segments per row), exact ties and the full vocabulary."""
import numpy as np
import pytest
import torch

from oracle import lilicorr_oracle as O
from synth import f32_to_bf16_bits, make_workload
from tests.gpu_util import LSE_ATOL, dev_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as m
    return m


def _run(lc, x, ldtype, K):
    """x: float32 [batch, B, V] (values representable in ldtype)."""
    if ldtype == "bf16":
        bits = f32_to_bf16_bits(x)
        t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
        exact = np.frombuffer((bits.astype(np.uint32) << 16).tobytes(), np.float32).reshape(x.shape)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
        exact = x.astype(np.float32)
    cid, cv, lse = lc.topk_lse(t, K)
    torch.cuda.synchronize()
    return exact.astype(np.float64), cid.cpu().numpy(), cv.cpu().numpy(), lse.cpu().numpy()


def _check(exact, cid, cv, lse, K):
    for b in range(exact.shape[0]):
        ids, vals, l = O.logit_pass(exact[b], K)
        assert np.array_equal(cid[b], ids), f"block {b}"
        assert np.array_equal(cv[b], vals.astype(np.float32))
        assert np.abs(lse[b] - l).max() <= LSE_ATOL, np.abs(lse[b] - l).max()


CASES = [  # (ldtype, batch, B, V, K)
    ("f32", 1, 16, 1024, 4),
    ("bf16", 2, 16, 1001, 8),          # rows not 16-byte aligned: head and tail elements
    ("bf16", 3, 16, 2 * 8192 + 13, 16),  # several stages + ragged tail
    ("bf16", 3, 16, 2 * 8192 + 13, 17),  # the smallest K whose floor takes 64 thread groups
    ("f32", 4, 16, 40_000, 24),          # 64 groups, f32 rows of several stages
    ("f32", 2, 5, 4097, 32),
    ("bf16", 1, 3, 5, 5),              # K = V, body-free rows
    ("f32", 1, 2, 1, 1),               # V = 1
    ("bf16", 1, 16, 151_936, 8),       # full vocabulary, few rows -> split rows
    ("bf16", 1, 4, 151_936, 32),
    ("f32", 40, 16, 3000, 16),         # many short rows
    # many unsplit rows of varying alignment (each its own CTA)
    ("bf16", 64, 16, 16397, 16),       # 960 unaligned rows of 3 stages
    ("f32", 30, 16, 9001, 32),         # 450 unaligned f32 rows, K = 32
    ("bf16", 200, 16, 700, 8),         # 3,000 one-stage rows: ~10 rows per CTA
]


@pytest.mark.parametrize("ldtype,batch,B,V,K", CASES)
def test_logit_pass_random(lc, ldtype, batch, B, V, K):
    rng = np.random.default_rng(V * 31 + K)
    x = (rng.standard_normal((batch, B, V)) * 2.0).astype(np.float32)
    _check(*_run(lc, x, ldtype, K), K)


@pytest.mark.parametrize("ldtype", ["f32", "bf16"])
def test_logit_pass_exact_ties_and_neg_inf(lc, ldtype):
    rng = np.random.default_rng(7)
    V = 20000
    x = np.full((1, 6, V), 1.25, np.float32)                      # row 1: all equal
    x[0, 2] = np.round(rng.standard_normal(V) * 2) / 2            # row 2: heavy ties
    x[0, 3] = -np.inf
    x[0, 3, rng.choice(V, 5, replace=False)] = 0.5                # row 3: 5 finite values
    x[0, 4] = np.round(rng.standard_normal(V) * 4) / 4
    x[0, 4, rng.choice(V, 300, replace=False)] = 9.0              # row 4: 300-way tie at top
    x[0, 5] = -np.inf
    x[0, 5, V - 1] = -3.0                                         # row 5: single finite value
    _check(*_run(lc, x, ldtype, 32), 32)
    _check(*_run(lc, x, ldtype, 7), 7)


def test_logit_pass_near_tie_generator(lc):
    wl = make_workload("widepool", batch=2, V=40000)
    t = dev_logits(wl)
    cid, cv, lse = lc.topk_lse(t, wl.K)
    torch.cuda.synchronize()
    _check(wl.logits_f32().astype(np.float64), cid.cpu().numpy(), cv.cpu().numpy(),
           lse.cpu().numpy(), wl.K)


def test_logit_pass_full_size_sampled_rows(lc):
    """The high-concurrency workload at full size (batch 256, V 151,936, K 16): every
    output of 48 sampled rows against the oracle, plus a run-to-run bit-identity check."""
    wl = make_workload("highconc", tier="medium")
    t = dev_logits(wl)
    cid, cv, lse = lc.topk_lse(t, wl.K)
    cid2, cv2, lse2 = lc.topk_lse(t, wl.K)
    torch.cuda.synchronize()
    assert torch.equal(cid, cid2) and torch.equal(cv, cv2) and torch.equal(lse, lse2)
    rng = np.random.default_rng(0)
    cid, cv, lse = cid.cpu().numpy(), cv.cpu().numpy(), lse.cpu().numpy()
    for r in rng.choice(wl.batch * (wl.B - 1), 48, replace=False):
        b, s = divmod(int(r), wl.B - 1)
        row = wl.logits_f32(slice(b, b + 1))[0, s + 1].astype(np.float64)[None]
        ids = O.topk_rows(row, wl.K)[0]
        assert np.array_equal(cid[b, s], ids)
        assert np.array_equal(cv[b, s], row[0, ids].astype(np.float32))
        assert abs(lse[b, s] - O.logsumexp_rows(row)[0]) <= LSE_ATOL
