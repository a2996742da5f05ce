"""Pins of the CPU oracle against things other than itself: closed forms, library
routines (scipy, numpy, torch float64 modules), brute force and hand-worked examples.

Nothing here needs a GPU.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import lilicorr_oracle as O
from synth import make_workload
from tests.conftest import oracle_inputs, weights_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------- bf16

def test_bf16_round_matches_torch_conversion(rng):
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-30, 1e-3, 1.0, 1e3, 1e30)])
    x32 = x.astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(x32.astype(np.float64)), ref)


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 sits halfway between 1 and 1 + 2^-7: even significand is 1.
    assert O.bf16_round(np.array([1 + 2.0 ** -8]))[0] == 1.0
    # 1 + 3*2^-8 sits halfway between 1 + 2^-7 and 1 + 2^-6: even is 1 + 2^-6.
    assert O.bf16_round(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert O.bf16_round(np.array([-(1 + 3 * 2.0 ** -8)]))[0] == -(1 + 2.0 ** -6)
    # just above the halfway point rounds up
    assert O.bf16_round(np.array([1 + 2.0 ** -8 + 2.0 ** -30]))[0] == 1 + 2.0 ** -7
    assert O.bf16_round(np.array([0.0]))[0] == 0.0


# ----------------------------------------------------------------------------- lse

def test_lse_constant_row_closed_form():
    for c, V in [(0.0, 1024), (-3.5, 151936), (12.25, 7)]:
        row = np.full((1, V), c)
        assert abs(O.logsumexp_rows(row)[0] - (c + math.log(V))) < 1e-12


def test_lse_planted_spike_closed_form():
    V = 1024
    row = np.zeros((1, V))
    row[0, 517] = 4.0
    assert abs(O.logsumexp_rows(row)[0] - math.log(math.exp(4.0) + (V - 1))) < 1e-12


def test_lse_matches_scipy_and_shift(rng):
    from scipy.special import logsumexp
    rows = rng.standard_normal((6, 3001)) * 3.0
    rows[2, ::7] = -np.inf
    assert np.allclose(O.logsumexp_rows(rows), logsumexp(rows, axis=1), rtol=0, atol=1e-12)
    assert np.allclose(O.logsumexp_rows(rows + 1000.0), O.logsumexp_rows(rows) + 1000.0,
                       rtol=0, atol=1e-9)


# ----------------------------------------------------------------------------- top-K

def _brute_topk(row, K):
    return sorted(range(len(row)), key=lambda v: (-row[v], v))[:K]


@pytest.mark.parametrize("V,K", [(1, 1), (9, 4), (31, 31), (64, 8), (65, 16), (257, 32)])
def test_topk_brute_force_with_ties(rng, V, K):
    for _ in range(5):
        row = np.round(rng.standard_normal(V) * 2) / 2      # many exact ties
        assert O.topk_rows(row[None], K)[0].tolist() == _brute_topk(row.tolist(), K)


def test_topk_lexsort_cross_check(rng):
    rows = np.round(rng.standard_normal((4, 5000)) * 8) / 8
    for r in rows:
        ref = np.lexsort((np.arange(r.size), -r))[:24]
        assert O.topk_rows(r[None], 24)[0].tolist() == ref.tolist()


def test_topk_all_equal_and_signed_zero():
    assert O.topk_rows(np.full((1, 100), 2.5), 7)[0].tolist() == list(range(7))
    row = np.full(10, -1.0)
    row[6], row[3] = -0.0, 0.0                      # -0.0 == +0.0 is a tie: id order
    assert O.topk_rows(row[None], 2)[0].tolist() == [3, 6]
    row[2] = -np.inf
    assert O.topk_rows(row[None], 10)[0].tolist()[-1] == 2


def test_lm_head_logits_brute_force(rng):
    """The projection against explicit per-element sums of Python floats."""
    h = rng.standard_normal((3, 5))
    w = rng.standard_normal((7, 5))
    got = O.lm_head_logits(h, w)
    for r in range(3):
        for v in range(7):
            assert math.isclose(got[r, v], math.fsum(h[r, d] * w[v, d] for d in range(5)),
                                rel_tol=1e-14, abs_tol=1e-14)


def test_lm_head_topk_lse_identity_matrix_is_the_logit_pass(rng):
    """With the vocabulary matrix the identity (V = D), the logits are the hidden rows
    themselves: the fused pass reduces to the plain top-K and log-partition."""
    h = np.round(rng.standard_normal((4, 40)) * 4) / 4  # ties included
    ids, vals, lse = O.lm_head_topk_lse(h, np.eye(40), 6)
    ref = np.argsort(-h, axis=1, kind="stable")[:, :6]
    assert np.array_equal(ids, ref)
    assert np.array_equal(vals, np.take_along_axis(h, ref, axis=1))
    assert np.allclose(lse, np.log(np.exp(h).sum(axis=1)), rtol=0, atol=1e-12)


def test_logit_pass_ignores_anchor_row(rng):
    blk = rng.standard_normal((5, 300))
    a = O.logit_pass(blk, 3)
    blk2 = blk.copy()
    blk2[0] = 100.0
    b = O.logit_pass(blk2, 3)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    assert a[0].shape == (4, 3) and a[2].shape == (4,)


# ----------------------------------------------------------------------------- features

def test_confidence_features_closed_forms(rng):
    rows = rng.standard_normal((15, 777))
    ids, vals, lse = O.logit_pass(np.vstack([rows[:1], rows]), 6)
    rank = np.tile(np.arange(6), (15, 1))
    f = O.confidence_features(vals, lse, rank, 6)
    # log-probs normalise over the full row
    assert np.allclose(np.exp(rows - lse[:, None]).sum(1), 1.0, atol=1e-12)
    assert np.allclose(f[..., 0], vals - lse[:, None])
    assert np.allclose(f[..., 1], np.exp(f[..., 0]))
    assert np.all(f[:, 0, 2] == 0.0) and np.all(f[..., 2] <= 0)
    assert np.allclose(f[..., 3], rank / 5.0) and f[..., 3].min() == 0 and f[..., 3].max() == 1
    assert np.array_equal(f[..., 4], (rank == 0).astype(float))
    f1 = O.confidence_features(vals[:, :1], lse, rank[:, :1], 1)
    assert np.all(f1[..., 3] == 0.0)


# ----------------------------------------------------------------------------- modules vs torch

def _tiny_weights(seed=5, H=32, nh=2, F=64, E=16, V=50, Bm=16, Km=4, layers=1, gain_jitter=0.2):
    from synth import make_weights
    dims = dict(layers=layers, hidden=H, heads=nh, ffn=F, d_e=E, B_max=Bm, K_max=Km, V=V)
    return dims, weights_f64(make_weights(dims, seed, std=0.2, gain_jitter=gain_jitter))


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a))


def test_conf_mlp_matches_torch_modules(rng):
    dims, w = _tiny_weights()
    H = dims["hidden"]
    feat = rng.standard_normal((7, 3, 5))
    net = torch.nn.Sequential(torch.nn.Linear(5, H), torch.nn.SiLU(), torch.nn.Linear(H, H)).double()
    with torch.no_grad():
        net[0].weight.copy_(_t(w["conf.w1"])); net[0].bias.copy_(_t(w["conf.b1"]))
        net[2].weight.copy_(_t(w["conf.w2"])); net[2].bias.copy_(_t(w["conf.b2"]))
        ref = net(_t(feat)).numpy()
    assert np.allclose(O.conf_mlp(feat, w, mirror=False), ref, atol=1e-12)


def test_node_terms_each_land_in_place(rng):
    dims, w = _tiny_weights(Km=4)
    K, Bm1, H = 4, 5, dims["hidden"]
    zero = {k: np.zeros_like(v) for k, v in w.items()}
    cid = rng.integers(0, dims["V"], size=(Bm1, K))
    val = rng.standard_normal((Bm1, K))
    lse = np.full(Bm1, 3.0)
    rank = np.tile(np.arange(K), (Bm1, 1))
    # embedding term only
    z = dict(zero, embed=w["embed"])
    assert np.array_equal(O.node_vectors(cid, val, lse, rank, K, z, None, False),
                          w["embed"][cid].reshape(-1, H))
    # slot table only: slot s (1-based) reads row s-1
    z = dict(zero, slot_table=w["slot_table"])
    got = O.node_vectors(cid, val, lse, rank, K, z, None, False).reshape(Bm1, K, H)
    assert np.array_equal(got, np.broadcast_to(w["slot_table"][:Bm1, None], got.shape))
    # rank table only, with a permuted rank order
    prank = np.array([rng.permutation(K) for _ in range(Bm1)])
    z = dict(zero, rank_table=w["rank_table"])
    got = O.node_vectors(cid, val, lse, prank, K, z, None, False).reshape(Bm1, K, H)
    assert np.array_equal(got, w["rank_table"][prank])
    # drafter hidden: slot s reads hidden[s]; hidden[0] (anchor) is never read
    hid = rng.standard_normal((Bm1 + 1, H))
    got = O.node_vectors(cid, val, lse, rank, K, zero, hid, False).reshape(Bm1, K, H)
    assert np.array_equal(got, np.broadcast_to(hid[1:, None], got.shape))


def test_rmsnorm_matches_torch(rng):
    x = rng.standard_normal((9, 48)) * 3
    g = rng.standard_normal(48)
    ref = F.rms_norm(_t(x), (48,), _t(g), eps=1e-6).numpy()
    assert np.allclose(O.rmsnorm(x, g), ref, atol=1e-12)


def _torch_mha(w_l, H, nh):
    m = torch.nn.MultiheadAttention(H, nh, bias=True, batch_first=True).double()
    with torch.no_grad():
        m.in_proj_weight.copy_(_t(w_l["in_proj_w"])); m.in_proj_bias.copy_(_t(w_l["in_proj_b"]))
        m.out_proj.weight.copy_(_t(w_l["out_proj_w"])); m.out_proj.bias.copy_(_t(w_l["out_proj_b"]))
    return m


def test_attention_matches_torch_multihead(rng):
    dims, w = _tiny_weights()
    H, nh, K, Bm1 = dims["hidden"], dims["heads"], 3, 6
    lw = O.layer_weights(w, 0)
    slots = np.repeat(np.arange(1, Bm1 + 1), K)
    a = rng.standard_normal((Bm1 * K, H))
    mine = O.mha(a, lw, slots, nh, dims["B_max"], mirror=False) @ lw["out_proj_w"].T + lw["out_proj_b"]
    bias = O.attention_bias(slots, lw["dist_bias"], lw["same_bias"], dims["B_max"])
    m = _torch_mha(lw, H, nh)
    with torch.no_grad():
        ref, _ = m(_t(a)[None], _t(a)[None], _t(a)[None], attn_mask=_t(bias), need_weights=False)
    assert np.allclose(mine, ref[0].numpy(), atol=1e-12)


def test_attention_bias_direction_is_key_minus_query(rng):
    """With a huge bias at slot distance +1 only, each query attends to the next slot's
    tokens: the output of slot s is the mean of slot s+1's values (key minus query)."""
    dims, w = _tiny_weights()
    H, nh, K, Bm1, Bm = dims["hidden"], dims["heads"], 2, 5, dims["B_max"]
    lw = dict(O.layer_weights(w, 0))
    lw["in_proj_w"] = np.zeros_like(lw["in_proj_w"])
    lw["in_proj_w"][2 * H:] = np.eye(H)                  # v = a, q = k = 0
    lw["in_proj_b"] = np.zeros_like(lw["in_proj_b"])
    lw["dist_bias"] = np.zeros_like(lw["dist_bias"])
    lw["dist_bias"][:, (Bm - 2) + 1] = 200.0
    lw["same_bias"] = np.zeros_like(lw["same_bias"])
    slots = np.repeat(np.arange(1, Bm1 + 1), K)
    a = rng.standard_normal((Bm1 * K, H))
    out = O.mha(a, lw, slots, nh, Bm, mirror=False).reshape(Bm1, K, H)
    a3 = a.reshape(Bm1, K, H)
    for s in range(Bm1 - 1):
        assert np.allclose(out[s], a3[s + 1].mean(0)[None], atol=1e-9)


def test_same_slot_bias_adds_to_distance_zero(rng):
    dims, w = _tiny_weights()
    lw = O.layer_weights(w, 0)
    slots = np.repeat(np.arange(1, 4), 2)
    b = O.attention_bias(slots, lw["dist_bias"], lw["same_bias"], dims["B_max"])
    z = O.attention_bias(slots, lw["dist_bias"], np.zeros_like(lw["same_bias"]), dims["B_max"])
    d = b - z
    assert np.allclose(d[:, 0, 1], lw["same_bias"]) and np.allclose(d[:, 0, 2], 0.0)


def test_encoder_layer_matches_torch_composition(rng):
    dims, w = _tiny_weights()
    H, nh, K, Bm1 = dims["hidden"], dims["heads"], 4, 5
    lw = O.layer_weights(w, 0)
    slots = np.repeat(np.arange(1, Bm1 + 1), K)
    x = rng.standard_normal((Bm1 * K, H))
    bias = O.attention_bias(slots, lw["dist_bias"], lw["same_bias"], dims["B_max"])
    m = _torch_mha(lw, H, nh)
    ffn = torch.nn.Sequential(torch.nn.Linear(H, dims["ffn"]), torch.nn.SiLU(),
                              torch.nn.Linear(dims["ffn"], H)).double()
    with torch.no_grad():
        ffn[0].weight.copy_(_t(lw["ffn.w1"])); ffn[0].bias.copy_(_t(lw["ffn.b1"]))
        ffn[2].weight.copy_(_t(lw["ffn.w2"])); ffn[2].bias.copy_(_t(lw["ffn.b2"]))
        xt = _t(x)
        a = F.rms_norm(xt, (H,), _t(lw["norm1"]), eps=1e-6)[None]
        xt = xt + m(a, a, a, attn_mask=_t(bias), need_weights=False)[0][0]
        xt = xt + ffn(F.rms_norm(xt, (H,), _t(lw["norm2"]), eps=1e-6))
    assert np.allclose(O.encoder_layer(x, lw, slots, nh, dims["B_max"], mirror=False),
                       xt.numpy(), atol=1e-12)


def test_encoder_layer_zero_weights_is_identity(rng):
    dims, w = _tiny_weights()
    lw = {k: (v if "norm" in k else np.zeros_like(v)) for k, v in O.layer_weights(w, 0).items()}
    x = rng.standard_normal((12, dims["hidden"]))
    slots = np.repeat(np.arange(1, 4), 4)
    assert np.array_equal(O.encoder_layer(x, lw, slots, dims["heads"], dims["B_max"], True), x)


def test_single_token_attention_is_value_path(rng):
    dims, w = _tiny_weights()
    H = dims["hidden"]
    lw = O.layer_weights(w, 0)
    a = rng.standard_normal((1, H))
    got = O.mha(a, lw, np.array([1]), dims["heads"], dims["B_max"], mirror=False)
    v = a @ lw["in_proj_w"][2 * H:].T + lw["in_proj_b"][2 * H:]
    assert np.allclose(got, v, atol=1e-13)


# ----------------------------------------------------------------------------- fusion, heads, scores

def test_fuse_heads_match_torch(rng):
    dims, w = _tiny_weights()
    H = dims["hidden"]
    h = rng.standard_normal((10, H))
    t = rng.standard_normal(H)
    o, i = O.fuse_heads(h, t, w, mirror=False)
    ht, tt = _t(h), _t(np.broadcast_to(t, h.shape))
    f = F.silu(F.linear(torch.cat([ht, tt, ht * tt], -1), _t(w["fuse.w"]), _t(w["fuse.b"])))
    ro = F.normalize(F.linear(f, _t(w["head_out.w"]), _t(w["head_out.b"])), dim=-1, eps=1e-12)
    ri = F.normalize(F.linear(f, _t(w["head_in.w"]), _t(w["head_in.b"])), dim=-1, eps=1e-12)
    assert np.allclose(o, ro.numpy(), atol=1e-13) and np.allclose(i, ri.numpy(), atol=1e-13)
    assert np.allclose(np.linalg.norm(o, axis=1), 1.0) and np.allclose(np.linalg.norm(i, axis=1), 1.0)
    o0 = O.anchor_out(t, w)
    ra = F.normalize(F.linear(_t(t), _t(w["head_anchor.w"]), _t(w["head_anchor.b"])), dim=0)
    assert np.allclose(o0, ra.numpy(), atol=1e-13)


def test_pair_scores_match_cosine_similarity(rng):
    Bm1, K, E = 5, 3, 8
    o = rng.standard_normal((Bm1 * K, E))
    i = rng.standard_normal((Bm1 * K, E))
    o0 = rng.standard_normal(E)
    on, inn, o0n = O.nrm(o), O.nrm(i), O.nrm(o0)
    sc = O.pair_scores(on, inn, o0n, Bm1, K, sigma=8.0)
    o3, i3 = o.reshape(Bm1, K, E), i.reshape(Bm1, K, E)
    for kk in range(K):
        assert abs(sc[0, 0, kk] - 8 * F.cosine_similarity(_t(o0), _t(i3[0, kk]), dim=0).item()) < 1e-12
    assert np.all(np.isneginf(sc[0, 1:]))
    for s in range(1, Bm1):          # pair s: slot s's out (row s-1) vs slot s+1's in (row s)
        for k in range(K):
            for kk in range(K):
                ref = 8 * F.cosine_similarity(_t(o3[s - 1, k]), _t(i3[s, kk]), dim=0).item()
                assert abs(sc[s, k, kk] - ref) < 1e-12
    assert np.all(np.abs(sc[np.isfinite(sc)]) <= 8.0 + 1e-12)


def test_pair_scores_orthogonal_and_equal_vectors():
    e = np.eye(4)
    o = np.stack([e[0], e[1]])            # slot 1 out vectors (K = 2)
    i = np.stack([e[0], e[1], e[1], e[0]])  # slot 1, slot 2 in vectors
    sc = O.pair_scores(np.vstack([o, o]), i, e[0], 2, 2, sigma=8.0)
    assert sc[0, 0].tolist() == [8.0, 0.0]
    assert sc[1].tolist() == [[0.0, 8.0], [8.0, 0.0]]


# ----------------------------------------------------------------------------- walk

def _lexi_max_path(sc, rank=None):
    """Brute force over all K^(B-1) paths: the maximum under the lexicographic order of
    (z_1, -rank(c_1), z_2, -rank(c_2), ...), i.e. each slot first by its step score, then
    by the lower rank, before any later slot is looked at."""
    Bm1, K, _ = sc.shape
    z = sc.astype(np.float32).astype(np.float64)
    rank = np.tile(np.arange(K), (Bm1, 1)) if rank is None else rank
    best, best_key = None, None
    for path in itertools.product(range(K), repeat=Bm1):
        steps, prev = [], 0
        for s, c in enumerate(path):
            steps.append(z[s, prev, c]); prev = c
        key = tuple(v for s, c in enumerate(path) for v in (steps[s], -rank[s, c]))
        if best_key is None or key > best_key:
            best, best_key = path, key
    return list(best)


@pytest.mark.parametrize("Bm1,K", [(1, 3), (3, 2), (4, 3), (6, 4), (5, 1)])
def test_greedy_is_lexicographic_maximiser(rng, Bm1, K):
    for trial in range(6):
        sc = np.round(rng.standard_normal((Bm1, K, K)) * (2 if trial % 2 else 8)) / 2
        sc[0, 1:] = -np.inf
        choice, path, margin = O.greedy_walk(sc)
        assert choice.tolist() == _lexi_max_path(sc)
        prev = 0
        for s, c in enumerate(choice):
            assert path[s] == sc[s, prev, c]; prev = c


def test_greedy_ties_follow_rank_not_position(rng):
    sc = np.zeros((3, 3, 3)); sc[0, 1:] = -np.inf
    rank = np.array([[2, 0, 1], [1, 2, 0], [0, 1, 2]])
    choice, _, _ = O.greedy_walk(sc, rank)
    assert choice.tolist() == _lexi_max_path(sc, rank) == [1, 2, 0]


def test_exact_path_matches_brute_force(rng):
    for Bm1, K in [(3, 2), (5, 3), (6, 4)]:
        for _ in range(5):
            sc = np.round(rng.standard_normal((Bm1, K, K)) * 4) / 4
            sc[0, 1:] = -np.inf
            z = sc.astype(np.float32).astype(np.float64)
            best = max(sum(z[s, ([0] + list(p))[s], p[s]] for s in range(Bm1))
                       for p in itertools.product(range(K), repeat=Bm1))
            choice, g = O.viterbi(sc)
            prev, tot = 0, 0.0
            for s, c in enumerate(choice):
                tot += z[s, prev, c]; prev = c
            assert g == best and tot == best
            assert g >= O.greedy_walk(sc)[1].sum()


def test_golden_greedy_vs_exact():
    gd = json.load(open(os.path.join(GOLDEN, "greedy_vs_exact_path.json")))
    sc = np.array([[[float(v) for v in r] for r in p] for p in gd["scores"]])
    choice, path, _ = O.greedy_walk(sc)
    assert choice.tolist() == gd["greedy_choice"]
    assert path.tolist() == gd["greedy_path_score"] and path.sum() == gd["greedy_g"]
    cid = np.array(gd["cand_id"])
    toks = [gd["anchor_id"]] + [int(cid[s, c]) for s, c in enumerate(choice)]
    assert toks == gd["greedy_tokens"]
    ex, g = O.viterbi(sc)
    assert ex.tolist() == gd["exact_choice"] and g == gd["exact_g"]


# ----------------------------------------------------------------------------- whole path

def _tiny_workload(**kw):
    return make_workload("tiny", **kw)


def test_k1_reproduces_per_slot_argmax():
    for seed in range(3):
        wl = _tiny_workload(K=1, seed=seed, K_max=4)
        inp = oracle_inputs(wl)
        r = O.rerank(inp["logits"], 1, inp["w"], wl.dims, inp["target"], None, inp["anchor"])
        rows = inp["logits"][0, 1:]
        ref = [int(np.flatnonzero(r_ == r_.max())[0]) for r_ in rows]
        assert r["tokens"][0, 1:].tolist() == ref
        assert r["tokens"][0, 0] == wl.anchor_ids[0]


def test_permutation_invariance_of_candidate_order(rng):
    wl = _tiny_workload(seed=3)
    inp = oracle_inputs(wl)
    blk = inp["logits"][0]
    cid, cval, lse = O.logit_pass(blk, wl.K)
    rank = np.tile(np.arange(wl.K), (cid.shape[0], 1))
    args = (inp["w"], wl.dims, inp["target"][0], None, int(wl.anchor_ids[0]))
    base = O.rerank_candidates(cid, cval, lse, rank, *args)
    for _ in range(4):
        perm = np.array([rng.permutation(wl.K) for _ in range(cid.shape[0])])
        take = lambda a: np.take_along_axis(a, perm, axis=1)
        r = O.rerank_candidates(take(cid), take(cval), lse, take(rank), *args)
        assert np.array_equal(r["tokens"], base["tokens"])
        assert np.allclose(r["path_score"], base["path_score"], atol=1e-5)


def test_mirror_changes_little(rng):
    wl = _tiny_workload(seed=1)
    inp = oracle_inputs(wl)
    a = O.rerank(inp["logits"], wl.K, inp["w"], wl.dims, inp["target"], None, inp["anchor"], mirror=True)
    b = O.rerank(inp["logits"], wl.K, inp["w"], wl.dims, inp["target"], None, inp["anchor"], mirror=False)
    fin = np.isfinite(a["pair_scores"])
    d = np.abs(a["pair_scores"][fin] - b["pair_scores"][fin]).max()
    assert 0 < d < 0.1


# ----------------------------------------------------------------------------- sampled commit

def test_sample_walk_zero_temperature_is_greedy(rng):
    sc = np.round(rng.standard_normal((7, 5, 5)) * 4) / 4
    sc[0, 1:] = -np.inf
    g_choice, g_path, _ = O.greedy_walk(sc)
    choice, path, prop = O.sample_walk(sc, 0.0, np.full(7, 0.5))
    assert choice.tolist() == g_choice.tolist() and np.array_equal(path, g_path)
    assert np.array_equal(prop, np.eye(5)[g_choice])


def test_sample_walk_proposal_is_softmax(rng):
    import scipy.special
    sc = rng.standard_normal((6, 8, 8)) * 3
    sc[0, 1:] = -np.inf
    T = 0.7
    u = rng.random(6)
    choice, path, prop = O.sample_walk(sc, T, u)
    z = sc.astype(np.float32).astype(np.float64)
    prev = np.concatenate([[0], choice[:-1]])
    for s in range(6):
        ref = scipy.special.softmax(z[s, prev[s]] / T)
        assert np.allclose(prop[s], ref, rtol=1e-12, atol=1e-15)
        assert path[s] == z[s, prev[s], choice[s]]


def test_sample_walk_draw_frequencies_match_softmax(rng):
    """Many independent first-slot draws: the histogram follows softmax(z / T) within
    five binomial standard deviations (a reversed CDF, a missing 1/T or an off-by-one
    in the inverse CDF all fail)."""
    import scipy.special
    K, T, N = 6, 1.3, 40000
    sc = np.full((1, K, K), -np.inf)
    sc[0, 0] = np.array([1.0, -0.5, 2.0, 0.25, 2.0, -3.0])
    counts = np.zeros(K)
    for u in rng.random(N):
        c, _, _ = O.sample_walk(sc, T, np.array([u]))
        counts[c[0]] += 1
    p = scipy.special.softmax(sc[0, 0] / T)
    sd = np.sqrt(N * p * (1 - p))
    assert np.all(np.abs(counts - N * p) <= 5 * sd + 1)


def test_sample_walk_inverse_cdf_edges(rng):
    sc = np.full((1, 5, 5), -np.inf)
    sc[0, 0] = np.array([-np.inf, 0.3, -0.2, 0.1, -np.inf])
    assert O.sample_walk(sc, 1.0, np.array([0.0]))[0][0] == 1
    assert O.sample_walk(sc, 1.0, np.array([np.nextafter(np.float32(1), np.float32(0))]))[0][0] == 3
    picks = [O.sample_walk(sc, 1.0, np.array([u]))[0][0] for u in np.linspace(0, 0.999, 200)]
    assert picks == sorted(picks)  # an inverse CDF is monotone in u
    allinf = np.full((1, 3, 3), -np.inf)
    c, _, prop = O.sample_walk(allinf, 1.0, np.array([0.4]))
    assert c[0] == 0 and prop[0].tolist() == [1.0, 0.0, 0.0]


def test_sample_walk_conditions_on_the_previous_draw():
    # slot 1 draws candidate 1 (certain); slot 2 must then use row 1 of pair 1
    sc = np.full((2, 3, 3), -np.inf)
    sc[0, 0] = [-np.inf, 0.0, -np.inf]
    sc[1, 0] = [0.0, -np.inf, -np.inf]
    sc[1, 1] = [-np.inf, -np.inf, 0.0]
    c, _, _ = O.sample_walk(sc, 1.0, np.array([0.5, 0.5]))
    assert c.tolist() == [1, 2]
