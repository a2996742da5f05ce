"""CPU oracle of the LiLiCorr draft-time rerank path (float64, numpy).

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline
leg may import this module.  The product path never calls it; it shares no code with
the CUDA library (the seeded generators in synth/ are the only common inputs).

Sources ("LiLiCorr: Lightweight Likelihood Correlation of Parallel Drafts for
Speculative Decoding", cited as LiLiCorr; "[Spec] Add LiLiCorr: a candidate-lattice
reranker for DFlash drafts", cited as the serving PR):

  * candidate retention, node = sum of four equal-width terms ... LiLiCorr Sec. 3.2
  * node terms, confidence scalars, transformer, fusion, heads ... LiLiCorr App. A
  * matching score phi = sigma * cos(o_{s,k}, i_{s+1,k'})   ..... LiLiCorr Sec. 3.2, Eq. 1
  * sigma = 8.0, B = 16, two layers ............................ LiLiCorr App. A, Table 4
  * greedy commit c_s = argmax_k phi(s-1, c_{s-1}, k) .......... LiLiCorr Sec. 3.5, Eq. 8
  * path score g(c) and its exact maximiser (Viterbi) ......... LiLiCorr App. E, Eq. 12
  * sampled commit from softmax(z_s / T), proposal published .. serving PR, "Sampling the
                                                                 committed path"; LiLiCorr Eq. 2
  * exact top-k + full-vocabulary log-partition, argmax ties
    to the lower index ........................................ serving PR, "Why the custom kernels"
  * attention parameter layout of nn.MultiheadAttention ........ serving PR, "Design notes" 3

Every step is computed in float64 from exactly widened inputs.  Readings where the
pages leave a step open (each listed in the design notes of the repository):

  R-anchor   row 0 of logits[b] is the anchor position; it is not read.
  R-topk     candidates ordered by (logit desc, token id asc); rank k = position.
  R-lse      natural log, temperature 1, over all V logits of the row.
  R-feat     five scalars: lp = l - lse, p = exp(lp), gap = lp - lp(top-1) <= 0,
             r = (k-1)/(K-1) (0 when K = 1), top = [k == 1].
  R-conf     two-layer network = Linear(5 -> H), SiLU, Linear(H -> H), with biases.
  R-embed    the embedding "projected down" is one pre-projected table E[V, H].
  R-hidden   drafter hidden and target state enter already at width H; absent = 0.
  R-enc      pre-norm blocks: x += Wo MHA(RMSNorm(x)) + bo; x += W2 SiLU(W1 RMSNorm(x)
             + b1) + b2.  RMSNorm with gain, eps 1e-6.  No final norm.
  R-bias     per layer and head: dist_bias[h, slot_j - slot_i + B_max - 2] plus
             same_bias[h] when slot_i == slot_j, added to q.k / sqrt(dh).
  R-fuse     f = SiLU(Wf [h; t; h*t] + bf); o = nrm(Wout f + bout); i = nrm(Win f + bin);
             o_0 = nrm(Wa t + ba); nrm(v) = v / max(||v||, 1e-12).
  R-score    z_s[k] = phi(s-1, c_{s-1}, k); the draft log-prob is not added to z.
  R-argmax   the argmax over scores is taken on scores rounded to float32 (the
             precision the kernels decide in); ties go to the lowest rank.
  R-sample   the sampled commit draws by inverse CDF from caller-supplied uniforms, with
             weights and their running sums in float64 over the float32 scores, in rank
             order (see sample_walk).

Precision: the default (mirror=False) is plain float64 math at every step, the
definition the CUDA path is held to.  mirror=True (or a set of point names) rounds to
bf16, round-to-nearest-even, at the points where a plain-bf16 tensor-core path would
round its operands; it is a diagnostic for studying such paths, not the parity default:
  M1 confidence-MLP hidden   M2 RMSNorm outputs       M3 q, k, v
  M4 attention probabilities M5 attention output      M6 FFN hidden
  M7 fusion inputs h, t, h*t M8 fusion output f
"""
from __future__ import annotations

import math
from typing import Dict, Optional

import numpy as np

SIGMA = 8.0          # cosine scale, LiLiCorr Table 4
RMS_EPS = 1e-6       # RMSNorm epsilon (reading R-enc)
NRM_EPS = 1e-12      # floor of the norm in nrm() (reading R-fuse)


# ---------------------------------------------------------------------------------
# bf16 rounding (the mirror)
# ---------------------------------------------------------------------------------

def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even; return float64.

    bf16 keeps 8 significant bits (1 implicit + 7 stored) and float32's exponent range.
    Written from that definition: x = m * 2^e with 0.5 <= |m| < 1, so m * 2^8 rounded
    to an integer (half to even) is the 8-bit significand.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    # below float32's smallest normal the significand loses bits like float32 does
    e_min = -125  # frexp exponent of 2^-126
    shift = np.where(e < e_min, 8 - (e_min - e), 8)
    r = np.ldexp(np.rint(np.ldexp(m, shift)), e - shift)
    return np.where(np.isfinite(x), r, x)


MIRROR_POINTS = frozenset({"M1", "M2", "M3", "M4", "M5", "M6", "M7", "M8"})


def _maybe(x: np.ndarray, mirror, point: str) -> np.ndarray:
    """Round to bf16 at mirror point `point` when mirror is True or names that point."""
    on = (point in mirror) if isinstance(mirror, (set, frozenset)) else bool(mirror)
    return bf16_round(x) if on else x


# ---------------------------------------------------------------------------------
# a1. fused logit pass: full-vocabulary log-partition + top-K
# ---------------------------------------------------------------------------------

def logsumexp_rows(rows: np.ndarray) -> np.ndarray:
    """log sum_v exp(l_v) per row (serving PR, "Why the custom kernels": the head needs
    log-probs normalised over the whole vocabulary).  Rows hold at least one finite
    value and no NaN."""
    rows = np.asarray(rows, dtype=np.float64)
    m = rows.max(axis=1)
    return m + np.log(np.exp(rows - m[:, None]).sum(axis=1))


def topk_rows(rows: np.ndarray, K: int) -> np.ndarray:
    """Ids of the K largest logits per row, by (value desc, id asc) (reading R-topk).

    A stable sort of -l keeps equal values in ascending id order."""
    rows = np.asarray(rows, dtype=np.float64)
    return np.argsort(-rows, axis=1, kind="stable")[:, :K].astype(np.int64)


def logit_pass(block_logits: np.ndarray, K: int):
    """Rows 1..B-1 of one block's logits [B, V] -> (cand_id [B-1,K], cand_logit, lse).

    LiLiCorr Sec. 3.2 (top-K retention) and App. A (log-prob under the full vocabulary);
    row 0 is the anchor and is not read (reading R-anchor)."""
    rows = np.asarray(block_logits[1:], dtype=np.float64)
    ids = topk_rows(rows, K)
    vals = np.take_along_axis(rows, ids, axis=1)
    return ids, vals, logsumexp_rows(rows)


def lm_head_logits(hidden: np.ndarray, w_lm: np.ndarray) -> np.ndarray:
    """logit[r, v] = sum_d hidden[r, d] * w_lm[v, d] in float64: the drafter's vocabulary
    projection, the stage before the logit pass (LiLiCorr Table 3, "LM-head projection";
    the serving PR's follow-ons fuse it with the top-k / log-partition pass)."""
    return np.asarray(hidden, np.float64) @ np.asarray(w_lm, np.float64).T


def lm_head_topk_lse(hidden: np.ndarray, w_lm: np.ndarray, K: int):
    """The fused projection + a1 on rows of drafter hidden states [rows, D] with the
    vocabulary matrix [V, D]: (cand_id [rows, K], cand_logit [rows, K], lse [rows]) of the
    projected logits, ordered as in reading R-topk."""
    rows = lm_head_logits(hidden, w_lm)
    ids = topk_rows(rows, K)
    return ids, np.take_along_axis(rows, ids, axis=1), logsumexp_rows(rows)


# ---------------------------------------------------------------------------------
# a2. node build (LiLiCorr Sec. 3.2 and App. A "Architecture")
# ---------------------------------------------------------------------------------

def confidence_features(cand_logit: np.ndarray, lse: np.ndarray, rank: np.ndarray,
                        K: int) -> np.ndarray:
    """Five scalars per candidate [B-1, K, 5] (reading R-feat).

    cand_logit [B-1, K], lse [B-1], rank [B-1, K] (0-based).  The slot's most likely
    token is its rank-0 candidate."""
    lp = cand_logit - lse[:, None]
    top_col = np.argmin(rank, axis=1)                   # position of rank 0 per slot
    lp_top = lp[np.arange(lp.shape[0]), top_col]
    gap = lp - lp_top[:, None]
    r = rank / (K - 1) if K > 1 else np.zeros_like(lp)
    top = (rank == 0).astype(np.float64)
    return np.stack([lp, np.exp(lp), gap, r, top], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def conf_mlp(feat: np.ndarray, w: Dict[str, np.ndarray], mirror: bool) -> np.ndarray:
    """Two-layer network over the five scalars (reading R-conf); [..., 5] -> [..., H]."""
    u = silu(feat @ w["conf.w1"].T + w["conf.b1"])
    u = _maybe(u, mirror, "M1")
    return u @ w["conf.w2"].T + w["conf.b2"]


def node_vectors(cand_id: np.ndarray, cand_logit: np.ndarray, lse: np.ndarray,
                 rank: np.ndarray, K: int, w: Dict[str, np.ndarray],
                 slot_hidden: Optional[np.ndarray], mirror: bool) -> np.ndarray:
    """x[s, k] = E[c] + hidden_s + conf(c) + slot_table[s-1] + rank_table[rank]
    (LiLiCorr Sec. 3.2, "formed by summing four terms of equal width", App. A).

    Returns the lattice [(B-1)*K, H] in slot-major order."""
    Bm1 = cand_id.shape[0]
    H = w["embed"].shape[1]
    feat = confidence_features(cand_logit, lse, rank, K)
    x = w["embed"][cand_id]                                        # [B-1, K, H]
    if slot_hidden is not None:
        x = x + slot_hidden[1:Bm1 + 1, None, :]
    x = x + conf_mlp(feat, w, mirror)
    x = x + w["slot_table"][:Bm1][:, None, :]
    x = x + w["rank_table"][rank]
    return x.reshape(Bm1 * K, H)


# ---------------------------------------------------------------------------------
# a3. lattice encoder (LiLiCorr App. A: two bidirectional layers, RMSNorm, SiLU,
# slot-distance and same-slot attention biases)
# ---------------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float = RMS_EPS) -> np.ndarray:
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def attention_bias(slots: np.ndarray, dist_bias: np.ndarray, same_bias: np.ndarray,
                   B_max: int) -> np.ndarray:
    """[nh, S, S] additive logits bias (reading R-bias)."""
    d = slots[None, :] - slots[:, None]                 # slot_j - slot_i
    bias = dist_bias[:, d + (B_max - 2)]                # [nh, S, S]
    same = (d == 0).astype(np.float64)
    return bias + same_bias[:, None, None] * same[None]


def mha(a: np.ndarray, lw: Dict[str, np.ndarray], slots: np.ndarray, nh: int,
        B_max: int, mirror: bool) -> np.ndarray:
    """Multi-head self-attention over the whole lattice with nn.MultiheadAttention's
    packed in_proj [3H, H] layout.  a: the normed input [S, H] -> [S, H] (before
    out_proj)."""
    S, H = a.shape
    dh = H // nh
    qkv = a @ lw["in_proj_w"].T + lw["in_proj_b"]
    qkv = _maybe(qkv, mirror, "M3")
    q, k, v = qkv[:, :H], qkv[:, H:2 * H], qkv[:, 2 * H:]
    bias = attention_bias(slots, lw["dist_bias"], lw["same_bias"], B_max)
    out = np.empty((S, H))
    for h in range(nh):
        sl = slice(h * dh, (h + 1) * dh)
        logits = (q[:, sl] @ k[:, sl].T) / math.sqrt(dh) + bias[h]
        logits = logits - logits.max(axis=1, keepdims=True)
        p = np.exp(logits)
        p = p / p.sum(axis=1, keepdims=True)
        p = _maybe(p, mirror, "M4")
        out[:, sl] = p @ v[:, sl]
    return out


def encoder_layer(x: np.ndarray, lw: Dict[str, np.ndarray], slots: np.ndarray, nh: int,
                  B_max: int, mirror: bool, eps: float = RMS_EPS) -> np.ndarray:
    """One pre-norm transformer layer (reading R-enc)."""
    a = _maybe(rmsnorm(x, lw["norm1"], eps), mirror, "M2")
    att = _maybe(mha(a, lw, slots, nh, B_max, mirror), mirror, "M5")
    x = x + att @ lw["out_proj_w"].T + lw["out_proj_b"]
    a = _maybe(rmsnorm(x, lw["norm2"], eps), mirror, "M2")
    u = _maybe(silu(a @ lw["ffn.w1"].T + lw["ffn.b1"]), mirror, "M6")
    return x + u @ lw["ffn.w2"].T + lw["ffn.b2"]


def layer_weights(w: Dict[str, np.ndarray], l: int) -> Dict[str, np.ndarray]:
    p = f"layers.{l}."
    return {k[len(p):]: v for k, v in w.items() if k.startswith(p)}


# ---------------------------------------------------------------------------------
# a4. target fusion, heads, matching scores (LiLiCorr Sec. 3.2 Eq. 1, App. A)
# ---------------------------------------------------------------------------------

def nrm(v: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(v * v, axis=-1, keepdims=True))
    return v / np.maximum(n, NRM_EPS)


def fuse_heads(h: np.ndarray, t: np.ndarray, w: Dict[str, np.ndarray], mirror: bool):
    """Per candidate: f = SiLU(Wf [h; t; h*t] + bf); o, i = unit-normed heads."""
    tt = np.broadcast_to(t, h.shape)
    cat = np.concatenate([_maybe(h, mirror, "M7"), _maybe(tt, mirror, "M7"),
                          _maybe(h * tt, mirror, "M7")], axis=-1)
    f = _maybe(silu(cat @ w["fuse.w"].T + w["fuse.b"]), mirror, "M8")
    o = nrm(f @ w["head_out.w"].T + w["head_out.b"])
    i = nrm(f @ w["head_in.w"].T + w["head_in.b"])
    return o, i


def anchor_out(t: np.ndarray, w: Dict[str, np.ndarray]) -> np.ndarray:
    """o_0 = nrm(Wa t + ba): the anchor's single out vector (LiLiCorr Sec. 3.2)."""
    return nrm(t @ w["head_anchor.w"].T + w["head_anchor.b"])


def pair_scores(o: np.ndarray, i: np.ndarray, o0: np.ndarray, Bm1: int, K: int,
                sigma: float = SIGMA) -> np.ndarray:
    """phi laid out [B-1, K, K]: entry [s, k, k'] = phi(s, k, k') of Eq. 1.

    Pair 0 couples the anchor (K_0 = 1) with slot 1: only row 0 exists; rows 1..K-1
    of pair 0 are -inf.  Vectors are unit-normed, so <o, i> is their cosine."""
    o = o.reshape(Bm1, K, -1)
    i = i.reshape(Bm1, K, -1)
    out = np.full((Bm1, K, K), -np.inf)
    out[0, 0, :] = sigma * (i[0] @ o0)
    for s in range(1, Bm1):
        out[s] = sigma * (o[s - 1] @ i[s].T)
    return out


# ---------------------------------------------------------------------------------
# a5. greedy walk and (next) exact best path
# ---------------------------------------------------------------------------------

def _argmax_lowest_rank(z: np.ndarray, rank: np.ndarray) -> int:
    best = np.flatnonzero(z == z.max())
    return int(best[np.argmin(rank[best])])


def greedy_walk(scores: np.ndarray, rank: Optional[np.ndarray] = None):
    """c_1 = argmax_k phi(0, 1, k); c_s = argmax_k phi(s-1, c_{s-1}, k)
    (LiLiCorr Sec. 3.5, Eq. 8).  Decided on float32-rounded scores (reading R-argmax);
    ties to the lowest rank.  Returns (choice [B-1], path_score [B-1], margin [B-1]):
    margin = top-1 minus top-2 score of each decision (inf when K = 1)."""
    z32 = scores.astype(np.float32).astype(np.float64)
    Bm1, K, _ = z32.shape
    rank = np.tile(np.arange(K), (Bm1, 1)) if rank is None else rank
    choice = np.zeros(Bm1, dtype=np.int64)
    path = np.zeros(Bm1)
    margin = np.full(Bm1, np.inf)
    prev = 0
    for s in range(Bm1):
        z = z32[s, prev]
        c = _argmax_lowest_rank(z, rank[s])
        choice[s], path[s] = c, z[c]
        if K > 1:
            margin[s] = z[c] - np.max(np.delete(z, c))
        prev = c
    return choice, path, margin


def sample_walk(scores: np.ndarray, temperature: float, u: np.ndarray,
                rank: Optional[np.ndarray] = None):
    """Sampled commit (serving PR, "Sampling the committed path"; LiLiCorr Sec. 3.3,
    Eq. 2): each slot draws c_s from softmax_k(z_s[k] / T) with z_s[k] = phi(s-1,
    c_{s-1}, k), given the previous draw.  T <= 0 is the greedy commit (same decisions as
    greedy_walk) with a one-hot proposal.

    Reading R-sample: the draw is by inverse CDF with one uniform u_s in [0, 1) per slot
    supplied by the caller: weights w_k = exp((z_k - max z) / T) in float64 from the
    float32-rounded scores, W = their sum taken in rank order, and c_s = the first
    candidate in rank order whose running sum exceeds u_s * W (the last candidate with
    w > 0 if rounding leaves none).  A slot whose scores are all -inf takes rank 0.
    Returns (choice [B-1], path_score [B-1], proposal [B-1, K]) with proposal[s] = w / W
    in candidate order."""
    z32 = scores.astype(np.float32).astype(np.float64)
    Bm1, K, _ = z32.shape
    rank = np.tile(np.arange(K), (Bm1, 1)) if rank is None else rank
    if temperature <= 0:
        choice, path, _ = greedy_walk(scores, rank)
        prop = np.zeros((Bm1, K))
        prop[np.arange(Bm1), choice] = 1.0
        return choice, path, prop
    choice = np.zeros(Bm1, dtype=np.int64)
    path = np.zeros(Bm1)
    prop = np.zeros((Bm1, K))
    prev = 0
    for s in range(Bm1):
        z = z32[s, prev]
        order = np.argsort(rank[s], kind="stable")
        m = z.max()
        if m == -np.inf:
            c = int(order[0])
            prop[s, c] = 1.0
        else:
            w = np.exp((z - m) / float(temperature))
            W = 0.0
            for k in order:
                W += w[k]
            thr = float(np.float32(u[s])) * W
            cum, c = 0.0, -1
            for k in order:
                cum += w[k]
                if cum > thr:
                    c = int(k)
                    break
            if c < 0:
                c = int([k for k in order if w[k] > 0][-1])
            prop[s] = w / W
        choice[s], path[s] = c, z[c]
        prev = c
    return choice, path, prop


def viterbi(scores: np.ndarray, rank: Optional[np.ndarray] = None):
    """Exact maximiser of g(c) = sum_s phi(s-1, c_{s-1}, c_s) (LiLiCorr App. E, Eq. 12)
    by dynamic programming over float32-rounded scores; ties to the lowest rank of the
    final candidate and, on traceback, of each predecessor.  Returns (choice, g)."""
    z = scores.astype(np.float32).astype(np.float64)
    Bm1, K, _ = z.shape
    rank = np.tile(np.arange(K), (Bm1, 1)) if rank is None else rank
    best = z[0, 0].copy()                         # best path score ending at slot 1, k
    back = np.zeros((Bm1, K), dtype=np.int64)
    for s in range(1, Bm1):
        cand = best[:, None] + z[s]               # [prev k, next k']
        new = np.empty(K)
        for kk in range(K):
            col = cand[:, kk]
            back[s, kk] = _argmax_lowest_rank(col, rank[s - 1])
            new[kk] = col[back[s, kk]]
        best = new
    choice = np.zeros(Bm1, dtype=np.int64)
    choice[-1] = _argmax_lowest_rank(best, rank[-1])
    for s in range(Bm1 - 1, 0, -1):
        choice[s - 1] = back[s, choice[s]]
    return choice, float(best[choice[-1]])


# ---------------------------------------------------------------------------------
# whole path, one block at a time
# ---------------------------------------------------------------------------------

def rerank_candidates(cand_id: np.ndarray, cand_logit: np.ndarray, lse: np.ndarray,
                      rank: np.ndarray, w: Dict[str, np.ndarray], dims: dict,
                      target: Optional[np.ndarray], slot_hidden: Optional[np.ndarray],
                      anchor_id: Optional[int], mirror=False, sigma: float = SIGMA,
                      eps: float = RMS_EPS) -> Dict[str, np.ndarray]:
    """Steps a2..a5 for one block, from its candidate arrays [B-1, K] (any order within
    a slot; each candidate carries its own rank)."""
    Bm1, K = cand_id.shape
    H = dims["hidden"]
    slots = np.repeat(np.arange(1, Bm1 + 1), K)
    x = node_vectors(cand_id, cand_logit, lse, rank, K, w, slot_hidden, mirror)
    nodes = x.copy()
    for l in range(dims["layers"]):
        x = encoder_layer(x, layer_weights(w, l), slots, dims["heads"], dims["B_max"],
                          mirror, eps)
    t = np.zeros(H) if target is None else target
    o, i = fuse_heads(x, t, w, mirror)
    o0 = anchor_out(t, w)
    sc = pair_scores(o, i, o0, Bm1, K, sigma)
    choice, path, margin = greedy_walk(sc, rank)
    tokens = np.empty(Bm1 + 1, dtype=np.int64)
    tokens[0] = -1 if anchor_id is None else anchor_id
    tokens[1:] = cand_id[np.arange(Bm1), choice]
    return dict(tokens=tokens, choice=choice, path_score=path, margin=margin,
                pair_scores=sc, nodes=nodes, hidden=x, out_vec=o, in_vec=i, anchor_vec=o0)


def rerank_block(block_logits: np.ndarray, K: int, w: Dict[str, np.ndarray], dims: dict,
                 target: Optional[np.ndarray] = None, slot_hidden: Optional[np.ndarray] = None,
                 anchor_id: Optional[int] = None, mirror=False,
                 sigma: float = SIGMA, eps: float = RMS_EPS) -> Dict[str, np.ndarray]:
    """The whole rerank of one block: logits [B, V] -> tokens [B] and scores."""
    cand_id, cand_logit, lse = logit_pass(block_logits, K)
    rank = np.tile(np.arange(K), (cand_id.shape[0], 1))
    out = rerank_candidates(cand_id, cand_logit, lse, rank, w, dims, target, slot_hidden,
                            anchor_id, mirror, sigma, eps)
    out.update(cand_id=cand_id, cand_logit=cand_logit, lse=lse)
    return out


def rerank(logits: np.ndarray, K: int, w: Dict[str, np.ndarray], dims: dict,
           target_state: Optional[np.ndarray] = None, slot_hidden: Optional[np.ndarray] = None,
           anchor_ids: Optional[np.ndarray] = None, blocks=None, mirror=False,
           sigma: float = SIGMA, eps: float = RMS_EPS) -> Dict[str, np.ndarray]:
    """Batched driver: logits [batch, B, V] (float64-exact values) -> stacked per-block
    results for the selected blocks (all by default)."""
    blocks = range(logits.shape[0]) if blocks is None else blocks
    res = []
    for b in blocks:
        res.append(rerank_block(
            logits[b], K, w, dims,
            None if target_state is None else target_state[b],
            None if slot_hidden is None else slot_hidden[b],
            None if anchor_ids is None else int(anchor_ids[b]), mirror, sigma, eps))
    return {k: np.stack([r[k] for r in res]) for k in res[0]}
