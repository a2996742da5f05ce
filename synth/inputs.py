"""Seeded synthetic workloads: drafter logits, head weights and the optional per-block
inputs of the LiLiCorr draft-time rerank.

The pages measure on public benchmarks (SPEED-Bench entropy tiers and a concurrency
sweep, "LiLiCorr: Lightweight Likelihood Correlation of Parallel Drafts for
Speculative Decoding", Sec. 4.1 and Sec. 4.3) with trained drafters, none of which
exist here.  These generators stand in for them with the same shapes: a block of
B = 16 positions (anchor + 15 drafted slots, Table 4), a 151,936-token vocabulary
(the Qwen3 vocabulary named in the serving PR's measurements), K candidates per slot,
bf16 logits, and random-init head weights of the stated widths.

Everything here is input construction: normal draws, a Zipf-ranked planted peak, a
temperature, bf16 packing.  No step of the rerank method is computed here.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

# ---------------------------------------------------------------------------------
# bf16 packing (input encoding only).  bf16 is the top half of an IEEE-754 float32.
# ---------------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Pack float32 values into bf16 bit patterns (uint16), round-to-nearest-even.

    Inputs are finite; this is how the generator makes bf16 tensors.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


# ---------------------------------------------------------------------------------
# Configurations.  Encoder sizes the workload descriptions leave open: FFN = 4 x hidden
# where unstated; the high-concurrency workload reuses the single-request encoder.
# ---------------------------------------------------------------------------------

QWEN3_VOCAB = 151_936

_ENC_TINY = dict(layers=2, hidden=64, heads=2, ffn=256, d_e=32)
_ENC_SMALL = dict(layers=2, hidden=256, heads=4, ffn=1024, d_e=128)
_ENC_WIDE = dict(layers=2, hidden=512, heads=8, ffn=2048, d_e=128)

CONFIGS: Dict[str, dict] = {
    # fp32 logits ~ N(0,1), one planted token per slot at +4.
    "tiny": dict(batch=1, B=16, V=1024, K=4, ldtype="f32", gen="planted", seed=0, **_ENC_TINY),
    # bf16 logits ~ N(0, 1.5^2) with a Zipf(1.1)-ranked peak per slot.
    "single": dict(batch=1, B=16, V=QWEN3_VOCAB, K=8, ldtype="bf16", gen="zipf_peak", seed=1,
                   **_ENC_SMALL),
    # Same shapes at batch 1..128, temperature set for ~1.5 nats mean entropy.
    "sweep": dict(batch=1, B=16, V=QWEN3_VOCAB, K=8, ldtype="bf16", gen="zipf_peak_entropy",
                  seed=2, batches=(1, 4, 16, 32, 64, 128), entropy=1.5, **_ENC_SMALL),
    # batch 256, K 16; tiers at temperature 0.5 / 1.0 / 2.0.
    "highconc": dict(batch=256, B=16, V=QWEN3_VOCAB, K=16, ldtype="bf16", gen="zipf_peak_temp",
                     seed=3, tiers={"low": 0.5, "medium": 1.0, "high": 2.0}, **_ENC_SMALL),
    # batch 64, K 32, 64 near-tied logits per slot; wider encoder.
    "widepool": dict(batch=64, B=16, V=QWEN3_VOCAB, K=32, ldtype="bf16", gen="near_ties", seed=4,
                     **_ENC_WIDE),
}


def weight_shapes(dims: dict) -> "list[tuple[str, tuple[int, ...]]]":
    """Names and shapes of the head's tensor set, in a fixed order.

    dims keys: layers, hidden (H), heads (nh), ffn (F), d_e, B_max, K_max, V.
    """
    H, F, E, nh = dims["hidden"], dims["ffn"], dims["d_e"], dims["heads"]
    Bm, Km, V = dims["B_max"], dims["K_max"], dims["V"]
    out = [
        ("embed", (V, H)),
        ("slot_table", (Bm - 1, H)),
        ("rank_table", (Km, H)),
        ("conf.w1", (H, 5)),
        ("conf.b1", (H,)),
        ("conf.w2", (H, H)),
        ("conf.b2", (H,)),
    ]
    for l in range(dims["layers"]):
        p = f"layers.{l}."
        out += [
            (p + "norm1", (H,)),
            (p + "in_proj_w", (3 * H, H)),
            (p + "in_proj_b", (3 * H,)),
            (p + "out_proj_w", (H, H)),
            (p + "out_proj_b", (H,)),
            (p + "dist_bias", (nh, 2 * Bm - 3)),
            (p + "same_bias", (nh,)),
            (p + "norm2", (H,)),
            (p + "ffn.w1", (F, H)),
            (p + "ffn.b1", (F,)),
            (p + "ffn.w2", (H, F)),
            (p + "ffn.b2", (H,)),
        ]
    out += [
        ("fuse.w", (H, 3 * H)),
        ("fuse.b", (H,)),
        ("head_out.w", (E, H)),
        ("head_out.b", (E,)),
        ("head_in.w", (E, H)),
        ("head_in.b", (E,)),
        ("head_anchor.w", (E, H)),
        ("head_anchor.b", (E,)),
    ]
    return out


def make_weights(dims: dict, seed: int, std: float = 0.02, gain_jitter: float = 0.02,
                 bias_std: Optional[float] = None) -> Dict[str, np.ndarray]:
    """Random-init head weights as bf16 bit patterns (uint16 arrays).

    Every tensor is N(0, std^2) except the RMSNorm gains, which are 1 + N(0, gain_jitter^2)
    (a non-unit gain keeps the gain multiplication observable in tests).  bias_std
    overrides the std of biases and bias tables when given.
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x11C0]))
    out = {}
    for name, shape in weight_shapes(dims):
        n = int(np.prod(shape))
        if name.endswith("norm1") or name.endswith("norm2"):
            v = 1.0 + gain_jitter * rng.standard_normal(n, dtype=np.float32)
        else:
            s = std
            is_bias = (name.endswith("_b") or name.endswith(".b") or name.endswith(".b1")
                       or name.endswith(".b2") or name.endswith("_bias"))
            if bias_std is not None and is_bias:
                s = bias_std
            v = s * rng.standard_normal(n, dtype=np.float32)
        out[name] = f32_to_bf16_bits(v.reshape(shape))
    return out


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    B: int
    V: int
    K: int
    ldtype: str                    # "f32" or "bf16"
    logits: np.ndarray             # [batch, B, V]: float32, or uint16 bf16 bits
    target_state: Optional[np.ndarray]   # [batch, H] uint16 bf16 bits, or None
    slot_hidden: Optional[np.ndarray]    # [batch, B, H] uint16 bf16 bits, or None
    anchor_ids: Optional[np.ndarray]     # [batch] int32, or None
    dims: dict
    weights: Dict[str, np.ndarray]
    temperature: float = 1.0
    seed: int = 0

    def logits_f32(self, rows: Optional[slice] = None) -> np.ndarray:
        """Logits widened to float32 (exact), optionally a block range."""
        x = self.logits if rows is None else self.logits[rows]
        return x if self.ldtype == "f32" else bf16_bits_to_f32(x).reshape(x.shape)


def _zipf_cdf(V: int, a: float) -> np.ndarray:
    w = np.arange(1, V + 1, dtype=np.float64) ** (-a)
    c = np.cumsum(w)
    return c / c[-1]


def _zipf_peak_rows(rng, nrows: int, V: int, cdf: np.ndarray) -> np.ndarray:
    """nrows rows of N(0, 1.5^2) with a Zipf(1.1)-ranked id raised to max(row) + 3."""
    x = 1.5 * rng.standard_normal((nrows, V), dtype=np.float32)
    ids = np.minimum(np.searchsorted(cdf, rng.random(nrows)), V - 1)
    x[np.arange(nrows), ids] = x.max(axis=1) + np.float32(3.0)
    return x


def _mean_entropy(x: np.ndarray, T: float) -> float:
    """Generator calibration only: mean softmax entropy (nats) of rows x / T."""
    y = x.astype(np.float64) / T
    y -= y.max(axis=1, keepdims=True)
    e = np.exp(y)
    z = e.sum(axis=1, keepdims=True)
    p = e / z
    ent = -(p * (y - np.log(z))).sum(axis=1)
    return float(ent.mean())


def _calibrate_temperature(seed: int, V: int, cdf: np.ndarray, target: float) -> float:
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0xCA1]))
    x = _zipf_peak_rows(rng, 32, V, cdf)
    lo, hi = np.log(1e-3), np.log(1e3)
    for _ in range(60):
        mid = 0.5 * (lo + hi)
        if _mean_entropy(x, float(np.exp(mid))) < target:
            lo = mid
        else:
            hi = mid
    return float(np.exp(0.5 * (lo + hi)))


def make_workload(config: str, batch: Optional[int] = None, tier: Optional[str] = None,
                  K: Optional[int] = None, V: Optional[int] = None, B: Optional[int] = None,
                  seed: Optional[int] = None, with_slot_hidden: bool = False,
                  with_target: bool = True, with_anchor: bool = True,
                  weights: Optional[Dict[str, np.ndarray]] = None,
                  K_max: Optional[int] = None, **enc_overrides) -> Workload:
    """Build one seeded workload of a named configuration.

    batch / K / V / B / seed override the configuration's values (tests use this to make
    small cases of the same distribution).  tier selects a temperature tier of the
    high-concurrency workload.  Encoder sizes can be overridden with layers=, hidden=,
    heads=, ffn=, d_e=.
    """
    cfg = dict(CONFIGS[config])
    batch = cfg["batch"] if batch is None else batch
    K = cfg["K"] if K is None else K
    V = cfg["V"] if V is None else V
    B = cfg["B"] if B is None else B
    seed = cfg["seed"] if seed is None else seed
    enc = {k: cfg[k] for k in ("layers", "hidden", "heads", "ffn", "d_e")}
    enc.update(enc_overrides)
    dims = dict(enc, B_max=max(16, B), K_max=K if K_max is None else K_max, V=V)
    H = dims["hidden"]

    rng = np.random.default_rng(np.random.SeedSequence([seed, batch, K, V, B]))
    gen = cfg["gen"]
    T = 1.0
    if gen == "planted":
        x = rng.standard_normal((batch, B, V), dtype=np.float32)
        ids = rng.integers(0, V, size=(batch, B))
        bi, si = np.meshgrid(np.arange(batch), np.arange(B), indexing="ij")
        x[bi, si, ids] += np.float32(4.0)
        logits = x
    elif gen in ("zipf_peak", "zipf_peak_entropy", "zipf_peak_temp"):
        cdf = _zipf_cdf(V, 1.1)
        if gen == "zipf_peak_entropy":
            T = _calibrate_temperature(seed, V, cdf, cfg["entropy"])
        elif gen == "zipf_peak_temp":
            T = cfg["tiers"][tier or "medium"]
        logits = np.empty((batch, B, V), dtype=np.uint16)
        for b in range(batch):
            rows = _zipf_peak_rows(rng, B, V, cdf)
            if T != 1.0:
                rows = rows / np.float32(T)
            logits[b] = f32_to_bf16_bits(rows)
    elif gen == "near_ties":
        logits = np.empty((batch, B, V), dtype=np.uint16)
        n_tied = min(64, V)
        for b in range(batch):
            rows = 1.5 * rng.standard_normal((B, V), dtype=np.float32)
            for s in range(B):
                ids = rng.choice(V, size=n_tied, replace=False)
                p = rows[s].max() + np.float32(2.0)
                rows[s, ids] = p + rng.uniform(0.0, 0.05, size=n_tied).astype(np.float32)
            logits[b] = f32_to_bf16_bits(rows)
    else:
        raise ValueError(gen)

    if cfg["ldtype"] == "bf16" and logits.dtype != np.uint16:
        logits = f32_to_bf16_bits(logits)

    target = f32_to_bf16_bits(rng.standard_normal((batch, H), dtype=np.float32)) if with_target else None
    hidden = (f32_to_bf16_bits(rng.standard_normal((batch, B, H), dtype=np.float32))
              if with_slot_hidden else None)
    anchor = rng.integers(0, V, size=batch).astype(np.int32) if with_anchor else None
    if weights is None:
        weights = make_weights(dims, seed)
    return Workload(name=config + (f"/{tier}" if tier else ""), batch=batch, B=B, V=V, K=K,
                    ldtype=cfg["ldtype"], logits=logits, target_state=target,
                    slot_hidden=hidden, anchor_ids=anchor, dims=dims, weights=weights,
                    temperature=T, seed=seed)
