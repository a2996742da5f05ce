"""CPU oracle of the LiLiCorr draft-time rerank path.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline
leg import this package.  It holds no compiled code and shares none with the CUDA
library.
"""
from . import lilicorr_oracle  # noqa: F401
from .lilicorr_oracle import (  # noqa: F401
    SIGMA,
    bf16_round,
    greedy_walk,
    logit_pass,
    rerank,
    rerank_block,
    rerank_candidates,
    viterbi,
)
