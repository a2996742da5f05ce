"""lilicorr_topk_lse_noalloc, the allocation-free form of the logit pass, for callers that
cannot allocate device memory when they run it (a serving loop whose memory belongs to
its own pool, code inside a CUDA-graph capture, a C host without a device allocator).

Called through the C ABI and checked against lilicorr_topk_lse (the workspace form) on
two calls in a row: the second call reuses the library's static scratch, which still
holds the first call's contents.  Shapes include split rows, the case that actually
uses the scratch.  This file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from tests.gpu_util import LSE_ATOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as m
    return m


@pytest.mark.parametrize("ldtype,batch,B,V,K", [
    ("bf16", 1, 16, 151_936, 8),     # 15 rows split across CTAs: scratch in use
    ("bf16", 2, 16, 151_936, 32),
    ("f32", 1, 9, 40_000, 16),
    ("bf16", 4, 16, 3001, 16),       # unaligned rows, one CTA per row
])
def test_noalloc_matches_workspace_entry_on_two_calls(lc, ldtype, batch, B, V, K):
    from draft_block_candidate_gb300 import _lib
    lib = _lib.lib()
    rng = np.random.default_rng(V + K)
    x = torch.from_numpy((rng.standard_normal((batch, B, V)) * 2).astype(np.float32)).cuda()
    if ldtype == "bf16":
        x = x.to(torch.bfloat16)
    code = _lib.BF16 if ldtype == "bf16" else _lib.F32
    ref_id, ref_val, ref_lse = lc.topk_lse(x, K)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        cid = torch.full((batch, B - 1, K), -7, dtype=torch.int32, device="cuda")
        cv = torch.full((batch, B - 1, K), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((batch, B - 1), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.lilicorr_topk_lse_noalloc(x.data_ptr(), code, batch, B, V, K, cid.data_ptr(),
                                           cv.data_ptr(), lse.data_ptr(), stream)
        assert st == 0, lib.lilicorr_last_error()
        torch.cuda.synchronize()
        assert torch.equal(cid, ref_id), f"call {call}: ids differ"
        assert torch.equal(cv, ref_val), f"call {call}: logits differ"
        assert (lse - ref_lse).abs().max().item() <= LSE_ATOL, f"call {call}: lse differs"


def test_noalloc_refuses_bad_arguments(lc):
    from draft_block_candidate_gb300 import _lib
    lib = _lib.lib()
    x = torch.zeros(1, 4, 100, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(64, dtype=torch.int32, device="cuda")
    f = torch.empty(64, dtype=torch.float32, device="cuda")
    assert lib.lilicorr_topk_lse_noalloc(x.data_ptr(), _lib.BF16, 1, 4, 100, 33, out.data_ptr(),
                                         f.data_ptr(), f.data_ptr(), None) == 1
    assert lib.lilicorr_topk_lse_noalloc(None, _lib.BF16, 1, 4, 100, 4, out.data_ptr(),
                                         f.data_ptr(), f.data_ptr(), None) == 1
