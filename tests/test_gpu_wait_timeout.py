"""The device-side timeouts, exercised without faulting, trapping or hanging the GPU.

Every wait of the library's kernels on an mbarrier is bounded: after its limit the
waiting warp records a site bit in the unit's device error word and the kernel returns,
so the context stays usable and the host learns of it through lilicorr_device_error.
lilicorr_diag_wait_timeout runs the logit pass on one row whose only bulk copy is
announced to its barrier but never issued, with a short limit: both the consumers'
stage wait and the producer's final drain must give up, report their bits and return,
and the next normal call must still produce correct results.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ERR_K1_FULL_WAIT, ERR_K1_DRAIN = 1 << 0, 1 << 1


@pytest.fixture(scope="module")
def lc():
    import __graft_entry__
    __graft_entry__.build()
    import draft_block_candidate_gb300 as m
    return m


def test_withheld_copy_times_out_and_reports_its_sites(lc):
    assert lc.device_error() == 0          # clean start (also clears older bits)
    row = torch.randn(4096, device="cuda").to(torch.bfloat16)
    lc.diag_wait_timeout(row, 200_000)     # ~0.1 ms per wait at GB300 clocks
    code = lc.device_error()
    assert code & ERR_K1_FULL_WAIT, hex(code)
    assert code & ERR_K1_DRAIN, hex(code)
    assert code < (1 << 8), hex(code)      # only logit-pass sites
    assert lc.device_error() == 0          # reading clears the word
    # the context is still usable: a normal logit pass is exact
    x = row.reshape(1, 1, -1).expand(1, 2, -1).contiguous()
    cid, cv, lse = lc.topk_lse(x, 4)
    torch.cuda.synchronize()
    xf = x[0, 1].float().cpu().numpy().astype(np.float64)
    ids = np.argsort(-xf, kind="stable")[:4]
    assert cid.cpu().numpy()[0, 0].tolist() == ids.tolist()
    ref = xf.max() + np.log(np.exp(xf - xf.max()).sum())
    assert abs(float(lse[0, 0]) - ref) <= 1e-5
    assert lc.device_error() == 0


def test_timeout_self_check_refuses_bad_arguments(lc):
    from draft_block_candidate_gb300 import _lib
    lib = _lib.lib()
    row = torch.zeros(40000, dtype=torch.bfloat16, device="cuda")
    o = torch.empty(4, dtype=torch.int32, device="cuda")
    f = torch.empty(4, dtype=torch.float32, device="cuda")
    # a row longer than one stage, a limit below the floor, a null output
    assert lib.lilicorr_diag_wait_timeout(row.data_ptr(), 40000, 100000, o.data_ptr(),
                                          f.data_ptr(), f.data_ptr(), None) == 1
    assert lib.lilicorr_diag_wait_timeout(row.data_ptr(), 4096, 10, o.data_ptr(),
                                          f.data_ptr(), f.data_ptr(), None) == 1
    assert lib.lilicorr_diag_wait_timeout(row.data_ptr(), 4096, 100000, None,
                                          f.data_ptr(), f.data_ptr(), None) == 1
