"""The C ABI without a GPU: the library loads, exports every declared entry point, and
refuses bad arguments and bad weight sets on the host before touching the device."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "lilicorr.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    from draft_block_candidate_gb300 import _lib
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lilicorr_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for must in ("lilicorr_rerank", "lilicorr_topk_lse", "lilicorr_greedy_walk",
                 "lilicorr_weights_create", "lilicorr_weights_destroy",
                 "lilicorr_workspace_bytes", "lilicorr_rerank_host"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from draft_block_candidate_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    for s in range(9):
        assert lib.lilicorr_status_string(s)
    assert lib.lilicorr_status_string(99) == b"unknown status"


def _tensors(dims, drop=None, extra=None, reshape=None, dtype=1):
    from synth import make_weights
    from draft_block_candidate_gb300 import _lib
    w = make_weights(dims, 0)
    if drop:
        w.pop(drop)
    if extra:
        w[extra] = np.zeros(3, np.uint16)
    if reshape:
        w[reshape] = np.zeros(w[reshape].size + 1, np.uint16)
    keep = []
    arr = (_lib.Tensor * len(w))()
    for i, (n, a) in enumerate(w.items()):
        nb = n.encode()
        keep += [a, nb]
        arr[i] = _lib.Tensor(nb, a.ctypes.data, dtype, a.ndim,
                             (C.c_int64 * 4)(*(list(a.shape) + [0] * (4 - a.ndim))))
    return arr, len(w), keep


DIMS = dict(layers=2, hidden=64, heads=2, ffn=256, d_e=32, B_max=16, K_max=4, V=1024)


def _create(lib, dims=DIMS, **kw):
    from draft_block_candidate_gb300 import _lib
    d = _lib.Dims(dims["layers"], dims["hidden"], dims["heads"], dims["ffn"], dims["d_e"],
                  dims["B_max"], dims["K_max"], dims["V"], 8.0, 1e-6)
    arr, n, keep = _tensors(dims, **kw)
    h = C.c_void_p()
    st = lib.lilicorr_weights_create(C.byref(d), arr, n, 0, C.byref(h))
    return st, h


@pytest.mark.parametrize("kw,code", [
    (dict(drop="layers.1.ffn.b2"), 3),
    (dict(drop="embed"), 3),
    (dict(extra="layers.2.norm1"), 4),
    (dict(extra="head_extra.w"), 4),
    (dict(reshape="fuse.w"), 5),
    (dict(dtype=0), 5),
])
def test_weight_set_is_checked_in_both_directions(lib, kw, code):
    st, h = _create(lib, **kw)
    assert st == code and not h.value


@pytest.mark.parametrize("bad", [dict(hidden=48), dict(heads=3), dict(K_max=33), dict(d_e=20),
                                 dict(B_max=1), dict(ffn=100)])
def test_bad_dims_refused(lib, bad):
    from draft_block_candidate_gb300 import _lib
    dims = dict(DIMS, **bad)
    d = _lib.Dims(dims["layers"], dims["hidden"], dims["heads"], dims["ffn"], dims["d_e"],
                  dims["B_max"], dims["K_max"], dims["V"], 8.0, 1e-6)
    h = C.c_void_p()
    assert lib.lilicorr_weights_create(C.byref(d), None, 0, 0, C.byref(h)) == 1


def test_topk_lse_argument_checks(lib):
    buf = (C.c_int32 * 64)()
    f = (C.c_float * 64)()
    p = C.cast(buf, C.c_void_p)
    q = C.cast(f, C.c_void_p)
    # K > 32, K > V, V < 1, B < 2, null pointers, bad dtype: refused before any launch
    assert lib.lilicorr_topk_lse(p, 1, 1, 16, 1000, 33, p, q, q, None, 0, None) == 1
    assert lib.lilicorr_topk_lse(p, 1, 1, 16, 3, 4, p, q, q, None, 0, None) == 1
    assert lib.lilicorr_topk_lse(p, 1, 1, 16, 0, 1, p, q, q, None, 0, None) == 1
    assert lib.lilicorr_topk_lse(p, 1, 1, 1, 100, 1, p, q, q, None, 0, None) == 1
    assert lib.lilicorr_topk_lse(None, 1, 1, 16, 100, 1, p, q, q, None, 0, None) == 1
    assert lib.lilicorr_topk_lse(p, 7, 1, 16, 100, 1, p, q, q, None, 0, None) == 1
    # misaligned bf16 pointer
    assert lib.lilicorr_topk_lse(p.value + 1, 1, 1, 16, 100, 1, p, q, q, None, 0, None) == 1


def test_greedy_walk_argument_checks(lib):
    x = (C.c_float * 16)()
    p = C.cast(x, C.c_void_p)
    assert lib.lilicorr_greedy_walk(p, p, None, 1, 16, 33, p, None, None, None) == 1
    assert lib.lilicorr_greedy_walk(None, p, None, 1, 16, 4, p, None, None, None) == 1
    assert lib.lilicorr_greedy_walk(p, p, None, 0, 16, 4, p, None, None, None) == 1
    assert lib.lilicorr_greedy_walk(p, p, None, 1, 65, 4, p, None, None, None) == 1


def test_rerank_refuses_null_weights(lib):
    x = (C.c_float * 16)()
    p = C.cast(x, C.c_void_p)
    assert lib.lilicorr_rerank(None, p, 1, 1, 16, 1024, 4, None, None, None, p, p, None, p, 1 << 20,
                               None) == 1
    assert lib.lilicorr_workspace_bytes(None, 1, 16, 4) == 0


def test_binding_refuses_without_library(monkeypatch, tmp_path):
    from draft_block_candidate_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no non-CUDA path"):
        _lib.lib()


def test_viterbi_argument_checks(lib):
    p = C.c_void_p(16)
    assert lib.lilicorr_viterbi(p, p, None, 1, 16, 33, p, None, None, None, None) == 1
    assert lib.lilicorr_viterbi(p, p, None, 1, 65, 4, p, None, None, None, None) == 1
    assert lib.lilicorr_viterbi(None, p, None, 1, 16, 4, p, None, None, None, None) == 1
    assert lib.lilicorr_viterbi(p, p, None, 0, 16, 4, p, None, None, None, None) == 1


def test_sample_walk_argument_checks(lib):
    p = C.c_void_p(16)
    f = lib.lilicorr_sample_walk
    assert f(p, p, None, p, None, 1, 16, 4, p, None, None, None, None) == 1  # T without u
    assert f(p, p, None, None, None, 1, 16, 33, p, None, None, None, None) == 1
    assert f(None, p, None, None, None, 1, 16, 4, p, None, None, None, None) == 1
    assert f(p, p, None, None, None, 0, 16, 4, p, None, None, None, None) == 1


def test_shard_entry_points_check_arguments(lib):
    p = C.c_void_p(256)
    assert lib.lilicorr_topk_lse_shard_record_bytes(16) == 16 * 8 + 8
    assert lib.lilicorr_topk_lse_shard_record_bytes(33) == 0
    f = lib.lilicorr_topk_lse_shard
    assert f(p, 1, 1, 16, 100, 99, 0, 8, p, None, 0, None) == 1     # stride < V_shard
    assert f(p, 1, 1, 16, 100, 100, -1, 8, p, None, 0, None) == 1   # negative offset
    assert f(p, 1, 1, 16, 100, 100, 0, 33, p, None, 0, None) == 1
    assert f(None, 1, 1, 16, 100, 100, 0, 8, p, None, 0, None) == 1
    m = lib.lilicorr_topk_lse_merge
    assert m(p, 0, 10, 8, p, p, p, None) == 1
    assert m(p, 2, 10, 33, p, p, p, None) == 1
    assert m(None, 2, 10, 8, p, p, p, None) == 1


def test_lm_head_entry_points_check_arguments(lib):
    p = C.c_void_p(256)
    ws = lib.lilicorr_lm_head_workspace_bytes
    assert ws(10, 1000, 100, 8) == 0    # D % 64 != 0
    assert ws(10, 1000, 128, 33) == 0   # K > 32
    assert ws(10, 4, 128, 8) == 0       # K > V
    assert ws(0, 1000, 128, 8) == 0     # no rows
    f = lib.lilicorr_lm_head_topk_lse
    assert f(None, p, 10, 1000, 128, 8, p, p, p, p, 1 << 20, None) == 1
    assert f(p, p, 10, 1000, 128, 8, None, p, p, p, 1 << 20, None) == 1
    assert f(p, p, 10, 1000, 100, 8, p, p, p, p, 1 << 20, None) == 1       # D % 64
    assert f(p, p, 10, 1000, 128, 0, p, p, p, p, 1 << 20, None) == 1       # K < 1
    assert f(C.c_void_p(258), p, 10, 1000, 128, 8, p, p, p, p, 1 << 20, None) == 1  # align


def test_logit_pass_scratch_stays_within_the_static_array(lib):
    """lilicorr_topk_lse_noalloc keeps its split-row scratch in a 4 MiB array compiled into
    the library and refuses shapes that need more.  Rows are split into segments only when
    fewer than 90 rows are given (at most 90 segment partials in all), so no shape reaches
    the limit: the largest need over a grid of shapes stays a few tens of KB."""
    worst = 0
    for batch in (1, 2, 3, 5, 6, 64):
        for B in (2, 3, 9, 16, 31):
            for V in (1, 1000, 16385, 151_936, 1 << 20, (1 << 30) - 7):
                for ld in (0, 1):
                    for K in (1, 8, 32):
                        if K > V:
                            continue
                        worst = max(worst, lib.lilicorr_topk_lse_workspace_bytes(batch, B, V, K, ld))
    assert 0 < worst <= 64 << 10
