"""ctypes declarations of the C ABI in include/lilicorr.h (no logic here)."""
from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblilicorr.so")

F32, BF16 = 0, 1

STATUS = {
    0: "LILICORR_OK", 1: "LILICORR_ERR_INVALID_ARG", 2: "LILICORR_ERR_UNSUPPORTED",
    3: "LILICORR_ERR_WEIGHTS_MISSING", 4: "LILICORR_ERR_WEIGHTS_SURPLUS",
    5: "LILICORR_ERR_WEIGHTS_SHAPE", 6: "LILICORR_ERR_CUDA", 7: "LILICORR_ERR_WORKSPACE",
    8: "LILICORR_ERR_DEVICE",
}

# Every function the header declares, with (restype, argtypes).
_P = C.c_void_p
SIGNATURES = {
    "lilicorr_weights_create": (C.c_int, [_P, _P, C.c_int32, C.c_int, C.POINTER(C.c_void_p)]),
    "lilicorr_weights_destroy": (None, [_P]),
    "lilicorr_weights_dims": (C.c_int, [_P, _P]),
    "lilicorr_workspace_bytes": (C.c_size_t, [_P, C.c_int64, C.c_int32, C.c_int32]),
    "lilicorr_rerank": (C.c_int, [_P, _P, C.c_int, C.c_int64, C.c_int32, C.c_int64, C.c_int32,
                                  _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "lilicorr_workspace_bytes_host": (C.c_size_t, [_P, C.c_int64, C.c_int32, C.c_int32, C.c_int]),
    "lilicorr_rerank_host": (C.c_int, [_P, _P, C.c_int, C.c_int64, C.c_int32, C.c_int64,
                                       C.c_int32, _P, _P, _P, _P, _P, _P, C.c_size_t, _P]),
    "lilicorr_topk_lse_workspace_bytes": (C.c_size_t, [C.c_int64, C.c_int32, C.c_int64,
                                                       C.c_int32, C.c_int]),
    "lilicorr_topk_lse": (C.c_int, [_P, C.c_int, C.c_int64, C.c_int32, C.c_int64, C.c_int32,
                                    _P, _P, _P, _P, C.c_size_t, _P]),
    "lilicorr_topk_lse_noalloc": (C.c_int, [_P, C.c_int, C.c_int64, C.c_int32, C.c_int64,
                                            C.c_int32, _P, _P, _P, _P]),
    "lilicorr_greedy_walk": (C.c_int, [_P, _P, _P, C.c_int64, C.c_int32, C.c_int32, _P, _P, _P,
                                       _P]),
    "lilicorr_viterbi": (C.c_int, [_P, _P, _P, C.c_int64, C.c_int32, C.c_int32, _P, _P, _P, _P,
                                   _P]),
    "lilicorr_sample_walk": (C.c_int, [_P, _P, _P, _P, _P, C.c_int64, C.c_int32, C.c_int32,
                                       _P, _P, _P, _P, _P]),
    "lilicorr_topk_lse_shard_record_bytes": (C.c_size_t, [C.c_int32]),
    "lilicorr_topk_lse_shard": (C.c_int, [_P, C.c_int, C.c_int64, C.c_int32, C.c_int64,
                                          C.c_int64, C.c_int64, C.c_int32, _P, _P, C.c_size_t,
                                          _P]),
    "lilicorr_topk_lse_merge": (C.c_int, [_P, C.c_int32, C.c_int64, C.c_int32, _P, _P, _P, _P]),
    "lilicorr_lm_head_workspace_bytes": (C.c_size_t, [C.c_int64, C.c_int64, C.c_int32,
                                                      C.c_int32]),
    "lilicorr_lm_head_topk_lse": (C.c_int, [_P, _P, C.c_int64, C.c_int64, C.c_int32, C.c_int32,
                                            _P, _P, _P, _P, C.c_size_t, _P]),
    "lilicorr_status_string": (C.c_char_p, [C.c_int]),
    "lilicorr_last_error": (C.c_char_p, []),
    "lilicorr_launch_count": (C.c_uint64, []),
    "lilicorr_device_error": (C.c_int, [C.POINTER(C.c_uint32)]),
    "lilicorr_diag_wait_timeout": (C.c_int, [_P, C.c_int64, C.c_uint32, _P, _P, _P, _P]),
    "lilicorr_stage_timing": (None, [C.c_int]),
    "lilicorr_stage_times": (C.c_int32, [C.POINTER(C.c_double), C.POINTER(C.c_int64),
                                         C.c_int32, C.POINTER(C.c_int64)]),
    "lilicorr_stage_name": (C.c_char_p, [C.c_int32]),
}


class Dims(C.Structure):
    _fields_ = [("layers", C.c_int32), ("hidden", C.c_int32), ("heads", C.c_int32),
                ("ffn", C.c_int32), ("d_e", C.c_int32), ("B_max", C.c_int32),
                ("K_max", C.c_int32), ("V", C.c_int64), ("sigma", C.c_float),
                ("rms_eps", C.c_float)]


class Tensor(C.Structure):
    _fields_ = [("name", C.c_char_p), ("host_data", C.c_void_p), ("dtype", C.c_int),
                ("ndim", C.c_int32), ("shape", C.c_int64 * 4)]


class Taps(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("choice", "cand_id", "cand_logit", "lse",
                                          "pair_scores", "nodes", "hidden", "out_vec",
                                          "in_vec", "anchor_vec")]


_lib = None


def lib():
    """The loaded library.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(nvcc, sm_103a); the rerank has no non-CUDA path")
        h = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib
