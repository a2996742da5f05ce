"""Python binding of the LiLiCorr rerank library: argument marshalling over the C ABI.

PyTorch provides device memory and streams only; every step of the path runs in the
library's CUDA kernels.  Functions raise LilicorrError on a non-OK status.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional

import numpy as np
import torch

from . import _lib as L


class LilicorrError(RuntimeError):
    def __init__(self, status: int, what: str):
        lib = L.lib()
        msg = lib.lilicorr_status_string(status).decode()
        extra = lib.lilicorr_last_error().decode()
        super().__init__(f"{what}: {L.STATUS.get(status, status)} ({msg}){' - ' + extra if extra else ''}")
        self.status = status


def _check(status: int, what: str) -> None:
    if status != 0:
        raise LilicorrError(status, what)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ldtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return L.BF16
    if t.dtype == torch.float32:
        return L.F32
    raise ValueError(f"logits must be bfloat16 or float32, got {t.dtype}")


class Weights:
    """Head weights in a library-owned device arena (lilicorr_weights_create).

    tensors: name -> uint16 numpy array of bf16 bit patterns (shapes as the header lists).
    """

    def __init__(self, dims: dict, tensors: Dict[str, np.ndarray], device: int = 0,
                 sigma: float = 8.0, rms_eps: float = 1e-6):
        lib = L.lib()
        self.dims = dict(dims)
        self.sigma, self.rms_eps = sigma, rms_eps
        d = L.Dims(dims["layers"], dims["hidden"], dims["heads"], dims["ffn"], dims["d_e"],
                   dims["B_max"], dims["K_max"], dims["V"], sigma, rms_eps)
        keep = []
        arr = (L.Tensor * len(tensors))()
        for i, (name, a) in enumerate(tensors.items()):
            a = np.ascontiguousarray(a)
            if a.dtype != np.uint16:
                raise ValueError(f"{name}: expected bf16 bit patterns (uint16), got {a.dtype}")
            nb = name.encode()
            keep += [a, nb]
            shp = (C.c_int64 * 4)(*(list(a.shape) + [0] * (4 - a.ndim)))
            arr[i] = L.Tensor(nb, a.ctypes.data, L.BF16, a.ndim, shp)
        h = C.c_void_p()
        _check(lib.lilicorr_weights_create(C.byref(d), arr, len(tensors), device, C.byref(h)),
               "lilicorr_weights_create")
        self._h = h
        self.device = device

    @property
    def handle(self):
        return self._h

    def close(self) -> None:
        if getattr(self, "_h", None):
            L.lib().lilicorr_weights_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace_bytes(self, batch: int, B: int, K: int) -> int:
        return int(L.lib().lilicorr_workspace_bytes(self._h, batch, B, K))

    def workspace(self, batch: int, B: int, K: int) -> torch.Tensor:
        n = self.workspace_bytes(batch, B, K)
        if n == 0:
            raise LilicorrError(1, "lilicorr_workspace_bytes")
        return torch.empty(n, dtype=torch.uint8, device=f"cuda:{self.device}")


TAP_NAMES = ("choice", "cand_id", "cand_logit", "lse", "pair_scores", "nodes", "hidden",
             "out_vec", "in_vec", "anchor_vec")


def rerank(w: Weights, logits: torch.Tensor, K: int, slot_hidden: Optional[torch.Tensor] = None,
           target_state: Optional[torch.Tensor] = None, anchor_ids: Optional[torch.Tensor] = None,
           taps=False, workspace: Optional[torch.Tensor] = None, out=None,
           stream=None) -> Dict[str, torch.Tensor]:
    """lilicorr_rerank on device tensors.  logits [batch, B, V] bf16/f32 on the GPU.

    taps: False, True (all) or an iterable of tap names.  Returns tokens, path_score and
    the requested taps.  `out` may hold preallocated tokens/path_score tensors."""
    batch, B, V = logits.shape
    dev = logits.device
    H, E = w.dims["hidden"], w.dims["d_e"]
    S = (B - 1) * K
    if out is None:
        out = {"tokens": torch.empty(batch, B, dtype=torch.int32, device=dev),
               "path_score": torch.empty(batch, B - 1, dtype=torch.float32, device=dev)}
    tap_ptr = None
    if taps:
        names = TAP_NAMES if taps is True else tuple(taps)
        shapes = {"choice": ((batch, B - 1), torch.int32), "cand_id": ((batch, B - 1, K), torch.int32),
                  "cand_logit": ((batch, B - 1, K), torch.float32), "lse": ((batch, B - 1), torch.float32),
                  "pair_scores": ((batch, B - 1, K, K), torch.float32),
                  "nodes": ((batch, S, H), torch.float32), "hidden": ((batch, S, H), torch.float32),
                  "out_vec": ((batch, S, E), torch.float32), "in_vec": ((batch, S, E), torch.float32),
                  "anchor_vec": ((batch, E), torch.float32)}
        tp = L.Taps()
        for n in names:
            shp, dt = shapes[n]
            out[n] = torch.empty(shp, dtype=dt, device=dev)
            setattr(tp, n, out[n].data_ptr())
        tap_ptr = C.byref(tp)
    if workspace is None:
        workspace = w.workspace(batch, B, K)
    st = L.lib().lilicorr_rerank(
        w.handle, _ptr(logits), _ldtype(logits), batch, B, V, K, _ptr(slot_hidden),
        _ptr(target_state), _ptr(anchor_ids), _ptr(out["tokens"]), _ptr(out["path_score"]),
        tap_ptr, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "lilicorr_rerank")
    return out


def rerank_host_workspace(w: Weights, batch: int, B: int, K: int, ldtype: int) -> torch.Tensor:
    n = int(L.lib().lilicorr_workspace_bytes_host(w.handle, batch, B, K, ldtype))
    if n == 0:
        raise LilicorrError(1, "lilicorr_workspace_bytes_host")
    return torch.empty(n, dtype=torch.uint8, device=f"cuda:{w.device}")


def rerank_host(w: Weights, logits: torch.Tensor, K: int, target_state=None, slot_hidden=None,
                anchor_ids=None, tokens: Optional[torch.Tensor] = None,
                path_score: Optional[torch.Tensor] = None, workspace=None, stream=None):
    """lilicorr_rerank_host: host (ideally pinned) CPU tensors in and out; synchronous."""
    batch, B, V = logits.shape
    ld = _ldtype(logits)
    if tokens is None:
        tokens = torch.empty(batch, B, dtype=torch.int32)
    if path_score is None:
        path_score = torch.empty(batch, B - 1, dtype=torch.float32)
    if workspace is None:
        workspace = rerank_host_workspace(w, batch, B, K, ld)
    st = L.lib().lilicorr_rerank_host(
        w.handle, _ptr(logits), ld, batch, B, V, K, _ptr(slot_hidden), _ptr(target_state),
        _ptr(anchor_ids), _ptr(tokens), _ptr(path_score), _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check(st, "lilicorr_rerank_host")
    return tokens, path_score


def topk_lse_workspace(batch: int, B: int, V: int, K: int, ldtype: int, device) -> Optional[torch.Tensor]:
    n = int(L.lib().lilicorr_topk_lse_workspace_bytes(batch, B, V, K, ldtype))
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def topk_lse(logits: torch.Tensor, K: int, workspace: Optional[torch.Tensor] = None, out=None,
             stream=None):
    """lilicorr_topk_lse: (cand_id [batch,B-1,K] int32, cand_logit f32, lse [batch,B-1] f32)."""
    batch, B, V = logits.shape
    ld = _ldtype(logits)
    dev = logits.device
    if out is None:
        out = (torch.empty(batch, B - 1, K, dtype=torch.int32, device=dev),
               torch.empty(batch, B - 1, K, dtype=torch.float32, device=dev),
               torch.empty(batch, B - 1, dtype=torch.float32, device=dev))
    if workspace is None:
        workspace = topk_lse_workspace(batch, B, V, K, ld, dev)
    st = L.lib().lilicorr_topk_lse(_ptr(logits), ld, batch, B, V, K, _ptr(out[0]), _ptr(out[1]),
                                   _ptr(out[2]), _ptr(workspace),
                                   0 if workspace is None else workspace.numel(), _stream(stream))
    _check(st, "lilicorr_topk_lse")
    return out


def topk_lse_shard(logits_slice: torch.Tensor, id_offset: int, K: int,
                   records: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """lilicorr_topk_lse_shard on one vocabulary slice [batch,B,V_shard] (last dimension
    contiguous, rows may be strided, e.g. a column slice of the whole logits): returns
    the packed row records as a uint8 tensor [batch*(B-1), record_bytes]."""
    batch, B, Vs = logits_slice.shape
    if logits_slice.stride(2) != 1 or logits_slice.stride(0) != B * logits_slice.stride(1):
        raise ValueError("slice rows must have a uniform stride and contiguous columns")
    ld = _ldtype(logits_slice)
    rb = int(L.lib().lilicorr_topk_lse_shard_record_bytes(K))
    rows = batch * (B - 1)
    if records is None:
        records = torch.empty(rows, rb, dtype=torch.uint8, device=logits_slice.device)
    ws = topk_lse_workspace(batch, B, Vs, min(K, Vs), ld, logits_slice.device)
    # a strided view by design (rows row_stride apart): its pointer is passed as it is
    st = L.lib().lilicorr_topk_lse_shard(logits_slice.data_ptr(), ld, batch, B, Vs,
                                         logits_slice.stride(1), id_offset, K, _ptr(records),
                                         _ptr(ws), 0 if ws is None else ws.numel(),
                                         _stream(stream))
    _check(st, "lilicorr_topk_lse_shard")
    return records


def topk_lse_merge(records: torch.Tensor, K: int, stream=None):
    """lilicorr_topk_lse_merge of records [n_shards, rows, record_bytes] (uint8):
    (cand_id [rows,K] int32, cand_logit [rows,K] f32, lse [rows] f32)."""
    n, rows, _ = records.shape
    dev = records.device
    cid = torch.empty(rows, K, dtype=torch.int32, device=dev)
    cv = torch.empty(rows, K, dtype=torch.float32, device=dev)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    st = L.lib().lilicorr_topk_lse_merge(_ptr(records.contiguous()), n, rows, K, _ptr(cid),
                                         _ptr(cv), _ptr(lse), _stream(stream))
    _check(st, "lilicorr_topk_lse_merge")
    return cid, cv, lse


def lm_head_workspace_bytes(rows: int, V: int, D: int, K: int) -> int:
    """lilicorr_lm_head_workspace_bytes (0 for unsupported sizes)."""
    return int(L.lib().lilicorr_lm_head_workspace_bytes(rows, V, D, K))


def lm_head_topk_lse(hidden: torch.Tensor, w_lm: torch.Tensor, K: int,
                     workspace: Optional[torch.Tensor] = None, out=None, stream=None):
    """lilicorr_lm_head_topk_lse: the projection hidden [rows, D] x w_lm [V, D]^T (bf16)
    fused with the top-K / log-sum-exp pass.  Returns (cand_id [rows,K] int32,
    cand_logit [rows,K] f32, lse [rows] f32); the logits themselves are never stored."""
    if hidden.dtype != torch.bfloat16 or w_lm.dtype != torch.bfloat16:
        raise ValueError("hidden and w_lm must be bfloat16")
    rows, D = hidden.shape
    V, D2 = w_lm.shape
    if D2 != D:
        raise ValueError("hidden and w_lm disagree on D")
    dev = hidden.device
    if out is None:
        out = (torch.empty(rows, K, dtype=torch.int32, device=dev),
               torch.empty(rows, K, dtype=torch.float32, device=dev),
               torch.empty(rows, dtype=torch.float32, device=dev))
    if workspace is None:
        n = int(L.lib().lilicorr_lm_head_workspace_bytes(rows, V, D, K))
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    st = L.lib().lilicorr_lm_head_topk_lse(_ptr(hidden), _ptr(w_lm), rows, V, D, K,
                                           _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                                           _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "lilicorr_lm_head_topk_lse")
    return out


def greedy_walk(pair_scores: torch.Tensor, cand_id: torch.Tensor,
                anchor_ids: Optional[torch.Tensor] = None, stream=None):
    """lilicorr_greedy_walk on given scores [batch,B-1,K,K]: (tokens, choice, path_score)."""
    batch, Bm1, K, _ = pair_scores.shape
    B = Bm1 + 1
    dev = pair_scores.device
    tokens = torch.empty(batch, B, dtype=torch.int32, device=dev)
    choice = torch.empty(batch, Bm1, dtype=torch.int32, device=dev)
    path = torch.empty(batch, Bm1, dtype=torch.float32, device=dev)
    st = L.lib().lilicorr_greedy_walk(_ptr(pair_scores), _ptr(cand_id), _ptr(anchor_ids), batch,
                                      B, K, _ptr(tokens), _ptr(choice), _ptr(path),
                                      _stream(stream))
    _check(st, "lilicorr_greedy_walk")
    return tokens, choice, path


def viterbi(pair_scores: torch.Tensor, cand_id: torch.Tensor,
            anchor_ids: Optional[torch.Tensor] = None, stream=None):
    """lilicorr_viterbi on given scores [batch,B-1,K,K]: the exact best path,
    (tokens, choice, path_score, total)."""
    batch, Bm1, K, _ = pair_scores.shape
    B = Bm1 + 1
    dev = pair_scores.device
    tokens = torch.empty(batch, B, dtype=torch.int32, device=dev)
    choice = torch.empty(batch, Bm1, dtype=torch.int32, device=dev)
    path = torch.empty(batch, Bm1, dtype=torch.float32, device=dev)
    total = torch.empty(batch, dtype=torch.float64, device=dev)
    st = L.lib().lilicorr_viterbi(_ptr(pair_scores), _ptr(cand_id), _ptr(anchor_ids), batch, B, K,
                                  _ptr(tokens), _ptr(choice), _ptr(path), _ptr(total),
                                  _stream(stream))
    _check(st, "lilicorr_viterbi")
    return tokens, choice, path, total


def sample_walk(pair_scores: torch.Tensor, cand_id: torch.Tensor,
                temperature: Optional[torch.Tensor] = None,
                uniforms: Optional[torch.Tensor] = None,
                anchor_ids: Optional[torch.Tensor] = None, stream=None):
    """lilicorr_sample_walk on given scores [batch,B-1,K,K] with per-row temperature
    [batch] and uniforms [batch,B-1]: (tokens, choice, path_score, proposal)."""
    batch, Bm1, K, _ = pair_scores.shape
    B = Bm1 + 1
    dev = pair_scores.device
    tokens = torch.empty(batch, B, dtype=torch.int32, device=dev)
    choice = torch.empty(batch, Bm1, dtype=torch.int32, device=dev)
    path = torch.empty(batch, Bm1, dtype=torch.float32, device=dev)
    prop = torch.empty(batch, Bm1, K, dtype=torch.float32, device=dev)
    st = L.lib().lilicorr_sample_walk(_ptr(pair_scores), _ptr(cand_id), _ptr(anchor_ids),
                                      _ptr(temperature), _ptr(uniforms), batch, B, K,
                                      _ptr(tokens), _ptr(choice), _ptr(path), _ptr(prop),
                                      _stream(stream))
    _check(st, "lilicorr_sample_walk")
    return tokens, choice, path, prop


def launch_count() -> int:
    return int(L.lib().lilicorr_launch_count())


def device_error() -> int:
    code = C.c_uint32(0)
    st = L.lib().lilicorr_device_error(C.byref(code))
    if st not in (0, 8):
        _check(st, "lilicorr_device_error")
    return int(code.value)


def stage_timing(enable: bool) -> None:
    L.lib().lilicorr_stage_timing(1 if enable else 0)


def stage_times() -> Dict[str, dict]:
    """Per-kernel timing accumulated since the last read: {name: {"ms": total ms,
    "launches": n}} plus "calls"."""
    n = 32
    ms = (C.c_double * n)()
    la = (C.c_int64 * n)()
    calls = C.c_int64(0)
    k = L.lib().lilicorr_stage_times(ms, la, n, C.byref(calls))
    out = {L.lib().lilicorr_stage_name(i).decode(): {"ms": ms[i], "launches": int(la[i])}
           for i in range(k)}
    out["calls"] = int(calls.value)
    return out


def diag_wait_timeout(logits_row: torch.Tensor, limit_cycles: int, stream=None) -> None:
    """lilicorr_diag_wait_timeout on one bf16 row [V] (V <= 16384): a logit pass whose only
    copy is withheld, so its bounded waits give up; read the result with device_error()."""
    if logits_row.dtype != torch.bfloat16 or logits_row.dim() != 1:
        raise ValueError("expected one bf16 row")
    dev = logits_row.device
    cid = torch.empty(1, dtype=torch.int32, device=dev)
    cv = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(1, dtype=torch.float32, device=dev)
    st = L.lib().lilicorr_diag_wait_timeout(_ptr(logits_row), logits_row.numel(), limit_cycles,
                                            _ptr(cid), _ptr(cv), _ptr(lse), _stream(stream))
    _check(st, "lilicorr_diag_wait_timeout")
