"""Attention-score vision-token pruning on GB300: Python binding of libtsel.

Every function here marshals torch tensors into the C ABI of ``include/tsel.h``
(device pointers, sizes, the current CUDA stream) and calls the library; all
the work runs in the library's CUDA kernels. PyTorch only provides device
memory and streams. If ``libtsel.so`` has not been built the first call raises;
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from ._build import LIB_PATH, build

__all__ = [
    "TselError", "load_library", "build",
    "tsel_importance_workspace_size", "tsel_importance", "tsel_importance_noalloc",
    "tsel_select_topk_workspace_size", "tsel_select_topk",
    "tsel_score_select_workspace_size", "tsel_score_select",
    "tsel_select_topk_hist_workspace_size", "tsel_select_topk_hist", "TSEL_SEL_STAGE_TOPK",
    "tsel_gather_compact_workspace_size", "tsel_gather_compact", "tsel_gather_compact_counted",
    "tsel_dynamic_budget", "TSEL_KEEP_FROM_DEVICE",
    "tsel_keep_count", "tsel_read_device_status", "tsel_clear_device_status",
    "tsel_importance_redo_pairs", "tsel_select_path_counts", "tsel_importance_one_launch",
    "tsel_status_string", "tsel_last_error", "tsel_probe_ex2",
    "TSEL_DEV_SEQLENS", "TSEL_DEV_REQUESTS", "TSEL_DEV_KEEP_IDX", "TSEL_DEV_TIMEOUT", "TSEL_DEV_NAN",
    "TSEL_IMP_LSE_PROVIDED", "TSEL_IMP_FP8_E4M3", "TSEL_IMP_SCORE_SUM", "TSEL_IMP_ROWREF_FIXED", "TSEL_IMP_ROWREF_MOVING", "TSEL_IMP_TWO_PASS", "TSEL_IMP_TEST_STALL", "TSEL_IMP_STAGE_PREP", "TSEL_IMP_STAGE_PASS1", "TSEL_IMP_STAGE_PASS2",
]

TSEL_OK = 0
TSEL_ERR_INVALID_VALUE = 1
TSEL_ERR_UNSUPPORTED = 2
TSEL_ERR_WORKSPACE = 3
TSEL_ERR_CUDA = 4
TSEL_ERR_DEVICE_CHECK = 5

TSEL_DEV_SEQLENS = 0x1
TSEL_DEV_REQUESTS = 0x2
TSEL_DEV_KEEP_IDX = 0x4
TSEL_DEV_TIMEOUT = 0x8
TSEL_DEV_NAN = 0x10

TSEL_KEEP_FROM_DEVICE = -1

TSEL_IMP_LSE_PROVIDED = 0x1
TSEL_IMP_FP8_E4M3 = 0x2
TSEL_IMP_SCORE_SUM = 0x4
TSEL_IMP_ROWREF_FIXED = 0x8
TSEL_IMP_ROWREF_MOVING = 0x20
TSEL_IMP_TWO_PASS = 0x40
TSEL_IMP_TEST_STALL = 0x10000
TSEL_IMP_STAGE_PREP = 0x100
TSEL_IMP_STAGE_PASS1 = 0x200
TSEL_IMP_STAGE_PASS2 = 0x400
TSEL_SEL_STAGE_TOPK = 0x800

_c_int, _c_i64, _c_size, _c_float, _c_uint, _p = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                                   ctypes.c_float, ctypes.c_uint, ctypes.c_void_p)

_SIGNATURES = {
    "tsel_importance_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int]),
    "tsel_importance": (_c_int, [_p, _c_i64, _p, _c_i64, _p, _p, _c_int, _c_int, _c_int, _c_int,
                                 _c_int, _c_int, _c_int, _c_int, _c_float, _c_uint, _p, _p, _p,
                                 _c_size, _p]),
    "tsel_select_topk_workspace_size": (_c_size, [_c_int]),
    "tsel_select_topk": (_c_int, [_p, _c_int, _p, _c_int, _p, _c_int, _p, _p, _p, _c_size, _p]),
    "tsel_gather_compact_workspace_size": (_c_size, []),
    "tsel_gather_compact": (_c_int, [_p, _c_i64, _c_int, _c_int, _p, _c_int, _p, _c_int, _c_int,
                                     _p, _c_int, _p, _p, _p, _p, _p, _c_size, _p]),
    "tsel_gather_compact_counted": (_c_int, [_p, _c_i64, _c_int, _c_int, _p, _c_int, _p, _c_int,
                                             _c_int, _p, _p, _c_int, _p, _p, _p, _p, _p, _c_size,
                                             _p]),
    "tsel_dynamic_budget": (_c_int, [_p, _c_int, _p, _c_int, _c_int, _c_int, _c_int, _p, _p, _p,
                                     _c_size, _p]),
    "tsel_keep_count": (_c_int, [_c_int, _c_int]),
    "tsel_importance_one_launch": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                            _c_uint]),
    "tsel_read_device_status": (_c_int, [_p, ctypes.POINTER(ctypes.c_uint32), _p]),
    "tsel_clear_device_status": (_c_int, [_p, _p]),
    "tsel_importance_redo_pairs": (_c_int, [_p, ctypes.POINTER(ctypes.c_int32), _p]),
    "tsel_select_path_counts": (_c_int, [_p, ctypes.POINTER(ctypes.c_int32), _p]),
    "tsel_status_string": (ctypes.c_char_p, [_c_int]),
    "tsel_last_error": (ctypes.c_char_p, []),
    "tsel_probe_ex2": (_c_int, [_c_int, _c_int, _p, _p]),
    "tsel_score_select_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "tsel_score_select": (_c_int, [_p, _c_i64, _p, _c_i64, _p, _p, _c_int, _c_int, _c_int, _c_int,
                                   _c_int, _c_int, _c_int, _c_int, _c_float, _c_uint, _p, _p,
                                   _p, _c_int, _p, _c_int, _p, _p, _p, _c_size, _p]),
    "tsel_select_topk_hist_workspace_size": (_c_size, [_c_int]),
    "tsel_select_topk_hist": (_c_int, [_p, _c_int, _p, _c_int, _p, _c_int, _p, _p, _p, _c_size,
                                       _p]),
    "tsel_importance_noalloc": (_c_int, [_p, _c_i64, _p, _c_i64, _p, _p, _c_int, _c_int, _c_int,
                                         _c_int, _c_int, _c_int, _c_int, _c_int, _c_float, _p, _p,
                                         _p, _p]),
}

_lib: Optional[ctypes.CDLL] = None


class TselError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} [status {status}]")
        self.status = status


def load_library() -> ctypes.CDLL:
    """Loads the in-tree libtsel.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtsel.so is not built at {LIB_PATH}: call "
                               "attention_score_vision_gb300.build() (nvcc, sm_103a) first")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int) -> None:
    if status != TSEL_OK:
        lib = load_library()
        name = lib.tsel_status_string(status).decode()
        detail = lib.tsel_last_error().decode()
        raise TselError(status, f"{name}: {detail}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, dtype, name: str) -> None:
    if t.dtype != dtype or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA {dtype} tensor")


def _new_workspace(nbytes: int, device) -> torch.Tensor:
    # zeroed so the device status word starts clear
    return torch.zeros(max(nbytes, 1024), dtype=torch.uint8, device=device)


def _check_qk(q: torch.Tensor, k: torch.Tensor, cu_seqlens_q: torch.Tensor,
              cu_seqlens_k: torch.Tensor, allow_fp8: bool):
    """Checks the importance inputs the C ABI cannot see (dtypes, devices, the
    [rows, heads, head_dim] layout the TMA maps are built from); returns
    (Tq, H, d, Tk, Hkv, fp8)."""
    fp8_types = (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8))
    fp8 = allow_fp8 and q.dtype in fp8_types and k.dtype in fp8_types
    if fp8:
        if not (q.is_cuda and k.is_cuda):
            raise TypeError("q and k must be CUDA tensors")
    else:
        _need(q, torch.bfloat16, "q")
        _need(k, torch.bfloat16, "k")
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q and k must be [rows, heads, head_dim] tensors")
    tq, H, d = q.shape
    tk, Hkv, dk = k.shape
    if dk != d:
        raise ValueError("q and k head_dim differ")
    for t, name in ((q, "q"), (k, "k")):
        if t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must have contiguous [heads, head_dim] rows")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    for t in (k, cu_seqlens_q, cu_seqlens_k):
        if t.device != q.device:
            raise ValueError("q, k and cu_seqlens must be on the same device")
    return tq, H, d, tk, Hkv, fp8


# ---------------------------------------------------------------------------
# Importance
# ---------------------------------------------------------------------------

def tsel_importance_workspace_size(num_seg: int, total_q: int, total_k: int, num_heads: int) -> int:
    return int(load_library().tsel_importance_workspace_size(num_seg, total_q, total_k, num_heads))


def tsel_importance(q: torch.Tensor, k: torch.Tensor, cu_seqlens_q: torch.Tensor,
                    cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, *,
                    softmax_scale: float = 0.0, flags: int = 0,
                    lse: Optional[torch.Tensor] = None, scores: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, want_lse: bool = True,
                    stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Mean attention received per key token; returns (scores [Tk], lse [H, Tq] or None).

    q: bf16 [Tq, H, d] (rows may be strided, head dim contiguous);
    k: bf16 [Tk, Hkv, d]; cu_seqlens_*: int32 [G+1] on the same device.
    With flags containing TSEL_IMP_LSE_PROVIDED, `lse` (fp32 [H, Tq], natural
    log) is an input and only the column pass runs. uint8 / float8_e4m3fn q and
    k are E4M3 inputs; softmax_scale then includes their dequantisation scales.
    """
    tq, H, d, tk, Hkv, fp8 = _check_qk(q, k, cu_seqlens_q, cu_seqlens_k, allow_fp8=True)
    if fp8:
        flags |= TSEL_IMP_FP8_E4M3   # E4M3 bytes; softmax_scale must carry the dequant scales
    G = cu_seqlens_k.numel() - 1
    dev = q.device
    if scores is None:
        scores = torch.empty(tk, dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((H, tq), dtype=torch.float32, device=dev)
    nbytes = tsel_importance_workspace_size(G, tq, tk, H)
    if workspace is None:
        workspace = _new_workspace(nbytes, dev)
    lib = load_library()
    with torch.cuda.device(dev):   # the library works on the current device
        st = lib.tsel_importance(_ptr(q), q.stride(0), _ptr(k), k.stride(0), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_k), G, tq, tk, int(max_seqlen_q),
                                 int(max_seqlen_k), H, Hkv, d, float(softmax_scale), int(flags),
                                 _ptr(lse), _ptr(scores), _ptr(workspace), workspace.numel(),
                                 _stream(stream, dev))
    _check(st)
    return scores, lse


def tsel_importance_noalloc(q: torch.Tensor, k: torch.Tensor, cu_seqlens_q: torch.Tensor,
                            cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int, *,
                            softmax_scale: float = 0.0, lse: Optional[torch.Tensor] = None,
                            scores: Optional[torch.Tensor] = None,
                            device_status: Optional[torch.Tensor] = None, want_lse: bool = True,
                            stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """tsel_importance with the library's static scratch array instead of a
    workspace (for callers that cannot allocate device memory). Output
    tensors passed in are used as they are; calls on one device must not
    overlap on the GPU."""
    tq, H, d, tk, Hkv, _ = _check_qk(q, k, cu_seqlens_q, cu_seqlens_k, allow_fp8=False)
    if device_status is not None:
        _need(device_status, torch.int32, "device_status")
        if device_status.device != q.device:
            raise ValueError("device_status must be on q's device")
    G = cu_seqlens_k.numel() - 1
    dev = q.device
    if scores is None:
        scores = torch.empty(tk, dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((H, tq), dtype=torch.float32, device=dev)
    # the static scratch array is looked up on the current device: make it q's
    with torch.cuda.device(dev):
        st = load_library().tsel_importance_noalloc(
            _ptr(q), q.stride(0), _ptr(k), k.stride(0), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), G,
            tq, tk, int(max_seqlen_q), int(max_seqlen_k), H, Hkv, d, float(softmax_scale),
            _ptr(lse), _ptr(scores), _ptr(device_status), _stream(stream, dev))
    _check(st)
    return scores, lse


def tsel_score_select_workspace_size(num_seg: int, total_q: int, total_k: int, num_heads: int,
                                     num_req: int) -> int:
    return int(load_library().tsel_score_select_workspace_size(num_seg, total_q, total_k,
                                                                num_heads, num_req))


def tsel_score_select(q: torch.Tensor, k: torch.Tensor, cu_seqlens_q: torch.Tensor,
                      cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int,
                      req_tok_offsets: torch.Tensor, keep_per_req: torch.Tensor, total_keep: int,
                      *, softmax_scale: float = 0.0, flags: int = 0,
                      lse: Optional[torch.Tensor] = None, scores: Optional[torch.Tensor] = None,
                      keep_idx: Optional[torch.Tensor] = None,
                      cu_keep: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, want_lse: bool = True,
                      stream=None):
    """tsel_importance + tsel_select_topk in one call (the top-B starts from the
    score histograms the column pass builds); returns (scores, lse, keep_idx, cu_keep)."""
    tq, H, d, tk, Hkv, fp8 = _check_qk(q, k, cu_seqlens_q, cu_seqlens_k, allow_fp8=True)
    if fp8:
        flags |= TSEL_IMP_FP8_E4M3
    _need(req_tok_offsets, torch.int32, "req_tok_offsets")
    _need(keep_per_req, torch.int32, "keep_per_req")
    G = cu_seqlens_k.numel() - 1
    R = keep_per_req.numel()
    dev = q.device
    if scores is None:
        scores = torch.empty(tk, dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((H, tq), dtype=torch.float32, device=dev)
    if keep_idx is None:
        cap = tk if int(total_keep) == TSEL_KEEP_FROM_DEVICE else int(total_keep)
        keep_idx = torch.empty(cap, dtype=torch.int32, device=dev)
    if cu_keep is None:
        cu_keep = torch.empty(R + 1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _new_workspace(tsel_score_select_workspace_size(G, tq, tk, H, R), dev)
    with torch.cuda.device(dev):
        st = load_library().tsel_score_select(
            _ptr(q), q.stride(0), _ptr(k), k.stride(0), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), G,
            tq, tk, int(max_seqlen_q), int(max_seqlen_k), H, Hkv, d, float(softmax_scale),
            int(flags), _ptr(lse), _ptr(scores), _ptr(req_tok_offsets), R, _ptr(keep_per_req),
            int(total_keep), _ptr(keep_idx), _ptr(cu_keep), _ptr(workspace), workspace.numel(),
            _stream(stream, dev))
    _check(st)
    return scores, lse, keep_idx, cu_keep


# ---------------------------------------------------------------------------
# Top-B
# ---------------------------------------------------------------------------

def tsel_select_topk_workspace_size(num_req: int) -> int:
    return int(load_library().tsel_select_topk_workspace_size(num_req))


def tsel_select_topk(scores: torch.Tensor, req_tok_offsets: torch.Tensor,
                     keep_per_req: torch.Tensor, total_keep: int, *,
                     keep_idx: Optional[torch.Tensor] = None, cu_keep: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Pooled top-B per request; returns (keep_idx int32 [total_keep], cu_keep int32 [R+1]).

    total_keep = TSEL_KEEP_FROM_DEVICE takes budgets computed on the device
    (tsel_dynamic_budget): keep_idx then has room for every token and
    cu_keep[R] holds the kept count."""
    _need(scores, torch.float32, "scores")
    _need(req_tok_offsets, torch.int32, "req_tok_offsets")
    _need(keep_per_req, torch.int32, "keep_per_req")
    R = keep_per_req.numel()
    dev = scores.device
    if keep_idx is None:
        cap = scores.numel() if int(total_keep) == TSEL_KEEP_FROM_DEVICE else int(total_keep)
        keep_idx = torch.empty(cap, dtype=torch.int32, device=dev)
    if cu_keep is None:
        cu_keep = torch.empty(R + 1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _new_workspace(tsel_select_topk_workspace_size(R), dev)
    st = load_library().tsel_select_topk(_ptr(scores), scores.numel(), _ptr(req_tok_offsets), R,
                                         _ptr(keep_per_req), int(total_keep), _ptr(keep_idx),
                                         _ptr(cu_keep), _ptr(workspace), workspace.numel(),
                                         _stream(stream, dev))
    _check(st)
    return keep_idx, cu_keep


def tsel_select_topk_hist_workspace_size(num_req: int) -> int:
    return int(load_library().tsel_select_topk_hist_workspace_size(num_req))


def tsel_select_topk_hist(scores: torch.Tensor, req_tok_offsets: torch.Tensor,
                          keep_per_req: torch.Tensor, total_keep: int, *,
                          keep_idx: Optional[torch.Tensor] = None,
                          cu_keep: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None,
                          stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """tsel_select_topk started from per-request score histograms (built by one
    extra launch); same results. Returns (keep_idx, cu_keep)."""
    _need(scores, torch.float32, "scores")
    _need(req_tok_offsets, torch.int32, "req_tok_offsets")
    _need(keep_per_req, torch.int32, "keep_per_req")
    R = keep_per_req.numel()
    dev = scores.device
    if keep_idx is None:
        cap = scores.numel() if int(total_keep) == TSEL_KEEP_FROM_DEVICE else int(total_keep)
        keep_idx = torch.empty(cap, dtype=torch.int32, device=dev)
    if cu_keep is None:
        cu_keep = torch.empty(R + 1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _new_workspace(tsel_select_topk_hist_workspace_size(R), dev)
    with torch.cuda.device(dev):
        st = load_library().tsel_select_topk_hist(
            _ptr(scores), scores.numel(), _ptr(req_tok_offsets), R, _ptr(keep_per_req),
            int(total_keep), _ptr(keep_idx), _ptr(cu_keep), _ptr(workspace), workspace.numel(),
            _stream(stream, dev))
    _check(st)
    return keep_idx, cu_keep


def tsel_dynamic_budget(scores: torch.Tensor, req_tok_offsets: torch.Tensor, mass_permille: int,
                        min_permille: int = 0, max_permille: int = 1000, *,
                        keep_per_req: Optional[torch.Tensor] = None,
                        total_keep: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None,
                        stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-request budgets from the scores (fewest top tokens holding mass_permille of
    the request's score quanta, bounded); returns (keep_per_req int32 [R], total int32 [1])."""
    _need(scores, torch.float32, "scores")
    _need(req_tok_offsets, torch.int32, "req_tok_offsets")
    R = req_tok_offsets.numel() - 1
    dev = scores.device
    if keep_per_req is None:
        keep_per_req = torch.empty(max(R, 0), dtype=torch.int32, device=dev)
    if total_keep is None:
        total_keep = torch.empty(1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _new_workspace(tsel_select_topk_workspace_size(R), dev)
    st = load_library().tsel_dynamic_budget(_ptr(scores), scores.numel(), _ptr(req_tok_offsets), R,
                                            int(mass_permille), int(min_permille), int(max_permille),
                                            _ptr(keep_per_req), _ptr(total_keep), _ptr(workspace),
                                            workspace.numel(), _stream(stream, dev))
    _check(st)
    return keep_per_req, total_keep


# ---------------------------------------------------------------------------
# Compaction
# ---------------------------------------------------------------------------

def tsel_gather_compact_workspace_size() -> int:
    return int(load_library().tsel_gather_compact_workspace_size())


def tsel_gather_compact(hidden: torch.Tensor, pos: Optional[torch.Tensor], cu_seqlens_k: torch.Tensor,
                        keep_idx: torch.Tensor, *, out_hidden: Optional[torch.Tensor] = None,
                        out_pos: Optional[torch.Tensor] = None, out_img_id: Optional[torch.Tensor] = None,
                        out_cu_seqlens: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None):
    """Compacts kept rows; returns (out_hidden, out_pos, out_img_id, out_cu_seqlens)."""
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    _need(keep_idx, torch.int32, "keep_idx")
    if hidden.dim() != 2 or hidden.stride(1) != 1 or not hidden.is_cuda:
        raise ValueError("hidden must be a CUDA [T, D] tensor with contiguous rows")
    tk, D = hidden.shape
    K = keep_idx.numel()
    G = cu_seqlens_k.numel() - 1
    dev = hidden.device
    P = 0 if pos is None else pos.shape[1]
    if pos is not None:
        _need(pos, torch.int32, "pos")
        if not pos.is_contiguous() or pos.shape[0] != tk:
            raise ValueError("pos must be a contiguous int32 [T, P] tensor")
    if out_hidden is None:
        out_hidden = torch.empty((K, D), dtype=hidden.dtype, device=dev)
    if out_pos is None and P > 0:
        out_pos = torch.empty((K, P), dtype=torch.int32, device=dev)
    if out_img_id is None:
        out_img_id = torch.empty(K, dtype=torch.int32, device=dev)
    if out_cu_seqlens is None:
        out_cu_seqlens = torch.empty(G + 1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _new_workspace(tsel_gather_compact_workspace_size(), dev)
    st = load_library().tsel_gather_compact(
        _ptr(hidden), hidden.stride(0), D, hidden.element_size(), _ptr(pos), P, _ptr(cu_seqlens_k),
        G, tk, _ptr(keep_idx), K, _ptr(out_hidden), _ptr(out_pos), _ptr(out_img_id),
        _ptr(out_cu_seqlens), _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(st)
    return out_hidden, out_pos, out_img_id, out_cu_seqlens


def tsel_gather_compact_counted(hidden: torch.Tensor, pos: Optional[torch.Tensor],
                                cu_seqlens_k: torch.Tensor, keep_idx: torch.Tensor,
                                num_kept: torch.Tensor, max_kept: int, *,
                                out_hidden: Optional[torch.Tensor] = None,
                                out_pos: Optional[torch.Tensor] = None,
                                out_img_id: Optional[torch.Tensor] = None,
                                out_cu_seqlens: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None, stream=None):
    """tsel_gather_compact with the kept count read on the device (num_kept: int32
    device scalar, e.g. cu_keep[R:]); outputs have room for max_kept rows, of which
    the first *num_kept are written."""
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    _need(keep_idx, torch.int32, "keep_idx")
    _need(num_kept, torch.int32, "num_kept")
    if hidden.dim() != 2 or hidden.stride(1) != 1 or not hidden.is_cuda:
        raise ValueError("hidden must be a CUDA [T, D] tensor with contiguous rows")
    tk, D = hidden.shape
    K = int(max_kept)
    if keep_idx.numel() < K:
        raise ValueError("keep_idx has fewer than max_kept entries")
    G = cu_seqlens_k.numel() - 1
    dev = hidden.device
    P = 0 if pos is None else pos.shape[1]
    if pos is not None:
        _need(pos, torch.int32, "pos")
        if not pos.is_contiguous() or pos.shape[0] != tk:
            raise ValueError("pos must be a contiguous int32 [T, P] tensor")
    if out_hidden is None:
        out_hidden = torch.empty((K, D), dtype=hidden.dtype, device=dev)
    if out_pos is None and P > 0:
        out_pos = torch.empty((K, P), dtype=torch.int32, device=dev)
    if out_img_id is None:
        out_img_id = torch.empty(K, dtype=torch.int32, device=dev)
    if out_cu_seqlens is None:
        out_cu_seqlens = torch.empty(G + 1, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = _new_workspace(tsel_gather_compact_workspace_size(), dev)
    st = load_library().tsel_gather_compact_counted(
        _ptr(hidden), hidden.stride(0), D, hidden.element_size(), _ptr(pos), P, _ptr(cu_seqlens_k),
        G, tk, _ptr(keep_idx), _ptr(num_kept), K, _ptr(out_hidden), _ptr(out_pos), _ptr(out_img_id),
        _ptr(out_cu_seqlens), _ptr(workspace), workspace.numel(), _stream(stream, dev))
    _check(st)
    return out_hidden, out_pos, out_img_id, out_cu_seqlens


# ---------------------------------------------------------------------------
# Helpers
# ---------------------------------------------------------------------------

def tsel_importance_one_launch(num_seg: int, total_q: int, total_k: int, max_seqlen_q: int,
                               max_seqlen_k: int, num_heads: int, head_dim: int,
                               flags: int = 0) -> int:
    """1 if tsel_importance takes the one-launch path for these sizes and flags
    on the current device, 0 if the scheduled two-pass launches, -1 on a CUDA
    error."""
    return int(load_library().tsel_importance_one_launch(
        int(num_seg), int(total_q), int(total_k), int(max_seqlen_q), int(max_seqlen_k),
        int(num_heads), int(head_dim), int(flags)))


def tsel_keep_count(n_tokens: int, keep_permille: int) -> int:
    return int(load_library().tsel_keep_count(int(n_tokens), int(keep_permille)))


def tsel_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Device status bits of a workspace (synchronises the stream)."""
    bits = ctypes.c_uint32(0)
    st = load_library().tsel_read_device_status(_ptr(workspace), ctypes.byref(bits),
                                                _stream(stream, workspace.device))
    if st not in (TSEL_OK, TSEL_ERR_DEVICE_CHECK):
        _check(st)
    return int(bits.value)


def tsel_importance_redo_pairs(workspace: torch.Tensor, stream=None) -> int:
    """(head, query pair)s the last importance call on `workspace` redid with a
    moving reference (synchronises the stream)."""
    n = ctypes.c_int32(0)
    _check(load_library().tsel_importance_redo_pairs(_ptr(workspace), ctypes.byref(n),
                                                     _stream(stream, workspace.device)))
    return int(n.value)


def tsel_select_path_counts(workspace: torch.Tensor, stream=None) -> list:
    """Top-B requests per threshold path on `workspace` since it was zeroed:
    [radix rounds, histogram + rounds, histogram + candidates, candidates
    rejected, ranked in the one-launch importance kernel] (synchronises the
    stream)."""
    c = (ctypes.c_int32 * 5)()
    _check(load_library().tsel_select_path_counts(_ptr(workspace), c,
                                                  _stream(stream, workspace.device)))
    return [int(x) for x in c]


def tsel_clear_device_status(workspace: torch.Tensor, stream=None) -> None:
    _check(load_library().tsel_clear_device_status(_ptr(workspace), _stream(stream, workspace.device)))


def tsel_status_string(status: int) -> str:
    return load_library().tsel_status_string(int(status)).decode()


def tsel_last_error() -> str:
    return load_library().tsel_last_error().decode()


def tsel_probe_ex2(blocks: int, iters: int, sink: torch.Tensor, stream=None) -> None:
    """Enqueues the MUFU exp2 throughput probe (blocks*512*iters*8 exp2).
    sink[blocks*512:] receives block 0's SM cycles and nanoseconds (two
    int64 words), whose ratio is the SM clock during the probe."""
    _need(sink, torch.float32, "sink")
    if sink.numel() < blocks * 512 + 4:
        raise ValueError("sink needs blocks*512 + 4 floats")
    _check(load_library().tsel_probe_ex2(int(blocks), int(iters), _ptr(sink),
                                         _stream(stream, sink.device)))
