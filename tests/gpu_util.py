"""Helpers shared by the GPU tests: move a seeded workload to the device, run
the library path through the C ABI, and compare against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle

REL_TOL = 2e-3   # max relative error of importance scores vs the fp64 oracle


def bits_to_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def to_device(w):
    return {
        "q": bits_to_bf16(w.q_bits),
        "k": bits_to_bf16(w.k_bits),
        "cu_q": i32(w.cu_seqlens_q),
        "cu_k": i32(w.cu_seqlens_k),
        "req_off": i32(w.req_tok_offsets),
        "keep": i32(w.keep_per_req),
        "hidden": bits_to_bf16(w.hidden_bits),
        "pos": i32(w.pos),
    }


def run_path(tsel, w, dev=None, softmax_scale=0.0):
    """importance -> top-B -> compaction through the C ABI; returns host arrays."""
    dev = dev or to_device(w)
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k,
                                                         w.num_heads), dtype=torch.uint8,
                     device="cuda")
    scores, lse = tsel.tsel_importance(dev["q"], dev["k"], dev["cu_q"], dev["cu_k"],
                                       w.max_seqlen_q, w.max_seqlen_k,
                                       softmax_scale=softmax_scale, workspace=ws)
    keep_idx, cu_keep = tsel.tsel_select_topk(scores, dev["req_off"], dev["keep"], w.total_keep,
                                              workspace=ws)
    oh, op, oi, oc = tsel.tsel_gather_compact(dev["hidden"], dev["pos"], dev["cu_k"], keep_idx,
                                              workspace=ws)
    status = tsel.tsel_read_device_status(ws)
    torch.cuda.synchronize()
    return {
        "scores": scores.cpu().numpy(),
        "lse": lse.cpu().numpy(),
        "keep_idx": keep_idx.cpu().numpy(),
        "cu_keep": cu_keep.cpu().numpy(),
        "hidden": oh.view(torch.int16).cpu().numpy().view(np.uint16),
        "pos": op.cpu().numpy(),
        "img_id": oi.cpu().numpy(),
        "cu_seqlens_kept": oc.cpu().numpy(),
        "status": status,
    }


def max_rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    gpu = gpu.astype(np.float64)
    zero = ref == 0
    assert np.all(gpu[zero] == 0), "scores must be exactly 0 where the oracle gives 0"
    nz = ~zero
    if not np.any(nz):
        return 0.0
    return float(np.max(np.abs(gpu[nz] - ref[nz]) / np.abs(ref[nz])))


def check_selection_exact(w, out):
    """Top-B and compaction are bit-exact against the oracle fed the same fp32 scores."""
    k_ref, cu_ref = oracle.select_topk(out["scores"].astype(np.float32), w.req_tok_offsets,
                                       w.keep_per_req)
    assert np.array_equal(out["keep_idx"], k_ref)
    assert np.array_equal(out["cu_keep"], cu_ref)
    h_ref, p_ref, i_ref, c_ref = oracle.gather_compact(w.hidden_bits, w.pos, w.cu_seqlens_k, k_ref)
    assert np.array_equal(out["hidden"], h_ref)
    assert np.array_equal(out["pos"], p_ref)
    assert np.array_equal(out["img_id"], i_ref)
    assert np.array_equal(out["cu_seqlens_kept"], c_ref)


def check_keep_set_agreement(w, out, ref_scores):
    """The GPU keep set equals the oracle's, except tokens whose oracle score is
    within REL_TOL of the request's B-th oracle score."""
    k_ref, _ = oracle.select_topk(ref_scores, w.req_tok_offsets, w.keep_per_req)
    got = set(out["keep_idx"].tolist())
    exp = set(k_ref.tolist())
    off = w.req_tok_offsets
    for r in range(len(off) - 1):
        lo, hi, B = off[r], off[r + 1], int(w.keep_per_req[r])
        if B == 0 or B == hi - lo:
            continue
        s = ref_scores[lo:hi]
        bth = np.sort(s)[::-1][B - 1]
        for t in (got ^ exp):
            if lo <= t < hi:
                assert abs(ref_scores[t] - bth) <= REL_TOL * bth, (t, ref_scores[t], bth)


def segment_slice(w, g):
    """Q/K bits and local cu_seqlens of segment g alone."""
    q0, q1 = int(w.cu_seqlens_q[g]), int(w.cu_seqlens_q[g + 1])
    k0, k1 = int(w.cu_seqlens_k[g]), int(w.cu_seqlens_k[g + 1])
    return w.q_bits[q0:q1], w.k_bits[k0:k1], [0, q1 - q0], [0, k1 - k0], (q0, q1, k0, k1)


_ORACLE_FULL = {}


def oracle_full(name: str):
    """(lse, scores) of the fp64 oracle over a whole named workload (bf16 inputs),
    segments spread over a pool of host processes; computed once per test run."""
    if name not in _ORACLE_FULL:
        import workloads as W
        from oracle_pool import importance_by_segment
        _ORACLE_FULL[name] = importance_by_segment(W.make(name))
    return _ORACLE_FULL[name]


def keep_set_flips(w, keep_idx, ref_scores):
    """Tokens kept by exactly one of `keep_idx` and the oracle's top-B of
    `ref_scores`, with each one's relative distance from its request's B-th
    oracle score. Returns (flipped token indices, distances)."""
    k_ref, _ = oracle.select_topk(ref_scores, w.req_tok_offsets, w.keep_per_req)
    flips = np.array(sorted(set(np.asarray(keep_idx).tolist()) ^ set(k_ref.tolist())),
                     dtype=np.int64)
    dist = np.zeros(flips.size)
    off = w.req_tok_offsets
    for r in range(len(off) - 1):
        lo, hi, B = int(off[r]), int(off[r + 1]), int(w.keep_per_req[r])
        sel = (flips >= lo) & (flips < hi)
        if not np.any(sel):
            continue
        bth = np.sort(ref_scores[lo:hi])[::-1][B - 1]
        dist[sel] = np.abs(ref_scores[flips[sel]] - bth) / bth
    return flips, dist
