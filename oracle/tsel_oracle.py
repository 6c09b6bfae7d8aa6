"""fp64 CPU oracle for attention-score vision-token pruning.

TEST INFRASTRUCTURE ONLY. This module is the plain, slow, obviously correct
statement of what the CUDA library computes. Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import it; the library never calls it
and never falls back to it. It shares no code with the CUDA path.

What it follows (page titles and sections):

* "LiteVLM: A Low-Latency Vision-Language Model Inference Pipeline for
  Resource-Constrained Environments" (paper review), section 3.2 "Token
  Selection Module" and the "core formulas" paragraph: visual tokens are
  scored by attention, s_j = Attn(h, v_j), from the first decoder layer, and
  the most important are kept with keep ratio r (r = 0.8 keeps 80 %).
* The dynamic vision-token compression article, section 3.1 (VisionZip: a few
  dominant tokens identified by attention score), section 3.2 (score = the
  mean attention each visual token receives at a ViT layer; all images of a
  request share one candidate pool under one global budget; probabilities are
  rebuilt from the softmax LSE and reduced along columns, so only one score per
  token leaves the kernel; after pruning the lengths, image boundaries,
  original spatial indices and position ids are updated).

Readings taken where the pages are silent (each is also listed in the design
notes):

* Mean over heads and over the query rows of the token's own segment:
  score_j = (1 / (H * Nq_g)) * sum_h sum_i P[h, i, j].
* The softmax of a query row runs over the keys of its own segment only
  (block-diagonal varlen attention, no causal mask); scale 1/sqrt(d) unless
  given.
* GQA: query head h reads KV head floor(h / (H / Hkv)).
* A segment with no query rows gives its keys score 0; a query row with no
  keys has LSE = -inf.
* Budget: B = floor(r * N) in integer per-mille arithmetic.
* Top-B order: score descending, ties to the lowest token index; the kept
  indices are returned in ascending order, requests concatenated.
* Compaction copies rows and position ids of the kept tokens in ascending
  order; the image id of a token is the segment holding it; the new per-image
  boundaries are prefix sums of kept counts.
* Score normalisation: "mean" (the default above) or "sum" (the same total
  attention received, not divided by H * Nq_g).
* Dynamic keep ratio (the article's section 6.2 leaves the rule open): per
  request, the fewest top tokens whose scores hold a fraction tau of the
  request's total score, bounded by a floor and a ceiling ratio. Scores enter
  as integers q_j = floor(s_j * 2^(24 - E)), E the binary exponent with
  max_j s_j in [2^(E-1), 2^E), so the sums are exact and independent of the
  summation order.

Parity status: every function here is pinned by closed forms, invariants and
brute force in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# Input conversion
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp64 values, exactly (bf16 is a truncated fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """FP8 E4M3 (OCP 8-bit floating point, "FN" variant) -> fp64, exactly.

    1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
    subnormal (2^-6 * m/8); no infinities; S.1111.111 is NaN; largest finite
    magnitude 448. (LiteVLM's FP8 deployment quantises to this format.)
    """
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 15) & ((b & 0x7) == 7), np.nan, val)
    return sign * val


def decode_inputs(bits, fmt: str) -> np.ndarray:
    if fmt == "bf16":
        return bf16_bits_to_f64(bits)
    if fmt == "e4m3":
        return e4m3_bits_to_f64(bits)
    raise ValueError(f"unknown input format {fmt}")


# ---------------------------------------------------------------------------
# Importance (LiteVLM token selection; VisionZip-style mean attention received)
# ---------------------------------------------------------------------------

def attention_probabilities(q: np.ndarray, k: np.ndarray, scale: float):
    """Full attention matrix of one segment and one head, materialised.

    q: [Nq, d] fp64, k: [Nk, d] fp64. Returns (P [Nq, Nk], lse [Nq]) with
    P = softmax(scale * q k^T) row by row and lse the natural-log normaliser
    (the softmax LSE a FlashAttention-style kernel returns).
    """
    nq, nk = q.shape[0], k.shape[0]
    if nk == 0:
        return np.zeros((nq, 0)), np.full(nq, -np.inf)
    s = scale * (q @ k.T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    p = e / l
    lse = (m + np.log(l))[:, 0]
    return p, lse


def importance(q_bits, k_bits, cu_seqlens_q, cu_seqlens_k, softmax_scale=None, fmt="bf16",
               norm="mean"):
    """Mean attention probability received by every key token.

    q_bits: [Tq, H, d] and k_bits: [Tk, Hkv, d] as bit patterns of `fmt`
    ("bf16": uint16, "e4m3": uint8). cu_seqlens_q / cu_seqlens_k: int [G+1];
    segment g attends queries [cu_q[g], cu_q[g+1]) to keys [cu_k[g], cu_k[g+1]).
    softmax_scale multiplies q.k (defaults to 1/sqrt(d)); for quantised inputs
    it carries the dequantisation scales too. norm="sum" returns the total
    attention received (sum over heads and query rows) instead of the mean.
    Returns (lse [H, Tq] fp64 natural log, scores [Tk] fp64).
    """
    if norm not in ("mean", "sum"):
        raise ValueError(f"unknown normalisation {norm}")
    q = decode_inputs(q_bits, fmt)
    k = decode_inputs(k_bits, fmt)
    tq, H, d = q.shape
    tk, Hkv, _ = k.shape
    group = H // Hkv
    scale = (1.0 / np.sqrt(d)) if (softmax_scale is None or softmax_scale <= 0) else float(softmax_scale)
    cu_q = np.asarray(cu_seqlens_q, dtype=np.int64)
    cu_k = np.asarray(cu_seqlens_k, dtype=np.int64)
    lse = np.full((H, tq), -np.inf)
    scores = np.zeros(tk)
    for g in range(cu_k.shape[0] - 1):
        q0, q1 = cu_q[g], cu_q[g + 1]
        k0, k1 = cu_k[g], cu_k[g + 1]
        acc = np.zeros(k1 - k0)
        for h in range(H):
            p, lse_h = attention_probabilities(q[q0:q1, h, :], k[k0:k1, h // group, :], scale)
            lse[h, q0:q1] = lse_h
            acc += p.sum(axis=0)          # attention received = column sum
        n_rows = H * (q1 - q0)
        if norm == "sum":
            scores[k0:k1] = acc
        else:
            scores[k0:k1] = acc / n_rows if n_rows > 0 else 0.0
    return lse, scores


# ---------------------------------------------------------------------------
# Budget and pooled global top-B
# ---------------------------------------------------------------------------

def keep_count(n_tokens: int, keep_permille: int) -> int:
    """Tokens kept at keep ratio r = keep_permille / 1000: floor(r * n)."""
    return (int(n_tokens) * int(keep_permille)) // 1000


def select_topk(scores, req_tok_offsets, keep_per_req):
    """Global top-B per request over the pooled tokens of all its images.

    Order: score descending, then token index ascending. The comparison is
    made in the dtype of ``scores`` (fp32 scores are compared as fp32).
    Returns (keep_idx int32 [sum B], cu_keep int32 [R+1]); indices ascending
    inside each request, requests in order.
    """
    scores = np.asarray(scores)
    off = np.asarray(req_tok_offsets, dtype=np.int64)
    keep = np.asarray(keep_per_req, dtype=np.int64)
    out = []
    cu = [0]
    for r in range(off.shape[0] - 1):
        lo, hi = off[r], off[r + 1]
        idx = np.arange(lo, hi)
        order = np.lexsort((idx, -scores[lo:hi]))   # primary: -score, then index
        chosen = np.sort(idx[order[: keep[r]]])
        out.append(chosen)
        cu.append(cu[-1] + chosen.shape[0])
    keep_idx = np.concatenate(out) if out else np.zeros(0, np.int64)
    return keep_idx.astype(np.int32), np.asarray(cu, dtype=np.int32)


def score_quanta(scores) -> list:
    """Integer score quanta of one request: q_j = floor(s_j * 2^(24 - E)) with
    max_j s_j in [2^(E-1), 2^E); all zero when every score is 0. Exact: the
    scaling is by a power of two and the floor is taken in fp64 on fp32 inputs.
    Scores must be finite and >= 0."""
    s = np.asarray(scores, dtype=np.float64)
    if s.size == 0:
        return []
    smax = float(s.max())
    if smax <= 0.0:
        return [0] * s.size
    _, e = math.frexp(smax)          # smax = m * 2^e, m in [0.5, 1)
    return [int(math.floor(math.ldexp(float(v), 24 - e))) for v in s]


def dynamic_budget(scores, req_tok_offsets, mass_permille, min_permille, max_permille):
    """Per request: the fewest tokens, taken in top-B order (score descending,
    index ascending), whose quanta sum to at least T = ceil(tau * M) with
    tau = mass_permille / 1000 and M the request's total quanta; then bounded
    to [floor(n * min_permille / 1000), floor(n * max_permille / 1000)].
    Returns int32 [R]."""
    scores = np.asarray(scores)
    off = np.asarray(req_tok_offsets, dtype=np.int64)
    out = []
    for r in range(off.shape[0] - 1):
        lo, hi = int(off[r]), int(off[r + 1])
        n = hi - lo
        q = score_quanta(scores[lo:hi])
        M = sum(q)
        T = (M * int(mass_permille) + 999) // 1000
        b = 0
        if T > 0:
            idx = np.arange(lo, hi)
            order = np.lexsort((idx, -scores[lo:hi].astype(np.float64)))
            acc = 0
            for b, j in enumerate(order, start=1):
                acc += q[j]
                if acc >= T:
                    break
        floor_b = (n * int(min_permille)) // 1000
        ceil_b = (n * int(max_permille)) // 1000
        out.append(min(max(b, floor_b), ceil_b))
    return np.asarray(out, dtype=np.int32)


# ---------------------------------------------------------------------------
# Compaction with metadata
# ---------------------------------------------------------------------------

def gather_compact(hidden, pos, cu_seqlens_k, keep_idx):
    """Copy kept rows in ascending order and rebuild per-image metadata.

    hidden: [Tk, D] (any dtype, copied bit for bit); pos: int [Tk, P].
    Returns (out_hidden [K, D], out_pos [K, P], img_id int32 [K],
    cu_seqlens_kept int32 [G+1]).
    """
    keep_idx = np.asarray(keep_idx, dtype=np.int64)
    cu = np.asarray(cu_seqlens_k, dtype=np.int64)
    out_hidden = np.asarray(hidden)[keep_idx]
    out_pos = np.asarray(pos)[keep_idx]
    img_id = np.zeros(keep_idx.shape[0], dtype=np.int32)
    counts = np.zeros(cu.shape[0] - 1, dtype=np.int64)
    for n, t in enumerate(keep_idx):
        g = int(np.searchsorted(cu, t, side="right") - 1)   # segment holding token t
        img_id[n] = g
        counts[g] += 1
    cu_kept = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return out_hidden, out_pos, img_id, cu_kept


def prune(q_bits, k_bits, cu_seqlens_q, cu_seqlens_k, req_tok_offsets, keep_per_req,
          hidden, pos, softmax_scale=None, fmt="bf16"):
    """The whole path: importance, pooled top-B, compaction."""
    lse, scores = importance(q_bits, k_bits, cu_seqlens_q, cu_seqlens_k, softmax_scale, fmt)
    keep_idx, cu_keep = select_topk(scores, req_tok_offsets, keep_per_req)
    out_hidden, out_pos, img_id, cu_kept = gather_compact(hidden, pos, cu_seqlens_k, keep_idx)
    return {"lse": lse, "scores": scores, "keep_idx": keep_idx, "cu_keep": cu_keep,
            "hidden": out_hidden, "pos": out_pos, "img_id": img_id, "cu_seqlens_kept": cu_kept}
