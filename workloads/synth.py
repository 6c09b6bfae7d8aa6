"""Seeded synthetic inputs for attention-score vision-token pruning.

This module only draws numbers and lays them out. It holds none of the
scoring, selection or compaction arithmetic, so the fp64 oracle and the CUDA
library can both be fed from it without sharing any of the method.

Recipe (the same for every workload):

* One ``numpy.random.Generator(PCG64(seed))`` per workload, seed
  ``0x75E10000 + index``; draws happen in a fixed order (lengths, sinks,
  scales, Q, K, hidden).
* Q, K and hidden values are drawn in fp32 and rounded once to bf16 with
  round-to-nearest-even. Arrays are returned as raw bf16 bit patterns
  (``uint16``), so every consumer sees the same bits.
* "Sink" keys: chosen without replacement, uniformly within each segment; their
  K rows (all KV heads) are multiplied by 4 before rounding.
* Position ids: ``pos_dim == 1`` holds the token's index in the packed visual
  sequence; ``pos_dim == 3`` holds (image, row, col) with 64-token rows.

The five workloads follow the shapes the pages describe: a single 256-token
image; six 256-token camera views (LiteVLM, "Patch Selection" and the 2x3 view
composite); LiteVLM's first-decoder-layer scoring of 3072 visual keys by 142
text queries; a 30-image request with image sizes between 256 and 4096 tokens
(the page on dynamic vision-token compression, section 3.3); and a batch of
eight 16-image requests.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 0x75E10000


def f32_to_bf16_bits(x: np.ndarray, chunk: int = 1 << 20) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return bits.
    Works in cache-sized chunks (the result does not depend on the chunking)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    flat = b.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for i in range(0, flat.size, chunk):
        v = flat[i:i + chunk]
        rounding = np.uint32(0x7FFF) + ((v >> np.uint32(16)) & np.uint32(1))
        out[i:i + chunk] = (v + rounding) >> np.uint32(16)
    return out.reshape(b.shape)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Quantise to FP8 E4M3 (bias 7, 3 mantissa bits, subnormals below 2^-6):
    nearest value, ties to the even code, magnitudes above 448 saturate to 448
    (no NaN is produced)."""
    f = np.asarray(x, dtype=np.float32)
    a = np.minimum(np.abs(f), np.float32(448.0))
    bits = a.view(np.int32)
    exp = (bits >> 23) - 127 + 7                       # E4M3 exponent field if normal
    mant = bits & 0x7FFFFF
    # normal range: round the 23-bit mantissa to 3 bits, ties to even
    m = (mant + 0x7FFFF + ((mant >> 20) & 1)) >> 20
    exp = exp + (m >> 3)                               # mantissa overflow carries
    m = m & 7
    code_n = (exp << 3) | m
    # subnormal range |x| < 2^-6: multiples of 2^-9, round half to even
    code_s = np.rint(a * np.float32(512.0)).astype(np.int32)   # exact scaling by 2^9
    code = np.where(exp >= 1, code_n, code_s)
    code = np.minimum(code, 0x7E)
    neg = np.signbit(f) & (code != 0)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


@dataclass
class Workload:
    """One seeded problem: packed varlen Q/K, metadata, hidden rows and positions."""

    name: str
    q_bits: np.ndarray            # uint16 [Tq, H, d]   bf16 bits
    k_bits: np.ndarray            # uint16 [Tk, Hkv, d] bf16 bits
    cu_seqlens_q: np.ndarray      # int32 [G+1]
    cu_seqlens_k: np.ndarray      # int32 [G+1]
    req_tok_offsets: np.ndarray   # int32 [R+1], offsets into the key tokens
    keep_per_req: np.ndarray      # int32 [R]
    hidden_bits: np.ndarray       # uint16 [Tk, D] bf16 bits
    pos: np.ndarray               # int32 [Tk, P]
    softmax_scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_heads(self) -> int:
        return int(self.q_bits.shape[1])

    @property
    def num_kv_heads(self) -> int:
        return int(self.k_bits.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.q_bits.shape[2])

    @property
    def num_seg(self) -> int:
        return int(self.cu_seqlens_k.shape[0] - 1)

    @property
    def total_q(self) -> int:
        return int(self.q_bits.shape[0])

    @property
    def total_k(self) -> int:
        return int(self.k_bits.shape[0])

    @property
    def max_seqlen_q(self) -> int:
        return int(np.diff(self.cu_seqlens_q).max(initial=0))

    @property
    def max_seqlen_k(self) -> int:
        return int(np.diff(self.cu_seqlens_k).max(initial=0))

    @property
    def total_keep(self) -> int:
        return int(self.keep_per_req.sum())

    def attended_pairs(self) -> int:
        """Number of (head, query, key) pairs inside the block-diagonal mask."""
        nq = np.diff(self.cu_seqlens_q).astype(np.int64)
        nk = np.diff(self.cu_seqlens_k).astype(np.int64)
        return int(self.num_heads * (nq * nk).sum())


def _normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def _pos_index(total: int) -> np.ndarray:
    return np.arange(total, dtype=np.int32).reshape(total, 1)


def _pos_grid(cu: np.ndarray, row_width: int = 64) -> np.ndarray:
    """(image, row, col) per token for pos_dim 3."""
    total = int(cu[-1])
    out = np.empty((total, 3), dtype=np.int32)
    for g in range(cu.shape[0] - 1):
        lo, hi = int(cu[g]), int(cu[g + 1])
        i = np.arange(hi - lo, dtype=np.int32)
        out[lo:hi, 0] = g
        out[lo:hi, 1] = i // row_width
        out[lo:hi, 2] = i % row_width
    return out


def _sink_rows(rng: np.random.Generator, cu: np.ndarray, counts) -> np.ndarray:
    """Global row indices of sink keys, drawn without replacement per segment."""
    rows = []
    for g in range(cu.shape[0] - 1):
        lo, hi = int(cu[g]), int(cu[g + 1])
        n = int(counts[g])
        if n > 0 and hi > lo:
            rows.append(lo + rng.choice(hi - lo, size=min(n, hi - lo), replace=False))
    return np.concatenate(rows).astype(np.int64) if rows else np.zeros(0, np.int64)


def make_segments(lengths_q, lengths_k, num_heads, num_kv_heads, head_dim, *,
                  seed, q_std=1.0, k_std=1.0, sink_counts=None, sink_factor=4.0,
                  key_scales=None, hidden_dim=64, pos_dim=1, requests=None,
                  keep_per_req=None, name="custom", softmax_scale=None) -> Workload:
    """Build a packed varlen workload from per-segment lengths.

    ``requests`` lists how many consecutive segments form each request (one
    request holding every segment by default). ``keep_per_req`` defaults to
    half of each request's tokens.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    lq = np.asarray(lengths_q, dtype=np.int64)
    lk = np.asarray(lengths_k, dtype=np.int64)
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    G = lk.shape[0]
    sinks = _sink_rows(rng, cu_k, sink_counts if sink_counts is not None else np.zeros(G, np.int64))
    q = _normal_f32(rng, (tq, num_heads, head_dim)) * np.float32(q_std)
    k = _normal_f32(rng, (tk, num_kv_heads, head_dim)) * np.float32(k_std)
    if key_scales is not None:
        row_scale = np.repeat(np.asarray(key_scales, dtype=np.float32), lk)
        k *= row_scale[:, None, None]
    if sinks.size:
        k[sinks] *= np.float32(sink_factor)
    hidden = _normal_f32(rng, (tk, hidden_dim))
    if requests is None:
        requests = [G]
    seg_cuts = np.concatenate([[0], np.cumsum(requests)]).astype(np.int64)
    assert seg_cuts[-1] == G
    req_off = cu_k[seg_cuts].astype(np.int32)
    n_req = np.diff(req_off).astype(np.int64)
    if keep_per_req is None:
        keep_per_req = n_req // 2
    keep = np.asarray(keep_per_req, dtype=np.int32)
    pos = _pos_index(tk) if pos_dim == 1 else _pos_grid(cu_k)
    return Workload(
        name=name,
        q_bits=f32_to_bf16_bits(q),
        k_bits=f32_to_bf16_bits(k),
        cu_seqlens_q=cu_q,
        cu_seqlens_k=cu_k,
        req_tok_offsets=req_off,
        keep_per_req=keep,
        hidden_bits=f32_to_bf16_bits(hidden),
        pos=pos,
        softmax_scale=float(softmax_scale if softmax_scale is not None else 1.0 / np.sqrt(head_dim)),
        meta={"seed": seed, "sink_rows": sinks},
    )


def make_far_keys(lengths, num_heads, num_kv_heads, head_dim, *, seed, far_positions,
                  far_value, head_signs, noise=0.1, q_lead=4.0, name="far_keys") -> Workload:
    """Self-attention segments whose logits climb far above the first keys.

    Every Q and K entry is N(0, noise^2); query rows of head h add
    ``q_lead * head_signs[h]`` to dimension 0, and the keys at the local
    positions ``far_positions`` of every segment (those that exist) have
    dimension 0 set to ``far_value`` on every KV head. With the default
    1/sqrt(d) scale, such a key's logit is about
    ``q_lead * far_value / sqrt(d) * sign`` while every other logit stays
    within a few tenths of zero — a controlled gap between the largest logit
    of a row and the largest logit among its first keys.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    lk = np.asarray(lengths, dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    t = int(cu[-1])
    q = _normal_f32(rng, (t, num_heads, head_dim)) * np.float32(noise)
    k = _normal_f32(rng, (t, num_kv_heads, head_dim)) * np.float32(noise)
    q[:, :, 0] += np.float32(q_lead) * np.asarray(head_signs, dtype=np.float32)[None, :]
    for g in range(lk.shape[0]):
        for p in far_positions:
            if p < lk[g]:
                k[cu[g] + p, :, 0] = np.float32(far_value)
    hidden = _normal_f32(rng, (t, 16))
    req_off = np.array([0, t], dtype=np.int32)
    return Workload(
        name=name,
        q_bits=f32_to_bf16_bits(q),
        k_bits=f32_to_bf16_bits(k),
        cu_seqlens_q=cu,
        cu_seqlens_k=cu.copy(),
        req_tok_offsets=req_off,
        keep_per_req=np.array([t // 2], dtype=np.int32),
        hidden_bits=f32_to_bf16_bits(hidden),
        pos=_pos_index(t),
        softmax_scale=float(1.0 / np.sqrt(head_dim)),
        meta={"seed": seed, "far_positions": list(far_positions), "far_value": far_value},
    )


def first_images(w: "Workload", n_images: int, keep_permille: int = 600) -> "Workload":
    """The first n_images segments of a workload as one request keeping
    floor(keep_permille / 1000 of its tokens) (a smaller case of the same
    shapes, e.g. for profiling)."""
    g = max(1, min(int(n_images), w.num_seg))
    q1, k1 = int(w.cu_seqlens_q[g]), int(w.cu_seqlens_k[g])
    return Workload(name=f"{w.name}[:{g}]", q_bits=w.q_bits[:q1], k_bits=w.k_bits[:k1],
                    cu_seqlens_q=w.cu_seqlens_q[:g + 1].copy(),
                    cu_seqlens_k=w.cu_seqlens_k[:g + 1].copy(),
                    req_tok_offsets=np.array([0, k1], dtype=np.int32),
                    keep_per_req=np.array([keep_floor(k1, keep_permille)], dtype=np.int32),
                    hidden_bits=w.hidden_bits[:k1], pos=w.pos[:k1],
                    softmax_scale=w.softmax_scale, meta=dict(w.meta, first_images=g))


def keep_floor(n: int, permille: int) -> int:
    """floor(n * permille / 1000) in integer arithmetic (budget rounding)."""
    return (int(n) * int(permille)) // 1000


def _quantise_tensor_e4m3(bits: np.ndarray, chunk: int = 1 << 23):
    """bf16 tensor -> (E4M3 bits, scale) with amax mapped to 448, in chunks."""
    flat = bits.reshape(-1)
    amax = 0.0
    for i in range(0, flat.size, chunk):
        amax = max(amax, float(np.abs(bf16_bits_to_f32(flat[i:i + chunk])).max(initial=0.0)))
    scale = max(amax, 1e-30) / 448.0
    inv = np.float32(1.0 / scale)
    out = np.empty(flat.size, dtype=np.uint8)
    for i in range(0, flat.size, chunk):
        out[i:i + chunk] = f32_to_e4m3_bits(bf16_bits_to_f32(flat[i:i + chunk]) * inv)
    return out.reshape(bits.shape), scale


def to_e4m3(w: "Workload") -> "Workload":
    """The same problem with Q and K quantised to FP8 E4M3 with one scale per
    tensor (amax maps to 448); the scales are folded into softmax_scale."""
    qb, sq = _quantise_tensor_e4m3(w.q_bits)
    kb, sk = _quantise_tensor_e4m3(w.k_bits)
    meta = dict(w.meta)
    meta.update(fmt="e4m3", q_scale=sq, k_scale=sk)
    return Workload(name=w.name + "_e4m3", q_bits=qb, k_bits=kb, cu_seqlens_q=w.cu_seqlens_q,
                    cu_seqlens_k=w.cu_seqlens_k, req_tok_offsets=w.req_tok_offsets,
                    keep_per_req=w.keep_per_req, hidden_bits=w.hidden_bits, pos=w.pos,
                    softmax_scale=w.softmax_scale * sq * sk, meta=meta)


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

def single_image_256() -> Workload:
    """One 256-token image, self-attention, H=4, d=64, entries N(0,1)/8, 4 sinks."""
    seed = SEED_BASE + 1
    return make_segments([256], [256], 4, 4, 64, seed=seed, q_std=1 / 8, k_std=1 / 8,
                         sink_counts=[4], hidden_dim=256, pos_dim=1, keep_per_req=[64],
                         name="single_image_256")


def six_views_1536() -> Workload:
    """Six 256-token camera views, block-diagonal self-attention, H=16, d=64."""
    seed = SEED_BASE + 2
    L = [256] * 6
    sinks = [int(0.02 * 256)] * 6
    return make_segments(L, L, 16, 16, 64, seed=seed, sink_counts=sinks, hidden_dim=1024,
                         pos_dim=1, keep_per_req=[keep_floor(1536, 800)],
                         name="six_views_1536")


def text_query_3072() -> Workload:
    """142 text queries over 3072 visual keys, GQA 16/8, d=128, keep 858."""
    seed = SEED_BASE + 3
    return make_segments([142], [3072], 16, 8, 128, seed=seed, hidden_dim=2048, pos_dim=1,
                         keep_per_req=[858], name="text_query_3072")


def thirty_images(seed_offset: int = 4) -> Workload:
    """30 images of U{256..4096} tokens, H=16, d=80, 1-8% sinks, key scale U(0.5,2), keep 60%."""
    seed = SEED_BASE + seed_offset
    rng = np.random.Generator(np.random.PCG64(seed ^ 0x5EED))
    L = rng.integers(256, 4096, size=30, endpoint=True)
    frac = rng.uniform(0.01, 0.08, size=30)
    sinks = np.maximum(1, np.floor(frac * L)).astype(np.int64)
    scales = rng.uniform(0.5, 2.0, size=30)
    n = int(L.sum())
    return make_segments(L, L, 16, 16, 80, seed=seed, sink_counts=sinks, key_scales=scales,
                         hidden_dim=1280, pos_dim=3, keep_per_req=[keep_floor(n, 600)],
                         name="thirty_images")


def batch_8x16x1024(ratios_permille=(500, 600, 700, 800)) -> Workload:
    """8 requests x 16 images x 1024 tokens, H=16, d=80, 2% sinks, per-request keep ratio."""
    seed = SEED_BASE + 5
    L = [1024] * 128
    sinks = [int(0.02 * 1024)] * 128
    keep = [keep_floor(16 * 1024, ratios_permille[r % len(ratios_permille)]) for r in range(8)]
    return make_segments(L, L, 16, 16, 80, seed=seed, sink_counts=sinks, hidden_dim=1280,
                         pos_dim=3, requests=[16] * 8, keep_per_req=keep, name="batch_8x16x1024")


WORKLOADS = {
    "single_image_256": single_image_256,
    "six_views_1536": six_views_1536,
    "text_query_3072": text_query_3072,
    "thirty_images": thirty_images,
    "batch_8x16x1024": batch_8x16x1024,
}


def make(name: str) -> Workload:
    return WORKLOADS[name]()
