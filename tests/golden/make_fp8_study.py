#!/usr/bin/env python3
"""Writes tests/golden/fp8_study.json: what FP8 (E4M3) quantisation of Q and K
does to the importance scores and to the keep decision, on every seeded
workload, measured with the fp64 oracle alone.

The LiteVLM paper review (section 5, results table: the FP8 row at r = 0.9,
and the FP8 deployment paragraph) runs the token selection under FP8. For
each workload this script quantises Q and K to E4M3 with one scale per tensor
(amax maps to 448, the scales folded into the softmax scale; the recipe of
workloads.to_e4m3) and compares the oracle's scores on the E4M3 inputs with
the oracle's scores on the original bf16 inputs:

  eps_max / eps_median   max and median of |s_e4m3 / s_bf16 - 1| over tokens
  kept                   total budget sum B
  flips                  tokens kept by exactly one of the two keep sets
                         (each keep set: top-B of its own scores, ties to the
                         lowest index; symmetric difference)
  agreement              |kept by both| / sum B
  flip_band_max          max over flipped tokens of |s_bf16 - s_bf16_B| / s_bf16_B
                         (s_bf16_B: the request's B-th largest bf16 score)
  flips_outside_2e-3     flipped tokens farther than 2e-3 from s_bf16_B
  near_e4m3_4e-3         tokens whose E4M3 score lies within 4e-3 of the
                         request's B-th E4M3 score (a GPU path within 2e-3 of
                         the E4M3 oracle can flip at most these on top)

Only oracle/ (and the seeded input generators) is called. Run from the
repository root: python tests/golden/make_fp8_study.py
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
for p in (ROOT, os.path.dirname(HERE)):
    if p not in sys.path:
        sys.path.insert(0, p)


def bth_scores(scores, off, keep):
    """Per token: the B-th largest score of its request (nan where B is 0)."""
    out = np.full(scores.shape, np.nan)
    for r in range(len(off) - 1):
        lo, hi, B = int(off[r]), int(off[r + 1]), int(keep[r])
        if B > 0:
            out[lo:hi] = np.sort(scores[lo:hi])[::-1][B - 1]
    return out


def study(w, s16, s8):
    import oracle
    nz = s16 > 0
    rel = np.abs(s8[nz] / s16[nz] - 1.0)
    k16, _ = oracle.select_topk(s16, w.req_tok_offsets, w.keep_per_req)
    k8, _ = oracle.select_topk(s8, w.req_tok_offsets, w.keep_per_req)
    a, b = set(k16.tolist()), set(k8.tolist())
    flips = np.array(sorted(a ^ b), dtype=np.int64)
    b16 = bth_scores(s16, w.req_tok_offsets, w.keep_per_req)
    b8 = bth_scores(s8, w.req_tok_offsets, w.keep_per_req)
    band = np.abs(s16[flips] - b16[flips]) / b16[flips] if flips.size else np.zeros(0)
    near = np.abs(s8 - b8) <= 4e-3 * b8
    # requests that keep every token (or none) cannot flip
    full = np.zeros(s8.shape, bool)
    for r in range(len(w.req_tok_offsets) - 1):
        lo, hi = int(w.req_tok_offsets[r]), int(w.req_tok_offsets[r + 1])
        if int(w.keep_per_req[r]) in (0, hi - lo):
            full[lo:hi] = True
    return {
        "tokens": int(w.total_k),
        "kept": int(w.total_keep),
        "eps_max": float(rel.max(initial=0.0)),
        "eps_median": float(np.median(rel)) if rel.size else 0.0,
        "flips": int(flips.size),
        "agreement": float(len(a & b) / max(1, w.total_keep)),
        "flip_band_max": float(band.max(initial=0.0)),
        "flips_outside_2e-3": int(np.sum(band > 2e-3)),
        "near_e4m3_4e-3": int(np.sum(near & ~full)),
    }


def main():
    import workloads as W
    from oracle_pool import importance_by_segment
    out = {"_note": __doc__.split("\n\n")[1].replace("\n", " ").strip(),
           "recipe": "workloads.to_e4m3 (one scale per tensor, amax -> 448) against the bf16 "
                     "inputs; fp64 oracle on both",
           "workloads": {}}
    for name in W.WORKLOADS:
        w = W.make(name)
        w8 = W.to_e4m3(w)
        _, s16 = importance_by_segment(w)
        _, s8 = importance_by_segment(w8, softmax_scale=w8.softmax_scale, fmt="e4m3")
        out["workloads"][name] = study(w, s16, s8)
        print(name, out["workloads"][name], flush=True)
    with open(os.path.join(HERE, "fp8_study.json"), "w") as fh:
        json.dump(out, fh, indent=1)
        fh.write("\n")


if __name__ == "__main__":
    main()
