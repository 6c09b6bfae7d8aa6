"""GPU parity on seeded random problems: segment counts on both sides of the
one-warp schedule path (32 segments), empty, one-token and ragged segments,
self- and cross-attention lengths, every head_dim, GQA ratios, explicit
scales, several requests per call, random budgets — each compared with the
fp64 oracle (scores, LSE) and bit for bit on the selection and compaction fed
the same fp32 scores; the dynamic budget and the LSE-provided mode ride
along. A second set draws request layouts for the selection kernels alone
(one to sixty requests of up to 100K tokens, so every cluster size occurs)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import (REL_TOL, bits_to_bf16, check_selection_exact, i32, max_rel_err, run_path,
                      to_device)

pytestmark = pytest.mark.gpu

HEADS = [(1, 1), (2, 1), (4, 2), (6, 3), (8, 8), (12, 4), (16, 2), (3, 3)]
DIMS = [64, 80, 96, 112, 128]


@pytest.fixture(scope="module")
def tsel():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_score_vision_gb300 as t
    t.build()
    t.load_library()
    return t


def _random_problem(seed):
    rng = np.random.default_rng(seed)
    G = int(rng.choice([1, 2, 5, 17, 31, 32, 33, 45]))
    H, Hkv = HEADS[int(rng.integers(len(HEADS)))]
    d = int(rng.choice(DIMS))
    kind = rng.random()
    lk = rng.choice([0, 1, 2, 31, 127, 128, 129, 200, 255, 256, 257, 400], size=G)
    if kind < 0.5:
        lq = lk.copy()                                    # self-attention
    else:
        lq = rng.choice([0, 1, 5, 64, 130, 300], size=G)  # cross lengths
    # keep the oracle's work bounded
    while int(np.sum(lq * lk)) * H > 6_000_000:
        i = int(np.argmax(lq * lk))
        lk[i] //= 2
        lq[i] //= 2
    # requests: consecutive groups of segments
    cuts = sorted(set(rng.choice(np.arange(1, G), size=min(G - 1, int(rng.integers(0, 4))),
                                 replace=False).tolist())) if G > 1 else []
    groups = np.diff([0] + cuts + [G]).tolist()
    n_req = np.add.reduceat(lk, np.concatenate([[0], np.cumsum(groups)[:-1]])) if G else []
    keep = [int(rng.integers(0, n + 1)) for n in n_req]
    scale = float(rng.choice([0.0, 0.05, 0.3]))
    w = W.make_segments(lq, lk, H, Hkv, d, seed=10_000 + seed, q_std=float(rng.choice([0.2, 1.0, 2.0])),
                        sink_counts=rng.integers(0, 3, size=G), hidden_dim=int(rng.choice([64, 128])),
                        requests=groups, keep_per_req=keep, name=f"fuzz{seed}",
                        softmax_scale=scale if scale > 0 else None)
    return w, scale


@pytest.mark.parametrize("seed", range(24))
def test_random_problem_matches_oracle(tsel, seed):
    w, scale = _random_problem(seed)
    out = run_path(tsel, w, softmax_scale=scale)
    assert out["status"] == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                       softmax_scale=scale if scale > 0 else None)
    assert max_rel_err(out["scores"], s_ref) <= REL_TOL
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(out["lse"][~fin]))
    np.testing.assert_allclose(out["lse"][fin], lse_ref[fin], rtol=1e-5, atol=2e-4)
    check_selection_exact(w, out)
    # the dynamic budget on the same fp32 scores
    s32 = out["scores"].astype(np.float32)
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    keep, total = tsel.tsel_dynamic_budget(torch.from_numpy(s32).cuda(), i32(w.req_tok_offsets),
                                           850, 50, 950, workspace=ws)
    ref = oracle.dynamic_budget(s32, w.req_tok_offsets, 850, 50, 950)
    assert keep.cpu().tolist() == ref.tolist()
    assert int(total.item()) == int(ref.sum())


@pytest.mark.parametrize("seed", range(24, 30))
def test_random_problem_lse_provided(tsel, seed):
    w, scale = _random_problem(seed)
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                       softmax_scale=scale if scale > 0 else None)
    d = to_device(w)
    lse_in = torch.from_numpy(lse_ref.astype(np.float32)).cuda()
    s, _ = tsel.tsel_importance(d["q"], d["k"], d["cu_q"], d["cu_k"], max(w.max_seqlen_q, 1),
                                max(w.max_seqlen_k, 1), softmax_scale=scale,
                                flags=tsel.TSEL_IMP_LSE_PROVIDED, lse=lse_in)
    assert max_rel_err(s.cpu().numpy(), s_ref) <= REL_TOL


def _random_selection_problem(seed):
    """Random request layouts for the selection kernels alone: from one to
    sixty requests, each empty to 100K tokens (so every cluster size and
    slices of every length occur), score sets with heavy ties, signed zeros
    and values over many binades."""
    rng = np.random.default_rng(50_000 + seed)
    R = int(rng.choice([1, 2, 3, 8, 13, 60]))
    big = rng.random() < 0.5
    sizes = rng.integers(0, 100_000 if big else 5_000, size=R)
    if rng.random() < 0.3:
        sizes[rng.integers(R)] = 0
    n = int(sizes.sum())
    kind = int(rng.integers(4))
    if kind == 0:
        s = rng.random(n)
    elif kind == 1:
        s = rng.integers(0, 5, n) * 0.125                     # five values: ties everywhere
    elif kind == 2:
        s = np.exp2(rng.uniform(-60, 10, n))                  # many binades
    else:
        s = rng.exponential(1e-4, n)                          # attention-like
    s = s.astype(np.float32)
    if n:
        s[rng.integers(0, n, n // 50 + 1)] = np.float32(0.0)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64).tolist()
    keep = [int(rng.integers(0, int(z) + 1)) for z in sizes]
    return s, off, keep


@pytest.mark.parametrize("seed", range(24))
def test_random_selection_layouts(tsel, seed):
    s, off, keep = _random_selection_problem(seed)
    sd = torch.from_numpy(s).cuda()
    ws = torch.zeros(tsel.tsel_select_topk_workspace_size(len(keep)), dtype=torch.uint8, device="cuda")
    ki, cu = tsel.tsel_select_topk(sd, i32(off), i32(keep), int(sum(keep)), workspace=ws)
    ref, cref = oracle.select_topk(s, off, keep)
    assert tsel.tsel_read_device_status(ws) == 0
    assert np.array_equal(ki.cpu().numpy(), ref) and np.array_equal(cu.cpu().numpy(), cref)
    # the histogram-started top-B (candidate exchange, ranking or 8-bit rounds,
    # or its fallbacks, whichever the layout calls for) on the same layout
    wsh = torch.zeros(tsel.tsel_select_topk_hist_workspace_size(len(keep)), dtype=torch.uint8,
                      device="cuda")
    kh, ch = tsel.tsel_select_topk_hist(sd, i32(off), i32(keep), int(sum(keep)), workspace=wsh)
    assert tsel.tsel_read_device_status(wsh) == 0
    assert np.array_equal(kh.cpu().numpy(), ref) and np.array_equal(ch.cpu().numpy(), cref)
    # the dynamic budget on the same layout, and the device-count selection it feeds
    rng = np.random.default_rng(seed)
    tau, lo = int(rng.choice([1, 300, 900, 1000])), int(rng.choice([0, 100]))
    hi = int(rng.choice([lo, 900, 1000]))
    bk, bt = tsel.tsel_dynamic_budget(sd, i32(off), tau, lo, hi, workspace=ws)
    bref = oracle.dynamic_budget(s, off, tau, lo, hi)
    assert tsel.tsel_read_device_status(ws) == 0
    assert np.array_equal(bk.cpu().numpy(), bref) and int(bt.item()) == int(bref.sum())
    ki2, cu2 = tsel.tsel_select_topk(sd, i32(off), bk, tsel.TSEL_KEEP_FROM_DEVICE, workspace=ws)
    ref2, cref2 = oracle.select_topk(s, off, bref)
    n_kept = int(cu2[-1].item())
    assert n_kept == int(bref.sum())
    assert np.array_equal(ki2[:n_kept].cpu().numpy(), ref2) and np.array_equal(cu2.cpu().numpy(), cref2)
