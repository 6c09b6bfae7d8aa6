"""GPU: SUM score normalisation, the mass-based dynamic keep budget, and the
device-count path (budget -> top-B -> compaction with no host round trip).

The budget is an integer decided from fp32 scores: both sides decide it on the
same fp32 scores (the GPU's), so it must match the oracle exactly; the keep
set and the compacted rows then must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import REL_TOL, bits_to_bf16, i32, max_rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsel():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_score_vision_gb300 as t
    t.build()
    t.load_library()
    return t


def _budget(tsel, scores_np, offsets, tau, lo, hi):
    s = torch.from_numpy(np.ascontiguousarray(scores_np, dtype=np.float32)).cuda()
    off = i32(offsets)
    ws = torch.zeros(tsel.tsel_select_topk_workspace_size(len(offsets) - 1), dtype=torch.uint8,
                     device="cuda")
    keep, total = tsel.tsel_dynamic_budget(s, off, tau, lo, hi, workspace=ws)
    return keep.cpu().numpy(), int(total.item()), tsel.tsel_read_device_status(ws)


def _score_sets():
    rng = np.random.default_rng(900)
    sets = []
    # attention-like: heavy tail, a few dominant tokens, many near-ties
    a = (rng.random(5000) ** 6).astype(np.float32) * np.float32(1e-2)
    a[rng.choice(5000, 40, replace=False)] *= np.float32(50.0)
    sets.append(("heavy_tail", a, [0, 1000, 1000, 3500, 5000]))
    # few distinct values (ties everywhere), zeros and -0
    b = rng.choice(np.asarray([0.0, -0.0, 0.125, 0.25, 0.25, 0.5], np.float32), 3000)
    sets.append(("ties", b, [0, 3000]))
    # uniform and one-hot requests side by side
    c = np.concatenate([np.full(777, 1.0 / 777, np.float32), np.zeros(100, np.float32)])
    c[777 + 42] = np.float32(0.7)
    sets.append(("uniform_onehot", c, [0, 777, 877]))
    # subnormal and tiny scores
    d = np.concatenate([np.asarray([1e-40, 3e-42, 0.0, 2e-39], np.float32),
                        (rng.random(500) * 1e-30).astype(np.float32)])
    sets.append(("tiny", d, [0, 4, 504]))
    # one large request across many blocks
    e = rng.exponential(1e-4, 70000).astype(np.float32)
    sets.append(("large", e, [0, 70000]))
    # clusters of 4 and 8 CTAs (average request 10K and 20K tokens); slices
    # longer than the per-CTA key cache (300K tokens on 16 CTAs)
    f = (rng.random(40000) ** 3).astype(np.float32) * np.float32(3e-3)
    sets.append(("clusters4", f, [0, 9000, 20000, 30001, 40000]))
    sets.append(("clusters8", f, [0, 17000, 40000]))
    h = rng.exponential(1e-5, 300000).astype(np.float32)
    sets.append(("uncached", h, [0, 300000]))
    return sets


@pytest.mark.parametrize("tau,lo,hi", [(0, 0, 1000), (1, 0, 1000), (500, 0, 1000),
                                       (900, 100, 900), (999, 0, 1000), (1000, 0, 1000),
                                       (800, 600, 600)])
def test_dynamic_budget_matches_oracle_exactly(tsel, tau, lo, hi):
    for name, s, off in _score_sets():
        keep, total, st = _budget(tsel, s, off, tau, lo, hi)
        ref = oracle.dynamic_budget(s, off, tau, lo, hi)
        assert st == 0, name
        assert keep.tolist() == ref.tolist(), (name, tau, lo, hi)
        assert total == int(ref.sum())


def test_dynamic_budget_slice_past_two_to_the_twenty(tsel):
    # 300 small requests and one of 1.1M tokens: the average request is small,
    # so one CTA holds every key of the large one (more than 2^20, past its
    # key cache: every round re-reads the scores), and its per-bin quanta sums
    # pass 2^32
    rng = np.random.default_rng(902)
    sizes = [1_100_000] + rng.integers(1, 40, 300).tolist()
    off = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    s = rng.exponential(1e-6, off[-1]).astype(np.float32)
    keep, total, st = _budget(tsel, s, off, 900, 0, 1000)
    ref = oracle.dynamic_budget(s, off, 900, 0, 1000)
    assert st == 0
    assert np.array_equal(keep, ref) and total == int(ref.sum())


def test_dynamic_budget_many_large_requests(tsel):
    # twelve 40K-token requests (more than the device holds clusters of 16)
    rng = np.random.default_rng(903)
    off = (np.arange(13) * 40000).tolist()
    s = (rng.random(off[-1]) ** 4).astype(np.float32) * np.float32(1e-3)
    keep, total, st = _budget(tsel, s, off, 800, 50, 950)
    ref = oracle.dynamic_budget(s, off, 800, 50, 950)
    assert st == 0
    assert np.array_equal(keep, ref) and total == int(ref.sum())


def test_dynamic_budget_flags_nan_and_bad_offsets(tsel):
    s = np.asarray([0.5, np.nan, 0.25, 0.125], np.float32)
    keep, _, st = _budget(tsel, s, [0, 4], 1000, 0, 1000)
    assert st & tsel.TSEL_DEV_NAN
    # NaN adds no quantum; its rank is unspecified (as in the top-B), so it
    # may or may not sit in front of the three tokens that hold the mass
    assert keep.tolist() in ([3], [4])
    keep, _, st = _budget(tsel, np.ones(8, np.float32), [0, 5, 3, 8], 500, 0, 1000)
    assert st & tsel.TSEL_DEV_REQUESTS
    assert keep[1] == 0


def test_sum_normalisation_matches_oracle(tsel):
    w = W.make_segments([300, 0, 129], [257, 40, 500], 8, 2, 64, seed=901, sink_counts=[3, 1, 9],
                        hidden_dim=64)
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    cq, ck = i32(w.cu_seqlens_q), i32(w.cu_seqlens_k)
    s_sum, _ = tsel.tsel_importance(q, k, cq, ck, 300, 500, flags=tsel.TSEL_IMP_SCORE_SUM)
    s_mean, _ = tsel.tsel_importance(q, k, cq, ck, 300, 500)
    _, ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k, norm="sum")
    got = s_sum.cpu().numpy()
    assert max_rel_err(got, ref) <= REL_TOL
    # sum = mean x H x Nq_g (same partial sums, one fp32 division apart)
    mean = s_mean.cpu().numpy().astype(np.float64)
    nq = np.repeat(np.diff(w.cu_seqlens_q), np.diff(w.cu_seqlens_k)).astype(np.float64)
    np.testing.assert_allclose(got.astype(np.float64), mean * 8 * nq, rtol=1e-6, atol=0)


def _device_count_path(tsel, w, d, tau, lo, hi, flags=0):
    G, Tq, Tk, H = w.num_seg, w.total_q, w.total_k, w.num_heads
    ws = torch.zeros(tsel.tsel_importance_workspace_size(G, Tq, Tk, H), dtype=torch.uint8,
                     device="cuda")
    scores, _ = tsel.tsel_importance(d["q"], d["k"], d["cu_q"], d["cu_k"], w.max_seqlen_q,
                                     w.max_seqlen_k, flags=flags, workspace=ws, want_lse=False)
    keep, total = tsel.tsel_dynamic_budget(scores, d["req_off"], tau, lo, hi, workspace=ws)
    keep_idx, cu_keep = tsel.tsel_select_topk(scores, d["req_off"], keep,
                                              tsel.TSEL_KEEP_FROM_DEVICE, workspace=ws)
    R = keep.numel()
    oh, op, oi, oc = tsel.tsel_gather_compact_counted(d["hidden"], d["pos"], d["cu_k"], keep_idx,
                                                      cu_keep[R:], Tk, workspace=ws)
    status = tsel.tsel_read_device_status(ws)
    n = int(total.item())
    return {"scores": scores.cpu().numpy(), "keep": keep.cpu().numpy(), "total": n,
            "keep_idx": keep_idx[:n].cpu().numpy(), "cu_keep": cu_keep.cpu().numpy(),
            "hidden": oh[:n].view(torch.int16).cpu().numpy().view(np.uint16),
            "pos": op[:n].cpu().numpy(), "img_id": oi[:n].cpu().numpy(),
            "cu_kept": oc.cpu().numpy(), "status": status}


@pytest.mark.parametrize("name,tau,lo,hi,flags", [("six_views_1536", 900, 100, 900, 0),
                                                  ("text_query_3072", 800, 0, 1000, 0),
                                                  ("six_views_1536", 500, 0, 1000, 0x4)])
def test_dynamic_path_bit_exact_given_the_gpu_scores(tsel, name, tau, lo, hi, flags):
    w = W.make(name)
    d = to_device(w)
    out = _device_count_path(tsel, w, d, tau, lo, hi, flags)
    assert out["status"] == 0
    _, ref_scores = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                      norm="sum" if flags & 0x4 else "mean")
    assert max_rel_err(out["scores"], ref_scores) <= REL_TOL
    s32 = out["scores"]        # the integer decisions are taken on the same fp32 scores
    ref_keep = oracle.dynamic_budget(s32, w.req_tok_offsets, tau, lo, hi)
    assert out["keep"].tolist() == ref_keep.tolist()
    assert out["total"] == int(ref_keep.sum())
    ki, ck = oracle.select_topk(s32, w.req_tok_offsets, ref_keep)
    assert np.array_equal(out["keep_idx"], ki)
    assert np.array_equal(out["cu_keep"], ck)
    rh, rp, rimg, rcu = oracle.gather_compact(w.hidden_bits, w.pos, w.cu_seqlens_k, ki)
    assert np.array_equal(out["hidden"], rh)
    assert np.array_equal(out["pos"], rp)
    assert np.array_equal(out["img_id"], rimg)
    assert np.array_equal(out["cu_kept"], rcu)


def test_dynamic_path_on_the_thirty_image_request(tsel):
    """Full size: the budget, keep set and compaction checked exactly against
    the oracle's selection on the GPU's fp32 scores (the scores themselves are
    checked against the fp64 oracle by the parity tests)."""
    w = W.make("thirty_images")
    d = to_device(w)
    out = _device_count_path(tsel, w, d, 900, 100, 900)
    assert out["status"] == 0
    s32 = out["scores"]
    ref_keep = oracle.dynamic_budget(s32, w.req_tok_offsets, 900, 100, 900)
    assert out["keep"].tolist() == ref_keep.tolist()
    ki, _ = oracle.select_topk(s32, w.req_tok_offsets, ref_keep)
    assert np.array_equal(out["keep_idx"], ki)
    rh, rp, rimg, rcu = oracle.gather_compact(w.hidden_bits, w.pos, w.cu_seqlens_k, ki)
    assert np.array_equal(out["hidden"], rh)
    assert np.array_equal(out["img_id"], rimg)
    assert np.array_equal(out["cu_kept"], rcu)


def test_counted_gather_clamps_a_bad_count(tsel):
    hidden = torch.arange(64 * 8, dtype=torch.float32, device="cuda").view(64, 8)
    cu = i32([0, 64])
    keep_idx = i32(np.arange(0, 64, 2))
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    n = i32([40])   # more than max_kept = 32
    oh, _, oi, oc = tsel.tsel_gather_compact_counted(hidden, None, cu, keep_idx, n, 32, workspace=ws)
    assert tsel.tsel_read_device_status(ws) & tsel.TSEL_DEV_KEEP_IDX
    assert torch.equal(oh, hidden[0:64:2])
    assert oc.cpu().tolist() == [0, 32]


def test_dynamic_path_captures_into_a_cuda_graph(tsel):
    """Budget, top-B and compaction with device counts need no host round trip,
    so importance -> budget -> top-B -> compaction is one capturable sequence."""
    w = W.make("six_views_1536")
    d = to_device(w)
    G, Tq, Tk, H = w.num_seg, w.total_q, w.total_k, w.num_heads
    ws = torch.zeros(tsel.tsel_importance_workspace_size(G, Tq, Tk, H), dtype=torch.uint8,
                     device="cuda")
    scores = torch.empty(Tk, device="cuda")
    keep = torch.empty(1, dtype=torch.int32, device="cuda")
    total = torch.empty(1, dtype=torch.int32, device="cuda")
    keep_idx = torch.empty(Tk, dtype=torch.int32, device="cuda")
    cu_keep = torch.empty(2, dtype=torch.int32, device="cuda")
    oh = torch.empty((Tk, d["hidden"].shape[1]), dtype=torch.bfloat16, device="cuda")
    op = torch.empty((Tk, 1), dtype=torch.int32, device="cuda")
    oi = torch.empty(Tk, dtype=torch.int32, device="cuda")
    oc = torch.empty(G + 1, dtype=torch.int32, device="cuda")

    def path():
        tsel.tsel_importance(d["q"], d["k"], d["cu_q"], d["cu_k"], 256, 256, scores=scores,
                             workspace=ws, want_lse=False)
        tsel.tsel_dynamic_budget(scores, d["req_off"], 900, 100, 900, keep_per_req=keep,
                                 total_keep=total, workspace=ws)
        tsel.tsel_select_topk(scores, d["req_off"], keep, tsel.TSEL_KEEP_FROM_DEVICE,
                              keep_idx=keep_idx, cu_keep=cu_keep, workspace=ws)
        tsel.tsel_gather_compact_counted(d["hidden"], d["pos"], d["cu_k"], keep_idx, cu_keep[1:], Tk,
                                         out_hidden=oh, out_pos=op, out_img_id=oi,
                                         out_cu_seqlens=oc, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        path()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    n = int(total.item())
    ref = [t.clone() for t in (keep, keep_idx[:n], oh[:n], oc)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        path()
    for _ in range(3):
        for t in (keep_idx, oh, oc):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(total.item()) == n
        for a, b in zip(ref, (keep, keep_idx[:n], oh[:n], oc)):
            assert torch.equal(a, b)
    assert tsel.tsel_read_device_status(ws) == 0
