"""The fused score + select path (tsel_score_select) and the histogram-started
top-B (tsel_select_topk_hist) against the oracle and the separate calls.

The column pass counts each request's scores by the first 11 and 16 bits of
their order-preserving keys; the top-B starts from those counts. Whatever
path the top-B takes (candidate exchange, radix rounds from the second digit,
or from the first when the counts do not fit), the kept indices must equal
oracle.select_topk on the same fp32 scores, bit for bit. The path counters
show which path each request took, so every path is exercised on purpose.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import REL_TOL, check_selection_exact, i32, max_rel_err, to_device

pytestmark = pytest.mark.gpu

PLAIN, HIST_ROUNDS, CANDIDATES, REJECTED, IN_IMPORTANCE = range(5)


@pytest.fixture(scope="module")
def tsel():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_score_vision_gb300 as t
    t.build()
    t.load_library()
    return t


def _fused(tsel, w, dev, flags=0, lse_in=None, q=None, k=None, scale=0.0):
    R = w.keep_per_req.size
    ws = torch.zeros(tsel.tsel_score_select_workspace_size(w.num_seg, w.total_q, w.total_k,
                                                           w.num_heads, R),
                     dtype=torch.uint8, device="cuda")
    s, lse, kidx, cu = tsel.tsel_score_select(
        dev["q"] if q is None else q, dev["k"] if k is None else k, dev["cu_q"], dev["cu_k"],
        w.max_seqlen_q, w.max_seqlen_k, dev["req_off"], dev["keep"], w.total_keep, flags=flags,
        lse=lse_in, softmax_scale=scale, workspace=ws)
    st = tsel.tsel_read_device_status(ws)
    return s, lse, kidx, cu, st, tsel.tsel_select_path_counts(ws)


def _separate(tsel, w, dev, flags=0, lse_in=None, q=None, k=None, scale=0.0):
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k,
                                                         w.num_heads), dtype=torch.uint8,
                     device="cuda")
    s, lse = tsel.tsel_importance(dev["q"] if q is None else q, dev["k"] if k is None else k,
                                  dev["cu_q"], dev["cu_k"], w.max_seqlen_q, w.max_seqlen_k,
                                  flags=flags, lse=lse_in, softmax_scale=scale, workspace=ws)
    kidx, cu = tsel.tsel_select_topk(s, dev["req_off"], dev["keep"], w.total_keep, workspace=ws)
    st = tsel.tsel_read_device_status(ws)
    return s, lse, kidx, cu, st, tsel.tsel_select_path_counts(ws)


def _bits(t):
    return t.view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_fused_equals_separate_calls_and_oracle(tsel, name):
    w = W.make(name)
    dev = to_device(w)
    a = _fused(tsel, w, dev)
    b = _separate(tsel, w, dev)
    assert a[4] == 0 and b[4] == 0
    assert np.array_equal(_bits(a[0]), _bits(b[0]))         # scores
    assert np.array_equal(_bits(a[1]), _bits(b[1]))         # LSE
    assert np.array_equal(a[2].cpu().numpy(), b[2].cpu().numpy())
    assert np.array_equal(a[3].cpu().numpy(), b[3].cpu().numpy())
    k_ref, cu_ref = oracle.select_topk(a[0].cpu().numpy(), w.req_tok_offsets, w.keep_per_req)
    assert np.array_equal(a[2].cpu().numpy(), k_ref)
    assert np.array_equal(a[3].cpu().numpy(), cu_ref)
    R = w.keep_per_req.size
    assert b[5] == [R, 0, 0, 0, 0]                          # separate calls: no histograms
    if name in ("thirty_images", "batch_8x16x1024"):
        # requests split over clusters of CTAs start from the histograms
        assert a[5] == [0, 0, R, 0, 0], a[5]
    elif name == "single_image_256":
        # one image of 256 tokens: ranked inside the one-launch importance kernel
        assert a[5] == [0, 0, 0, 0, R], a[5]
    else:
        # one CTA per request: no histograms, plain radix rounds
        assert a[5] == [R, 0, 0, 0, 0], a[5]


def test_fused_lse_provided_and_fp8(tsel):
    w = W.make("thirty_images")
    dev = to_device(w)
    _, lse, *_ = _separate(tsel, w, dev)
    for flags in (tsel.TSEL_IMP_LSE_PROVIDED,):
        a = _fused(tsel, w, dev, flags=flags, lse_in=lse.clone())
        b = _separate(tsel, w, dev, flags=flags, lse_in=lse.clone())
        assert a[4] == 0 and b[4] == 0
        assert np.array_equal(_bits(a[0]), _bits(b[0]))
        assert np.array_equal(a[2].cpu().numpy(), b[2].cpu().numpy())
        assert a[5][CANDIDATES] == 1
    w8 = W.to_e4m3(w)
    q8, k8 = torch.from_numpy(w8.q_bits).cuda(), torch.from_numpy(w8.k_bits).cuda()
    a = _fused(tsel, w, dev, q=q8, k=k8, scale=w8.softmax_scale)
    b = _separate(tsel, w, dev, q=q8, k=k8, scale=w8.softmax_scale)
    assert a[4] == 0 and np.array_equal(_bits(a[0]), _bits(b[0]))
    assert np.array_equal(a[2].cpu().numpy(), b[2].cpu().numpy())


def test_fused_stages_run_apart(tsel):
    """Stage bits (as the benchmark times them): schedule, row-LSE pass, column
    pass, then the top-B alone, on one workspace."""
    w = W.make("thirty_images")
    dev = to_device(w)
    R = w.keep_per_req.size
    ws = torch.zeros(tsel.tsel_score_select_workspace_size(w.num_seg, w.total_q, w.total_k,
                                                           w.num_heads, R),
                     dtype=torch.uint8, device="cuda")
    scores = torch.empty(w.total_k, device="cuda")
    kidx = torch.empty(w.total_keep, dtype=torch.int32, device="cuda")
    cu = torch.empty(R + 1, dtype=torch.int32, device="cuda")
    for st in (tsel.TSEL_IMP_STAGE_PREP, tsel.TSEL_IMP_STAGE_PASS1, tsel.TSEL_IMP_STAGE_PASS2,
               tsel.TSEL_SEL_STAGE_TOPK):
        tsel.tsel_score_select(dev["q"], dev["k"], dev["cu_q"], dev["cu_k"], w.max_seqlen_q,
                               w.max_seqlen_k, dev["req_off"], dev["keep"], w.total_keep,
                               flags=st, scores=scores, keep_idx=kidx, cu_keep=cu, workspace=ws)
    assert tsel.tsel_read_device_status(ws) == 0
    assert tsel.tsel_select_path_counts(ws)[CANDIDATES] == R
    k_ref, _ = oracle.select_topk(scores.cpu().numpy(), w.req_tok_offsets, w.keep_per_req)
    assert np.array_equal(kidx.cpu().numpy(), k_ref)


def test_fused_mixed_segments_and_requests_vs_oracle(tsel):
    """Images of very different sizes in uneven requests (clusters of several
    sizes), scores against the fp64 oracle and selection bit-exact."""
    L = [1, 127, 128, 129, 300, 700, 1000, 64, 4096, 2, 2500, 900]
    w = W.make_segments(L, L, 8, 8, 80, seed=909, sink_counts=[0, 2, 3, 3, 6, 14, 20, 1, 40, 0, 9, 9],
                        key_scales=[1, 0.5, 2, 1, 1.5, 0.7, 1, 1.2, 1, 1, 0.8, 1.9],
                        hidden_dim=16, pos_dim=3, requests=[3, 1, 4, 1, 3],
                        keep_per_req=[100, 0, 1500, 2, 2000])
    dev = to_device(w)
    s, lse, kidx, cu, st, paths = _fused(tsel, w, dev)
    assert st == 0
    _, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s.cpu().numpy(), s_ref) <= REL_TOL
    out = {"scores": s.cpu().numpy(), "keep_idx": kidx.cpu().numpy(), "cu_keep": cu.cpu().numpy()}
    k_ref, cu_ref = oracle.select_topk(out["scores"], w.req_tok_offsets, w.keep_per_req)
    assert np.array_equal(out["keep_idx"], k_ref) and np.array_equal(out["cu_keep"], cu_ref)
    assert sum(paths) == 4          # the request with B = 0 returns before any path


def test_fused_malformed_requests_fall_back(tsel):
    """Request offsets out of order: no histograms; the top-B flags the bad
    requests exactly as the plain call does."""
    w = W.make("six_views_1536")
    dev = to_device(w)
    dev["req_off"] = i32([0, 800, 600, 1536])
    dev["keep"] = i32([10, 10, 10])
    w.keep_per_req = np.array([10, 10, 10], np.int32)
    a = _fused(tsel, w, dev)
    assert a[4] & tsel.TSEL_DEV_REQUESTS
    assert a[5][PLAIN] == 2   # the two valid requests, plain rounds


def test_fused_graph_capture(tsel):
    w = W.make("text_query_3072")
    dev = to_device(w)
    R = w.keep_per_req.size
    ws = torch.zeros(tsel.tsel_score_select_workspace_size(w.num_seg, w.total_q, w.total_k,
                                                           w.num_heads, R),
                     dtype=torch.uint8, device="cuda")
    scores = torch.empty(w.total_k, device="cuda")
    kidx = torch.empty(w.total_keep, dtype=torch.int32, device="cuda")
    cu = torch.empty(R + 1, dtype=torch.int32, device="cuda")

    def run(st):
        tsel.tsel_score_select(dev["q"], dev["k"], dev["cu_q"], dev["cu_k"], w.max_seqlen_q,
                               w.max_seqlen_k, dev["req_off"], dev["keep"], w.total_keep,
                               scores=scores, keep_idx=kidx, cu_keep=cu, workspace=ws, stream=st)
    run(None)
    torch.cuda.synchronize()
    ref = kidx.cpu().numpy().copy()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        run(side)
    torch.cuda.current_stream().wait_stream(side)
    kidx.fill_(-1)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(kidx.cpu().numpy(), ref)
    assert tsel.tsel_read_device_status(ws) == 0


# --------------------------------------------- histogram start on given scores

def _topk_hist(tsel, scores, off, keep, total_keep=None):
    R = len(keep)
    ws = torch.zeros(tsel.tsel_select_topk_hist_workspace_size(R), dtype=torch.uint8,
                     device="cuda")
    tk = int(np.sum(keep)) if total_keep is None else total_keep
    k_idx, cu = tsel.tsel_select_topk_hist(torch.from_numpy(np.asarray(scores, np.float32)).cuda(),
                                           i32(off), i32(keep), tk, workspace=ws)
    return (k_idx.cpu().numpy(), cu.cpu().numpy(), tsel.tsel_read_device_status(ws),
            tsel.tsel_select_path_counts(ws))


def _check(got, cu, s, off, keep):
    clean = np.where(s == 0, 0.0, s).astype(np.float32)   # -0 ranks as +0
    ref, cref = oracle.select_topk(clean, off, keep)
    assert np.array_equal(got[:ref.size], ref)
    assert np.array_equal(cu, cref)


@pytest.mark.parametrize("n", [1, 5, 1000, 9000, 40000, 70000, 300000])
def test_hist_start_random_scores(tsel, n):
    # log-uniform over 20 binades: a few hundred keys per 16-bit bin at most
    rng = np.random.default_rng(n)
    s = np.exp2(rng.uniform(-20, 0, n)).astype(np.float32)
    for B in sorted({1, max(1, n // 2), max(1, n - 1), n}):
        got, cu, st, paths = _topk_hist(tsel, s, [0, n], [B])
        assert st == 0
        _check(got, cu, s, [0, n], [B])
        # one CTA below 8192 tokens: no histograms
        assert paths[CANDIDATES if n >= 8192 else PLAIN] == 1, (n, B, paths)


def test_hist_start_ties_across_slices(tsel):
    # 1,500 copies of one score spread over every slice of a 16-CTA cluster,
    # with the B-th score among them: the candidates are the tied keys and the
    # lowest indices must win across CTAs
    rng = np.random.default_rng(3)
    n = 60000
    s = rng.random(n).astype(np.float32)
    tie = np.sort(rng.choice(n, 1500, replace=False))
    s[tie] = np.float32(0.5)
    below = int(np.sum(s > 0.5))
    for B in (below + 1, below + 700, below + 1500):
        got, cu, st, paths = _topk_hist(tsel, s, [0, n], [B])
        assert st == 0
        _check(got, cu, s, [0, n], [B])
        assert paths[CANDIDATES] == 1


def _shared_prefix_count(s, B):
    """Keys sharing the first 16 bits of the B-th largest key (-0 as +0): the
    candidates the histogram start resolves the threshold among."""
    u = np.where(s == 0, np.float32(0), s).astype(np.float32).view(np.uint32)
    key = np.where(u & 0x80000000, ~u, u | 0x80000000).astype(np.uint32)
    thr = np.sort(key)[::-1][B - 1]
    return int(np.sum((key >> 16) == (thr >> 16)))


@pytest.mark.parametrize("ties, ranked", [(90, True), (1500, False)])
def test_hist_start_threshold_by_rank_or_rounds(tsel, ties, ranked):
    # log-uniform scores (about 25 keys per 16-bit bin near 0.5) plus `ties`
    # copies of 0.5 spread over every slice: at most 256 candidates are
    # ranked directly, more take the two 8-bit rounds; both must keep the
    # lowest indices of the tied keys across the cluster's CTAs
    rng = np.random.default_rng(11 + ties)
    n = 60000
    s = np.exp2(rng.uniform(-20, 0, n)).astype(np.float32)
    tie = np.sort(rng.choice(n, ties, replace=False))
    s[tie] = np.float32(0.5)
    above = int(np.sum(s > 0.5))
    for B in (above + 1, above + ties // 2, above + ties):
        assert (_shared_prefix_count(s, B) <= 256) == ranked
        got, cu, st, paths = _topk_hist(tsel, s, [0, n], [B])
        assert st == 0
        _check(got, cu, s, [0, n], [B])
        assert paths[CANDIDATES] == 1


def test_hist_start_too_many_candidates_uses_rounds(tsel):
    # few distinct values: the threshold's 16-bit bin holds far more than the
    # candidate list, so the top-B runs its rounds from the second digit
    rng = np.random.default_rng(4)
    n = 70000
    s = (rng.integers(0, 3, n).astype(np.float32) * 0.125)
    for B in (1, n // 3, n - 1):
        got, cu, st, paths = _topk_hist(tsel, s, [0, n], [B])
        assert st == 0
        _check(got, cu, s, [0, n], [B])
        assert paths[HIST_ROUNDS] == 1, paths


def test_hist_start_signed_zeros_and_negatives(tsel):
    rng = np.random.default_rng(5)
    n = 30000
    s = rng.random(n).astype(np.float32) - np.float32(0.3)
    s[::5] = np.float32(-0.0)
    s[1::5] = np.float32(0.0)
    for B in (1, 5000, 20000, 25000, n):
        got, cu, st, paths = _topk_hist(tsel, s, [0, n], [B])
        assert st == 0
        _check(got, cu, s, [0, n], [B])


def test_hist_start_many_requests(tsel):
    # 64 requests (histograms) and 65 (more than the histograms serve: plain)
    rng = np.random.default_rng(6)
    for R in (64, 65):
        sizes = rng.integers(8000, 14000, R)   # clusters of CTAs per request
        sizes[::9] = 0
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
        s = (rng.random(off[-1]) * 4).astype(np.float32)
        s[rng.integers(0, off[-1], off[-1] // 10)] = np.float32(1.0)
        keep = [int(x) for x in (sizes * rng.random(R)).astype(np.int64)]
        got, cu, st, paths = _topk_hist(tsel, s, off.tolist(), keep)
        assert st == 0
        _check(got, cu, s, off.tolist(), keep)
        served = sum(1 for k in keep if k > 0)
        if R == 64:
            assert paths[PLAIN] == 0 and sum(paths) == served
        else:
            assert paths == [served, 0, 0, 0, 0]


def test_hist_start_device_budgets(tsel):
    # budgets computed on the device (TSEL_KEEP_FROM_DEVICE): keep_idx has room
    # for every token and cu_keep[R] holds the kept count
    rng = np.random.default_rng(7)
    sizes = [20000, 0, 5000, 33000]
    off = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    s = rng.random(off[-1]).astype(np.float32)
    keep = [7000, 0, 4999, 1]
    got, cu, st, _ = _topk_hist(tsel, s, off, keep, total_keep=tsel.TSEL_KEEP_FROM_DEVICE)
    assert st == 0
    _check(got, cu, s, off, keep)


def test_hist_start_nan_scores(tsel):
    rng = np.random.default_rng(77)
    n, B = 50000, 20000
    s = rng.random(n).astype(np.float32)
    nan_at = np.sort(rng.choice(n, 12, replace=False))
    s[nan_at] = np.float32(np.nan)
    got, cu, st, _ = _topk_hist(tsel, s, [0, n], [B])
    assert st & tsel.TSEL_DEV_NAN
    assert got.shape == (B,) and cu.tolist() == [0, B]
    assert np.all(np.diff(got) > 0) and got[0] >= 0 and got[-1] < n
    rest = got[~np.isnan(s[got])]
    clean = np.where(np.isnan(s), np.float32(-1.0), s).astype(np.float32)
    ref, _ = oracle.select_topk(clean, [0, n], [rest.size])
    assert np.array_equal(rest, ref)
