"""GPU edge cases: ragged and empty segments, one-key segments, segments
without queries, every supported head_dim, GQA ratios, strided (packed QKV)
inputs, closed forms, top-B ties and budgets at the extremes, and the device
status word for malformed metadata (checked on the device, no fault)."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import REL_TOL, bits_to_bf16, check_selection_exact, i32, max_rel_err, run_path

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsel():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_score_vision_gb300 as t
    t.build()
    t.load_library()
    return t


def _importance(tsel, w, **kw):
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    s, lse = tsel.tsel_importance(q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k),
                                  max(w.max_seqlen_q, 1), max(w.max_seqlen_k, 1), workspace=ws, **kw)
    st = tsel.tsel_read_device_status(ws)
    return s.cpu().numpy(), lse.cpu().numpy(), st


@pytest.mark.parametrize("d", [64, 80, 96, 112, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (8, 2), (3, 1), (6, 3), (12, 4)])
def test_head_dims_and_gqa(tsel, d, H, Hkv):
    L = [1, 127, 128, 129, 257]
    w = W.make_segments(L, L, H, Hkv, d, seed=200 + d + H, sink_counts=[0, 1, 2, 3, 4], hidden_dim=64)
    s, lse, st = _importance(tsel, w)
    assert st == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s, s_ref) <= REL_TOL
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=1e-4)


def test_column_pass_rerun_is_bit_for_bit(tsel):
    # The column pass splits the query heads into groups whose partial sums
    # the last group of each 32-key slice adds up in group order: reruns of
    # the schedule + column pass on the stored LSE give the same bits.
    w = W.make_segments([700, 40, 300], [513, 1, 260], 8, 2, 64, seed=303, sink_counts=[5, 0, 2],
                        hidden_dim=64)
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    args = (q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), w.max_seqlen_q, w.max_seqlen_k)
    s_all, _ = tsel.tsel_importance(*args, workspace=ws)
    s_all = s_all.clone()
    runs = []
    for _ in range(3):
        s, _ = tsel.tsel_importance(*args, workspace=ws, want_lse=False,
                                    flags=tsel.TSEL_IMP_STAGE_PREP | tsel.TSEL_IMP_STAGE_PASS2)
        runs.append(s.clone())
    assert tsel.tsel_read_device_status(ws) == 0
    for s in runs:
        assert torch.equal(s, s_all)
    _, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s_all.cpu().numpy(), s_ref) <= REL_TOL


def test_long_segment_4096_and_cross_lengths(tsel):
    w = W.make_segments([4096, 5, 300], [4096, 777, 3], 2, 1, 64, seed=301, sink_counts=[40, 7, 0],
                        hidden_dim=64)
    s, lse, st = _importance(tsel, w)
    assert st == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s, s_ref) <= REL_TOL
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=1e-4)


def test_very_long_segment_8192(tsel):
    # one 8,192-token image (64 key tiles per row; 32 query pairs per head)
    w = W.make_segments([8192], [8192], 1, 1, 64, seed=308, sink_counts=[100], hidden_dim=64)
    s, lse, st = _importance(tsel, w)
    assert st == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s, s_ref) <= REL_TOL
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("H,Hkv,d", [(32, 8, 64), (64, 64, 64), (40, 5, 128), (255, 255, 64)])
def test_many_heads(tsel, H, Hkv, d):
    w = W.make_segments([130, 300, 1], [130, 300, 1], H, Hkv, d, seed=309 + H, sink_counts=[2, 3, 0],
                        hidden_dim=64)
    s, lse, st = _importance(tsel, w)
    assert st == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s, s_ref) <= REL_TOL
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=1e-4)


def test_empty_segments_and_missing_queries(tsel):
    # segment 1 is empty, segment 2 has keys but no queries (scores 0),
    # segment 3 has queries but no keys (lse -inf)
    w = W.make_segments([50, 0, 0, 9, 130], [60, 0, 33, 0, 1], 4, 4, 64, seed=302, hidden_dim=64)
    s, lse, st = _importance(tsel, w)
    assert st == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s, s_ref) <= REL_TOL
    assert np.all(s[60:93] == 0)
    assert s[93] == pytest.approx(1.0, rel=1e-6)      # one-key segment
    assert np.all(np.isneginf(lse[:, 50:59]))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("G,max_len,H,Hkv", [(1500, 40, 4, 2), (4000, 8, 2, 1)])
def test_thousands_of_small_segments(tsel, G, max_len, H, Hkv):
    # more segments than the schedule kernel has threads: its block-wide
    # bucket sort, scans and unit lists loop; many segments share a tile
    rng = np.random.default_rng(G)
    L = rng.integers(0, max_len + 1, size=G)
    n_req = 7
    cuts = np.linspace(0, G, n_req + 1).astype(int)
    groups = np.diff(cuts).tolist()
    per_req = np.add.reduceat(L, cuts[:-1])
    keep = [int(x) // 3 for x in per_req]
    w = W.make_segments(L, L, H, Hkv, 64, seed=310 + G, hidden_dim=64, requests=groups,
                        keep_per_req=keep)
    out = run_path(tsel, w)
    assert out["status"] == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(out["scores"], s_ref) <= REL_TOL
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(out["lse"][fin], lse_ref[fin], rtol=1e-5, atol=1e-4)
    assert np.all(np.isneginf(out["lse"][~fin]))
    check_selection_exact(w, out)


def test_zero_queries_uniform_and_one_hot_closed_form(tsel):
    nq, nk, d, H = 130, 300, 64, 2
    q = np.zeros((nq, H, d), np.float32)
    q[:, :, 0] = 2.0
    k = np.zeros((nk, H, d), np.float32)
    k[123, :, 0] = 2.0
    w = W.Workload("onehot", W.f32_to_bf16_bits(q), W.f32_to_bf16_bits(k), np.array([0, nq], np.int32),
                   np.array([0, nk], np.int32), np.array([0, nk], np.int32), np.array([10], np.int32),
                   np.zeros((nk, 8), np.uint16), np.zeros((nk, 1), np.int32), 1 / 8)
    s, lse, st = _importance(tsel, w)
    c = math.exp(4.0 / 8.0)
    expect = np.full(nk, 1 / (c + nk - 1))
    expect[123] = c / (c + nk - 1)
    assert np.max(np.abs(s - expect) / expect) <= REL_TOL
    np.testing.assert_allclose(lse, math.log(c + nk - 1), rtol=1e-5)
    w.q_bits[:] = 0
    s0, _, _ = _importance(tsel, w)
    np.testing.assert_allclose(s0, 1 / nk, rtol=REL_TOL)


def test_strided_packed_qkv_rows(tsel):
    """q and k as views into one packed [T, 3, H, d] buffer (row stride 3*H*d)."""
    L = [200, 90]
    w = W.make_segments(L, L, 4, 4, 80, seed=303, sink_counts=[2, 1], hidden_dim=64)
    T, H, d = w.total_q, 4, 80
    packed = torch.zeros((T, 3, H, d), dtype=torch.bfloat16, device="cuda")
    packed[:, 0] = bits_to_bf16(w.q_bits)
    packed[:, 1] = bits_to_bf16(w.k_bits)
    ws = torch.zeros(tsel.tsel_importance_workspace_size(2, T, T, H), dtype=torch.uint8, device="cuda")
    s, _ = tsel.tsel_importance(packed[:, 0], packed[:, 1], i32(w.cu_seqlens_q), i32(w.cu_seqlens_k),
                                200, 200, workspace=ws)
    _, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s.cpu().numpy(), s_ref) <= REL_TOL
    assert tsel.tsel_read_device_status(ws) == 0


def test_explicit_softmax_scale(tsel):
    w = W.make_segments([100], [140], 4, 4, 64, seed=304, hidden_dim=64)
    s, lse, st = _importance(tsel, w, softmax_scale=0.05)
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k, 0.05)
    assert max_rel_err(s, s_ref) <= REL_TOL
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=1e-4)


# ---------------------------------------------------------------- top-B / gather

def _topk(tsel, scores, off, keep):
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    k_idx, cu = tsel.tsel_select_topk(torch.from_numpy(np.asarray(scores, np.float32)).cuda(), i32(off),
                                      i32(keep), int(np.sum(keep)), workspace=ws)
    return k_idx.cpu().numpy(), cu.cpu().numpy(), tsel.tsel_read_device_status(ws)


def test_topk_ties_and_extreme_budgets(tsel):
    rng = np.random.default_rng(5)
    for n, vals in [(1, 3), (9, 2), (1000, 3), (5000, 1), (70000, 40)]:
        s = rng.integers(0, vals, n).astype(np.float32) * 0.125
        for B in sorted({0, 1, n // 3, n - 1, n}):
            if B < 0:
                continue
            got, cu, st = _topk(tsel, s, [0, n], [B])
            ref, cref = oracle.select_topk(s, [0, n], [B])
            assert st == 0
            assert np.array_equal(got, ref), (n, B)
            assert np.array_equal(cu, cref)


def test_topk_many_requests_and_negative_zero(tsel):
    rng = np.random.default_rng(6)
    s = rng.random(3000).astype(np.float32)
    s[::7] = -0.0
    s[1::7] = 0.0
    off = [0, 0, 10, 1000, 1001, 3000]
    keep = [0, 10, 300, 0, 1500]
    got, cu, st = _topk(tsel, s, off, keep)
    ref, cref = oracle.select_topk(np.where(s == 0, 0.0, s).astype(np.float32), off, keep)
    assert st == 0 and np.array_equal(got, ref) and np.array_equal(cu, cref)


@pytest.mark.parametrize("big", [4096, 4097, 9000])
def test_topk_small_requests_with_one_large(tsel, big):
    # one CTA per request (the average request is small); requests from
    # empty to thousands of tokens, sizes on both sides of 4096
    rng = np.random.default_rng(big)
    sizes = [big] + [10, 0, 37, 1, 256, 3, 99, 64]
    off = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    s = (rng.integers(0, 50, off[-1]).astype(np.float32) * 0.25)   # many ties
    keep = [big // 3, 10, 0, 20, 1, 255, 0, 99, 7]
    got, cu, st = _topk(tsel, s, off, keep)
    ref, cref = oracle.select_topk(s, off, keep)
    assert st == 0
    assert np.array_equal(got, ref) and np.array_equal(cu, cref)


@pytest.mark.parametrize("sizes", [[10000] * 4, [20000, 20001], [40000], [300000]])
def test_topk_cluster_sizes_and_uncached_slices(tsel, sizes):
    # clusters of 4, 8 and 16 CTAs (average request 10K, 20K, 40K tokens) and,
    # at 300K tokens, slices too long for the per-CTA key cache; scores span
    # many binades (every digit of every round is used), with negative values,
    # signed zeros and long runs of ties
    rng = np.random.default_rng(sum(sizes))
    off = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    n = off[-1]
    s = (np.exp2(rng.uniform(-40, 40, n)) * rng.choice([-1.0, 1.0], n, p=[0.1, 0.9])).astype(np.float32)
    s[rng.integers(0, n, n // 5)] = np.float32(0.75)
    s[rng.integers(0, n, n // 50)] = np.float32(-0.0)
    s[rng.integers(0, n, n // 50)] = np.float32(0.0)
    keep = [(i * 37 + 11) * sz // 97 % (sz + 1) for i, sz in enumerate(sizes)]
    got, cu, st = _topk(tsel, s, off, keep)
    ref, cref = oracle.select_topk(np.where(s == 0, 0.0, s).astype(np.float32), off, keep)
    assert st == 0
    assert np.array_equal(got, ref) and np.array_equal(cu, cref)


def test_gather_fp32_rows_and_no_pos(tsel):
    hidden = torch.randn(500, 12, device="cuda", dtype=torch.float32)
    cu = i32([0, 100, 100, 500])
    keep = torch.tensor([0, 5, 99, 100, 499], dtype=torch.int32, device="cuda")
    oh, op, oi, oc = tsel.tsel_gather_compact(hidden, None, cu, keep)
    assert op is None
    assert torch.equal(oh, hidden[keep.long()])
    assert oi.tolist() == [0, 0, 0, 2, 2]
    assert oc.tolist() == [0, 3, 3, 5]


@pytest.mark.parametrize("sizes,keep", [([100000, 5, 0, 3000, 1], [1000, 5, 0, 0, 1]),
                                        ([70000, 7], [69999, 2]),
                                        ([3, 65000, 40000, 2], [1, 0, 40000, 1])])
def test_topk_uneven_requests_in_clusters(tsel, sizes, keep):
    # the cluster size follows the average request, so small requests run on
    # clusters whose CTAs mostly hold no token; budgets of 0, all and all but one
    rng = np.random.default_rng(len(sizes) + sizes[0])
    off = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    s = rng.random(off[-1]).astype(np.float32)
    s[rng.integers(0, off[-1], off[-1] // 3)] = np.float32(0.5)   # ties across slices
    got, cu, st = _topk(tsel, s, off, keep)
    ref, cref = oracle.select_topk(s, off, keep)
    assert st == 0
    assert np.array_equal(got, ref) and np.array_equal(cu, cref)


def test_topk_more_large_requests_than_resident_clusters(tsel):
    # twelve 40K-token requests: clusters of 16 CTAs would not all fit on the
    # device at once, so the launch takes a smaller cluster size
    rng = np.random.default_rng(12)
    sizes = [40000] * 11 + [39999]
    off = np.concatenate([[0], np.cumsum(sizes)]).tolist()
    s = rng.random(off[-1]).astype(np.float32)
    s[rng.integers(0, off[-1], off[-1] // 4)] = np.float32(0.25)   # ties across slices
    keep = [(7919 * (i + 1)) % (sz + 1) for i, sz in enumerate(sizes)]
    got, cu, st = _topk(tsel, s, off, keep)
    ref, cref = oracle.select_topk(s, off, keep)
    assert st == 0
    assert np.array_equal(got, ref) and np.array_equal(cu, cref)


def test_topk_nan_in_cluster_slices(tsel):
    # NaN scores in several slices of a 16-CTA cluster: the status flags them;
    # their rank is unspecified, but every other kept token must be one of the
    # best non-NaN tokens (score descending, lowest index first), B in total,
    # ascending and in range
    rng = np.random.default_rng(77)
    n, B = 50000, 20000
    s = rng.random(n).astype(np.float32)
    nan_at = np.sort(rng.choice(n, 12, replace=False))
    s[nan_at] = np.float32(np.nan)
    got, cu, st = _topk(tsel, s, [0, n], [B])
    assert st & tsel.TSEL_DEV_NAN
    assert got.shape == (B,) and cu.tolist() == [0, B]
    assert np.all(np.diff(got) > 0) and got[0] >= 0 and got[-1] < n
    is_nan = np.isnan(s[got])
    rest = got[~is_nan]
    clean = np.where(np.isnan(s), np.float32(-1.0), s).astype(np.float32)
    ref, _ = oracle.select_topk(clean, [0, n], [rest.size])
    assert np.array_equal(rest, ref)


@pytest.mark.parametrize("D,dtype,G", [(8, torch.bfloat16, 1), (256, torch.bfloat16, 31),
                                       (1280, torch.bfloat16, 32), (2048, torch.bfloat16, 33),
                                       (1792, torch.bfloat16, 5), (5120, torch.bfloat16, 3),
                                       (700, torch.float32, 40), (4, torch.float64, 200)])
def test_gather_row_widths_and_segment_counts(tsel, D, dtype, G):
    # rows held whole in registers (1 to 8 16-byte vectors per lane) and rows
    # past 4 KB (5120 bf16, the hidden size of a 32B VLM) copied in a loop;
    # image ids by ballot (up to 31 segments) and by binary search (more);
    # rows read through a stride wider than the row; an odd number of kept rows
    rng = np.random.default_rng(D + G)
    L = rng.integers(0, 60, G)
    L[0] = max(L[0], 1)
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    Tk = int(cu[-1])
    full = torch.randn(Tk, D + 24, device="cuda").to(dtype)
    hidden = full[:, 8:8 + D]               # row stride D + 24 elements
    pos = torch.from_numpy(rng.integers(-1000, 1000, (Tk, 3)).astype(np.int32)).cuda()
    keep = np.sort(rng.choice(Tk, size=max(1, (Tk * 3) // 5) | 1, replace=False)).astype(np.int32)
    oh, op, oi, oc = tsel.tsel_gather_compact(hidden, pos, i32(cu), i32(keep))
    h_np = hidden.view(torch.int16 if dtype == torch.bfloat16 else
                       (torch.int32 if dtype == torch.float32 else torch.int64)).cpu().numpy()
    rh, rp, ri, rc = oracle.gather_compact(h_np, pos.cpu().numpy(), cu, keep)
    o_np = oh.view(torch.int16 if dtype == torch.bfloat16 else
                   (torch.int32 if dtype == torch.float32 else torch.int64)).cpu().numpy()
    assert np.array_equal(o_np, rh)
    assert np.array_equal(op.cpu().numpy(), rp)
    assert np.array_equal(oi.cpu().numpy(), ri)
    assert np.array_equal(oc.cpu().numpy(), rc)


def test_full_selection_bit_exact_on_mid_size(tsel):
    w = W.make_segments([333, 1200, 17], [333, 1200, 17], 4, 4, 64, seed=305, hidden_dim=1280,
                        pos_dim=3, requests=[2, 1], keep_per_req=[900, 5])
    out = run_path(tsel, w)
    assert out["status"] == 0
    check_selection_exact(w, out)


# ---------------------------------------------------------------- device checks

@pytest.mark.parametrize("two_pass", [False, True])
def test_malformed_cu_seqlens_sets_status(tsel, two_pass):
    # small enough for the one-launch path; TSEL_IMP_TWO_PASS checks the schedule kernel's test
    flags = tsel.TSEL_IMP_TWO_PASS if two_pass else 0
    q = torch.zeros((10, 2, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(tsel.tsel_importance_workspace_size(2, 10, 10, 2), dtype=torch.uint8, device="cuda")
    for cu in ([0, 7, 5], [0, 5, 9], [1, 5, 10], [0, 9, 10]):
        tsel.tsel_clear_device_status(ws)
        # [0, 9, 10] violates max_seqlen = 8
        tsel.tsel_importance(q, q, i32(cu), i32([0, 5, 10]), 8, 8, flags=flags, workspace=ws)
        assert tsel.tsel_read_device_status(ws) & tsel.TSEL_DEV_SEQLENS, cu


def test_bad_requests_and_keep_idx_set_status(tsel):
    s = torch.rand(100, device="cuda")
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    tsel.tsel_select_topk(s, i32([0, 50, 100]), i32([10, 60]), 70, workspace=ws)   # 60 > 50 tokens
    assert tsel.tsel_read_device_status(ws) & tsel.TSEL_DEV_REQUESTS
    tsel.tsel_clear_device_status(ws)
    tsel.tsel_select_topk(s, i32([0, 50, 100]), i32([10, 20]), 31, workspace=ws)   # sum != total
    assert tsel.tsel_read_device_status(ws) & tsel.TSEL_DEV_REQUESTS
    tsel.tsel_clear_device_status(ws)
    s[3] = float("nan")
    tsel.tsel_select_topk(s, i32([0, 100]), i32([10]), 10, workspace=ws)
    assert tsel.tsel_read_device_status(ws) & tsel.TSEL_DEV_NAN
    tsel.tsel_clear_device_status(ws)
    hidden = torch.zeros((20, 8), dtype=torch.bfloat16, device="cuda")
    for bad in ([3, 2], [1, 20], [-1, 4]):
        tsel.tsel_clear_device_status(ws)
        tsel.tsel_gather_compact(hidden, None, i32([0, 20]), i32(bad), workspace=ws)
        assert tsel.tsel_read_device_status(ws) & tsel.TSEL_DEV_KEEP_IDX, bad


# ---------------------------------------------------------------- LSE-provided mode

@pytest.mark.parametrize("name", ["six_views_1536", "text_query_3072"])
def test_lse_provided_matches_oracle(tsel, name):
    """Column pass only, fed the oracle's own LSE (the attention kernel's LSE in a
    serving stack): the scores match the oracle without running the row pass."""
    w = W.make(name)
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    lse_in = torch.from_numpy(lse_ref.astype(np.float32)).cuda()
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    s, lse_out = tsel.tsel_importance(q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), w.max_seqlen_q,
                                      w.max_seqlen_k, flags=tsel.TSEL_IMP_LSE_PROVIDED, lse=lse_in,
                                      workspace=ws)
    assert tsel.tsel_read_device_status(ws) == 0
    assert max_rel_err(s.cpu().numpy(), s_ref) <= REL_TOL
    assert lse_out.data_ptr() == lse_in.data_ptr()
    assert torch.equal(lse_in.cpu(), torch.from_numpy(lse_ref.astype(np.float32)))  # input untouched


def test_lse_provided_with_empty_and_keyless_segments(tsel):
    w = W.make_segments([50, 0, 0, 9, 300], [60, 0, 33, 0, 129], 4, 2, 80, seed=306, hidden_dim=64)
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    lse_in = torch.from_numpy(lse_ref.astype(np.float32)).cuda()    # -inf rows included
    s, _ = tsel.tsel_importance(bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits), i32(w.cu_seqlens_q),
                                i32(w.cu_seqlens_k), 300, 129, flags=tsel.TSEL_IMP_LSE_PROVIDED,
                                lse=lse_in)
    assert max_rel_err(s.cpu().numpy(), s_ref) <= REL_TOL


def test_lse_provided_agrees_with_full_path(tsel):
    w = W.make_segments([1000, 257, 3000], [1000, 257, 3000], 16, 16, 80, seed=307,
                        sink_counts=[20, 5, 60], hidden_dim=64)
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    cq, ck = i32(w.cu_seqlens_q), i32(w.cu_seqlens_k)
    s_full, lse = tsel.tsel_importance(q, k, cq, ck, 3000, 3000)
    s_imp, _ = tsel.tsel_importance(q, k, cq, ck, 3000, 3000, flags=tsel.TSEL_IMP_LSE_PROVIDED,
                                    lse=lse.clone())
    a, b = s_full.cpu().numpy().astype(np.float64), s_imp.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(a - b) / a) <= 1e-4


# ---------------------------------------------------------------- failure detection

def test_bounded_waits_report_timeout_and_context_survives(tsel):
    """The test hook makes the pass kernels' scheduler publish nothing: every
    waiting role gives up after its ~50 ms limit, sets TSEL_DEV_TIMEOUT and
    exits with no copy or MMA in flight. The next call on the same context
    works and matches the oracle. (TSEL_IMP_TWO_PASS: the scheduled passes;
    the one-launch kernel's form of the test is in test_gpu_one_launch.)"""
    w = W.make("six_views_1536")
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    cq, ck = i32(w.cu_seqlens_q), i32(w.cu_seqlens_k)
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    tsel.tsel_importance(q, k, cq, ck, 256, 256,
                         flags=tsel.TSEL_IMP_TEST_STALL | tsel.TSEL_IMP_TWO_PASS, workspace=ws)
    bits = tsel.tsel_read_device_status(ws)
    assert bits & tsel.TSEL_DEV_TIMEOUT
    tsel.tsel_clear_device_status(ws)
    s, _ = tsel.tsel_importance(q, k, cq, ck, 256, 256, workspace=ws)
    assert tsel.tsel_read_device_status(ws) == 0
    _, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s.cpu().numpy(), s_ref) <= REL_TOL


# ---------------------------------------------------------------- CUDA graph capture

def test_whole_path_captures_into_a_cuda_graph(tsel):
    """The three entry points enqueue kernels only (no allocation, no host
    synchronisation), so the whole path can be captured once and replayed —
    the launch-latency path for small requests. Replays match the eager run
    bit for bit (the kernels are deterministic)."""
    from gpu_util import to_device
    w = W.make("six_views_1536")
    d = to_device(w)
    G, Tq, Tk, H, K = w.num_seg, w.total_q, w.total_k, w.num_heads, w.total_keep
    ws = torch.zeros(tsel.tsel_importance_workspace_size(G, Tq, Tk, H), dtype=torch.uint8, device="cuda")
    scores = torch.empty(Tk, device="cuda")
    lse = torch.empty((H, Tq), device="cuda")
    keep_idx = torch.empty(K, dtype=torch.int32, device="cuda")
    cu_keep = torch.empty(2, dtype=torch.int32, device="cuda")
    oh = torch.empty((K, d["hidden"].shape[1]), dtype=torch.bfloat16, device="cuda")
    op = torch.empty((K, 1), dtype=torch.int32, device="cuda")
    oi = torch.empty(K, dtype=torch.int32, device="cuda")
    oc = torch.empty(G + 1, dtype=torch.int32, device="cuda")

    def path():
        tsel.tsel_importance(d["q"], d["k"], d["cu_q"], d["cu_k"], 256, 256, lse=lse, scores=scores,
                             workspace=ws)
        tsel.tsel_select_topk(scores, d["req_off"], d["keep"], K, keep_idx=keep_idx, cu_keep=cu_keep,
                              workspace=ws)
        tsel.tsel_gather_compact(d["hidden"], d["pos"], d["cu_k"], keep_idx, out_hidden=oh, out_pos=op,
                                 out_img_id=oi, out_cu_seqlens=oc, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        path()                       # eager warm-up (sets per-device launch attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (scores, keep_idx, oh, oi, oc)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        path()
    for _ in range(3):
        for t in (scores, keep_idx, oh, oi, oc):
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(ref, (scores, keep_idx, oh, oi, oc)):
            assert torch.equal(a, b)
    assert tsel.tsel_read_device_status(ws) == 0


# ---------------------------------------------------------------- FP8 E4M3 inputs

def _fp8_importance(tsel, w, **kw):
    q = torch.from_numpy(w.q_bits).cuda()
    k = torch.from_numpy(w.k_bits).cuda()
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    s, lse = tsel.tsel_importance(q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), max(w.max_seqlen_q, 1),
                                  max(w.max_seqlen_k, 1), softmax_scale=w.softmax_scale, workspace=ws,
                                  **kw)
    return s.cpu().numpy(), lse.cpu().numpy(), tsel.tsel_read_device_status(ws)


@pytest.mark.parametrize("d", [64, 80, 96, 112, 128])
def test_fp8_e4m3_head_dims(tsel, d):
    L = [1, 127, 128, 129, 300]
    w = W.to_e4m3(W.make_segments(L, L, 4, 2, d, seed=400 + d, sink_counts=[0, 1, 2, 3, 6],
                                  hidden_dim=16))
    s, lse, st = _fp8_importance(tsel, w)
    assert st == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                       w.softmax_scale, fmt="e4m3")
    assert max_rel_err(s, s_ref) <= REL_TOL
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("name", ["six_views_1536", "text_query_3072"])
def test_fp8_e4m3_workloads(tsel, name):
    w = W.to_e4m3(W.make(name))
    s, lse, st = _fp8_importance(tsel, w)
    assert st == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                       w.softmax_scale, fmt="e4m3")
    assert max_rel_err(s, s_ref) <= REL_TOL
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=1e-4)
    # LSE-provided works on FP8 inputs too
    s2, _, st2 = _fp8_importance(tsel, w, flags=tsel.TSEL_IMP_LSE_PROVIDED,
                                 lse=torch.from_numpy(lse_ref.astype(np.float32)).cuda())
    assert st2 == 0 and max_rel_err(s2, s_ref) <= REL_TOL


def test_fp8_thirty_images_sampled(tsel):
    from gpu_util import segment_slice
    w = W.to_e4m3(W.make("thirty_images"))
    s, lse, st = _fp8_importance(tsel, w)
    assert st == 0
    lens = np.diff(w.cu_seqlens_k)
    for g in sorted({int(np.argmin(lens)), int(np.argmax(lens)), 3}):
        qb, kb, cq, ck, (q0, q1, k0, k1) = segment_slice(w, g)
        lse_ref, s_ref = oracle.importance(qb, kb, cq, ck, w.softmax_scale, fmt="e4m3")
        assert max_rel_err(s[k0:k1], s_ref) <= REL_TOL
        np.testing.assert_allclose(lse[:, q0:q1], lse_ref, rtol=1e-5, atol=1e-4)
