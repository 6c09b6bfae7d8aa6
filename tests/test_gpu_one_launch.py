"""The one-launch importance path for small problems (every segment at most
256 query rows and 256 keys, bf16, at most 16 heads): parity with the fp64
oracle and with the scheduled two-pass launches on the same inputs, ragged and
empty segments, every head_dim and GQA ratio, determinism, the SUM
normalisation, its bounded waits, and which inputs take it."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import REL_TOL, bits_to_bf16, i32, max_rel_err, to_device

pytestmark = pytest.mark.gpu

# The two paths compute the same fp32 quantities in different orders (row
# reference per 64 keys vs per segment, the head sum over a cluster vs head
# groups); both sit ~1e-6 from the oracle, so they agree far inside REL_TOL.
PATH_TOL = 1e-4


@pytest.fixture(scope="module")
def tsel():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_score_vision_gb300 as t
    t.build()
    t.load_library()
    return t


def _one(tsel, w, flags=0):
    return tsel.tsel_importance_one_launch(w.num_seg, w.total_q, w.total_k, max(w.max_seqlen_q, 1),
                                           max(w.max_seqlen_k, 1), w.num_heads, w.head_dim, flags)


def _run(tsel, w, flags=0, fill=None):
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    sc = torch.empty(w.total_k, device="cuda")
    lse = torch.empty((w.num_heads, w.total_q), device="cuda")
    if fill is not None:
        sc.fill_(fill)
        lse.fill_(fill)
    tsel.tsel_importance(q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), max(w.max_seqlen_q, 1),
                         max(w.max_seqlen_k, 1), flags=flags, lse=lse, scores=sc, workspace=ws)
    st = tsel.tsel_read_device_status(ws)
    return sc.cpu().numpy(), lse.cpu().numpy(), st


def _check_both_paths(tsel, w, norm="mean"):
    extra = tsel.TSEL_IMP_SCORE_SUM if norm == "sum" else 0
    assert _one(tsel, w, extra) == 1
    assert _one(tsel, w, extra | tsel.TSEL_IMP_TWO_PASS) == 0
    s1, l1, st1 = _run(tsel, w, extra)
    s2, l2, st2 = _run(tsel, w, extra | tsel.TSEL_IMP_TWO_PASS)
    assert st1 == 0 and st2 == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k, norm=norm)
    assert max_rel_err(s1, s_ref) <= REL_TOL
    np.testing.assert_allclose(l1, lse_ref, rtol=1e-5, atol=1e-4)
    assert max_rel_err(s1, s2.astype(np.float64)) <= PATH_TOL
    np.testing.assert_allclose(l1, l2, rtol=1e-5, atol=1e-5)
    return s1


@pytest.mark.parametrize("d", [64, 80, 96, 112, 128])
@pytest.mark.parametrize("H,Hkv", [(1, 1), (4, 4), (4, 2), (3, 1), (12, 4), (16, 16), (16, 8)])
def test_head_dims_gqa_ragged(tsel, d, H, Hkv):
    Lq = [1, 127, 128, 129, 256]
    Lk = [256, 1, 129, 128, 64]
    w = W.make_segments(Lq, Lk, H, Hkv, d, seed=900 + d + 7 * H + Hkv,
                        sink_counts=[3, 0, 2, 1, 4], hidden_dim=64)
    _check_both_paths(tsel, w)


def test_empty_segments_and_segments_without_keys(tsel):
    # no queries -> scores 0; no keys -> nothing scored and LSE -inf
    w = W.make_segments([0, 5, 256, 0, 3, 40], [4, 0, 256, 7, 0, 1], 8, 4, 80, seed=931,
                        sink_counts=[0, 0, 3, 1, 0, 0], hidden_dim=64)
    s = _check_both_paths(tsel, w)
    assert np.all(s[0:4] == 0.0) and np.all(s[260:267] == 0.0)
    _, lse, _ = _run(tsel, w)
    assert np.all(np.isneginf(lse[:, 0:5])) and np.all(np.isneginf(lse[:, 261:264]))


def test_sum_normalisation(tsel):
    w = W.make_segments([200, 31], [256, 97], 16, 4, 128, seed=932, sink_counts=[4, 1], hidden_dim=64)
    _check_both_paths(tsel, w, norm="sum")


@pytest.mark.parametrize("name", ["single_image_256", "six_views_1536"])
def test_workloads_take_one_launch_and_are_deterministic(tsel, name):
    w = W.make(name)
    assert _one(tsel, w) == 1
    s = _check_both_paths(tsel, w)
    for _ in range(3):
        s_again, _, st = _run(tsel, w)
        assert st == 0
        assert np.array_equal(s_again.view(np.uint32), s.view(np.uint32))


def test_which_inputs_take_one_launch(tsel):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ok = dict(num_seg=6, total_q=1536, total_k=1536, max_seqlen_q=256, max_seqlen_k=256,
              num_heads=16, head_dim=80)
    assert tsel.tsel_importance_one_launch(**ok) == 1

    def q(**kw):
        a = dict(ok)
        flags = kw.pop("flags", 0)
        a.update(kw)
        return tsel.tsel_importance_one_launch(**a, flags=flags)

    assert q(max_seqlen_q=257) == 0
    assert q(max_seqlen_k=257) == 0
    assert q(num_heads=17) == 0
    assert q(num_seg=sms // 16 + 1) == 0          # more CTAs than SMs
    assert q(head_dim=72) == 0
    assert q(total_q=0) == 0 and q(total_k=0) == 0
    for f in ("TSEL_IMP_TWO_PASS", "TSEL_IMP_ROWREF_FIXED", "TSEL_IMP_ROWREF_MOVING",
              "TSEL_IMP_STAGE_PREP", "TSEL_IMP_STAGE_PASS2"):
        assert q(flags=getattr(tsel, f)) == 0, f
    for f in ("TSEL_IMP_SCORE_SUM", "TSEL_IMP_LSE_PROVIDED", "TSEL_IMP_FP8_E4M3"):
        assert q(flags=getattr(tsel, f)) == 1, f
    assert q(num_heads=1, head_dim=128, num_seg=1) == 1


def test_bounded_waits_run_out_in_one_launch(tsel):
    """With the test hook the one-launch kernel issues no loads: its MMA thread
    gives up after ~50 ms, sets TSEL_DEV_TIMEOUT, the epilogue warps see the
    abort and every CTA still passes its barriers and exits with nothing in
    flight; no score or LSE is written. The next call works."""
    w = W.make("six_views_1536")
    assert _one(tsel, w, tsel.TSEL_IMP_TEST_STALL) == 1
    s, lse, st = _run(tsel, w, tsel.TSEL_IMP_TEST_STALL, fill=7.0)
    assert st & tsel.TSEL_DEV_TIMEOUT
    assert np.all(s == 7.0) and np.all(lse == 7.0)
    s, _, st = _run(tsel, w)
    assert st == 0
    _, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s, s_ref) <= REL_TOL


def test_malformed_cu_seqlens_in_one_launch(tsel):
    q = torch.zeros((10, 2, 64), dtype=torch.bfloat16, device="cuda")
    assert tsel.tsel_importance_one_launch(2, 10, 10, 8, 8, 2, 64) == 1
    ws = torch.zeros(tsel.tsel_importance_workspace_size(2, 10, 10, 2), dtype=torch.uint8, device="cuda")
    sc = torch.full((10,), 7.0, device="cuda")
    for cu in ([0, 7, 5], [0, 5, 9], [1, 5, 10], [0, 9, 10]):
        tsel.tsel_clear_device_status(ws)
        tsel.tsel_importance(q, q, i32(cu), i32([0, 5, 10]), 8, 8, scores=sc, workspace=ws)
        assert tsel.tsel_read_device_status(ws) & tsel.TSEL_DEV_SEQLENS, cu
        assert torch.all(sc == 7.0)   # nothing is computed from malformed metadata


def test_large_logit_gaps_follow_the_row_max(tsel):
    """Keys whose logits stand ~128 nats above the rest of their row (past the
    first 64 keys): the one-launch kernel's row reference follows the max, so
    no term leaves the fp32 range and no redo exists to take them."""
    d = 64
    w = W.make_far_keys([200, 256, 129], 4, 2, d, seed=951, far_positions=[100, 400],
                        far_value=128.0 * np.sqrt(d) / 4.0, head_signs=[1, 1, -1, -1], name="far")
    assert _one(tsel, w) == 1
    s, lse, st = _run(tsel, w)
    assert st == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                       w.softmax_scale)
    assert max_rel_err(s, s_ref) <= REL_TOL
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=2e-4)


# ------------------------------------------------ top-B in the same launch

def _score_select(tsel, w, req_off, keep, total_keep=None, scale=0.0):
    dev = to_device(w)
    ws = torch.zeros(tsel.tsel_score_select_workspace_size(w.num_seg, w.total_q, w.total_k,
                                                           w.num_heads, len(keep)),
                     dtype=torch.uint8, device="cuda")
    tk = int(sum(keep)) if total_keep is None else total_keep
    s, _, kidx, cu = tsel.tsel_score_select(dev["q"], dev["k"], dev["cu_q"], dev["cu_k"],
                                            max(w.max_seqlen_q, 1), max(w.max_seqlen_k, 1),
                                            i32(req_off), i32(keep), tk, softmax_scale=scale,
                                            workspace=ws)
    st = tsel.tsel_read_device_status(ws)
    return (s.cpu().numpy(), kidx.cpu().numpy(), cu.cpu().numpy(), st,
            tsel.tsel_select_path_counts(ws))


@pytest.mark.parametrize("n,H,Hkv,d", [(256, 16, 16, 80), (200, 8, 2, 64), (1, 4, 4, 128),
                                       (129, 1, 1, 96), (37, 16, 8, 112)])
@pytest.mark.parametrize("frac", [0.0, 0.01, 0.6, 1.0])
def test_single_image_selected_in_the_importance_launch(tsel, n, H, Hkv, d, frac):
    """One image and one request: the one-launch kernel ranks the keys itself;
    keep_idx and cu_keep equal oracle.select_topk on the same fp32 scores, and
    the scores equal tsel_importance's bit for bit."""
    w = W.make_segments([n], [n], H, Hkv, d, seed=960 + n + H + d, sink_counts=[min(n, 3)],
                        hidden_dim=64)
    B = int(frac * n)
    s, kidx, cu, st, paths = _score_select(tsel, w, [0, n], [B])
    assert st == 0
    assert paths == [0, 0, 0, 0, 1 if B > 0 else 0], paths
    k_ref, cu_ref = oracle.select_topk(s, [0, n], [B])
    assert np.array_equal(kidx[:B], k_ref) and np.array_equal(cu, cu_ref)
    s_imp, _, _ = _run(tsel, w)
    assert np.array_equal(s.view(np.uint32), s_imp.view(np.uint32))
    _, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s, s_ref) <= REL_TOL


@pytest.mark.parametrize("lo,hi,B", [(17, 200, 50), (0, 128, 128), (255, 256, 1), (100, 100, 0)])
def test_selection_of_a_token_range(tsel, lo, hi, B):
    w = W.make_segments([256], [256], 8, 8, 80, seed=971, sink_counts=[4], hidden_dim=64)
    s, kidx, cu, st, paths = _score_select(tsel, w, [lo, hi], [B])
    assert st == 0
    k_ref, cu_ref = oracle.select_topk(s, [lo, hi], [B])
    assert np.array_equal(kidx[:B], k_ref) and np.array_equal(cu, cu_ref)


def test_selection_ties_keep_the_lowest_indices(tsel):
    # Q = 0: every probability of a row is equal, so every key's score is too
    w = W.make_segments([256], [256], 4, 4, 64, seed=972, hidden_dim=64)
    w.q_bits[:] = 0
    s, kidx, cu, st, _ = _score_select(tsel, w, [10, 250], [77])
    assert st == 0
    assert np.all(s == s[0])
    assert np.array_equal(kidx, np.arange(10, 87, dtype=np.int32))
    assert np.array_equal(cu, [0, 77])


@pytest.mark.parametrize("req_off,keep,total_keep", [([0, 257], [5], 5), ([0, 100], [101], 101),
                                                     ([50, 40], [1], 1), ([0, 256], [5], 6)])
def test_selection_bad_requests_set_status(tsel, req_off, keep, total_keep):
    w = W.make_segments([256], [256], 4, 4, 64, seed=973, hidden_dim=64)
    s, _, _, st, paths = _score_select(tsel, w, req_off, keep, total_keep)
    assert st & tsel.TSEL_DEV_REQUESTS
    assert paths == [0, 0, 0, 0, 0]
    _, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s, s_ref) <= REL_TOL   # the scores are still written


# ---------------------------------------------- the caller's LSE, one launch

@pytest.mark.parametrize("Lq,Lk,H,Hkv,d", [([256], [256], 16, 16, 80), ([1, 127, 200], [256, 3, 129], 8, 2, 64),
                                           ([0, 50, 9], [40, 0, 256], 4, 4, 128)])
def test_lse_provided_in_one_launch(tsel, Lq, Lk, H, Hkv, d):
    """TSEL_IMP_LSE_PROVIDED on the one-launch path: no row-LSE phase, the
    column sums from the caller's LSE (here the oracle's, rounded to fp32),
    against the oracle and against the two-pass form with the same LSE."""
    w = W.make_segments(Lq, Lk, H, Hkv, d, seed=1000 + H + d, sink_counts=[min(n, 2) for n in Lk],
                        hidden_dim=64)
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    F = tsel.TSEL_IMP_LSE_PROVIDED
    assert _one(tsel, w, F) == 1 and _one(tsel, w, F | tsel.TSEL_IMP_TWO_PASS) == 0
    out = []
    for flags in (F, F | tsel.TSEL_IMP_TWO_PASS):
        q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
        ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, w.num_heads),
                         dtype=torch.uint8, device="cuda")
        lse = torch.from_numpy(lse_ref.astype(np.float32)).cuda()
        s, _ = tsel.tsel_importance(q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k),
                                    max(w.max_seqlen_q, 1), max(w.max_seqlen_k, 1), flags=flags,
                                    lse=lse, workspace=ws)
        assert tsel.tsel_read_device_status(ws) == 0
        out.append(s.cpu().numpy())
    assert max_rel_err(out[0], s_ref) <= REL_TOL
    assert max_rel_err(out[0], out[1].astype(np.float64)) <= PATH_TOL


# ------------------------------------------------------- E4M3, one launch

@pytest.mark.parametrize("d", [64, 80, 96, 112, 128])
@pytest.mark.parametrize("lse_given", [False, True])
def test_fp8_in_one_launch(tsel, d, lse_given):
    """E4M3 Q/K (kind::f8f6f4 MMAs) on the one-launch path against the
    E4M3-decoding oracle and against the two-pass form on the same bytes."""
    L = [1, 127, 128, 129, 256]
    w = W.to_e4m3(W.make_segments(L, L, 8, 4, d, seed=1100 + d, sink_counts=[0, 1, 2, 3, 6],
                                  hidden_dim=16))
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                       w.softmax_scale, fmt="e4m3")
    F = tsel.TSEL_IMP_FP8_E4M3 | (tsel.TSEL_IMP_LSE_PROVIDED if lse_given else 0)
    assert _one(tsel, w, F) == 1
    out = []
    for flags in (0, tsel.TSEL_IMP_TWO_PASS):
        q = torch.from_numpy(w.q_bits).cuda()
        k = torch.from_numpy(w.k_bits).cuda()
        ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, w.num_heads),
                         dtype=torch.uint8, device="cuda")
        lse = torch.from_numpy(lse_ref.astype(np.float32)).cuda() if lse_given else None
        kw = {"flags": flags | (tsel.TSEL_IMP_LSE_PROVIDED if lse_given else 0)}
        s, lse_out = tsel.tsel_importance(q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), 256, 256,
                                          softmax_scale=w.softmax_scale, lse=lse, workspace=ws, **kw)
        assert tsel.tsel_read_device_status(ws) == 0
        out.append((s.cpu().numpy(), lse_out.cpu().numpy()))
    assert max_rel_err(out[0][0], s_ref) <= REL_TOL
    assert max_rel_err(out[0][0], out[1][0].astype(np.float64)) <= PATH_TOL
    if not lse_given:
        np.testing.assert_allclose(out[0][1], lse_ref, rtol=1e-5, atol=1e-4)


# ------------------------------------------------------ seeded random sweep

@pytest.mark.parametrize("seed", range(16))
def test_random_small_problems(tsel, seed):
    """Random problems that all take the one-launch path (segments of 0..256
    queries and keys, 1..9 segments, 1..16 heads with GQA, every head_dim,
    explicit scales): scores and LSE against the oracle and the two-pass form;
    a single image also gets a random budget selected in the same launch."""
    rng = np.random.default_rng(1200 + seed)
    G = int(rng.integers(1, 10))
    H = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
    while G * H > 144:
        G -= 1
    Hkv = int(rng.choice([x for x in range(1, H + 1) if H % x == 0]))
    d = int(rng.choice([64, 80, 96, 112, 128]))
    # as many segments as have their clusters resident at once
    while G > 1 and tsel.tsel_importance_one_launch(G, 256 * G, 256 * G, 256, 256, H, d) != 1:
        G -= 1
    lens = [0, 1, 2, 31, 64, 127, 128, 129, 200, 255, 256]
    lk = rng.choice(lens, size=G)
    lq = lk.copy() if rng.random() < 0.5 else rng.choice(lens, size=G)
    if lq.sum() == 0:
        lq[0] = 5
    if lk.sum() == 0:
        lk[0] = 7
    scale = float(rng.choice([0.0, 0.05, 0.3]))
    w = W.make_segments(lq, lk, H, Hkv, d, seed=1300 + seed, q_std=float(rng.choice([0.2, 1.0, 2.0])),
                        sink_counts=rng.integers(0, 3, size=G), hidden_dim=64,
                        softmax_scale=scale if scale > 0 else None)
    assert _one(tsel, w) == 1
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                       softmax_scale=scale if scale > 0 else None)
    outs = []
    for flags in (0, tsel.TSEL_IMP_TWO_PASS):
        q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
        ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, H),
                         dtype=torch.uint8, device="cuda")
        s, lse = tsel.tsel_importance(q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k),
                                      max(w.max_seqlen_q, 1), max(w.max_seqlen_k, 1), flags=flags,
                                      softmax_scale=scale, workspace=ws)
        assert tsel.tsel_read_device_status(ws) == 0
        outs.append((s.cpu().numpy(), lse.cpu().numpy()))
    s1, l1 = outs[0]
    assert max_rel_err(s1, s_ref) <= REL_TOL
    assert max_rel_err(s1, outs[1][0].astype(np.float64)) <= PATH_TOL
    fin = np.isfinite(lse_ref)
    assert np.all(np.isneginf(l1[~fin]))
    np.testing.assert_allclose(l1[fin], lse_ref[fin], rtol=1e-5, atol=2e-4)
    if G == 1 and w.total_k > 0:
        n = w.total_k
        B = int(rng.integers(0, n + 1))
        s_sel, kidx, cu, st, paths = _score_select(tsel, w, [0, n], [B], scale=scale)
        assert st == 0 and paths == [0, 0, 0, 0, 1 if B > 0 else 0]
        assert np.array_equal(s_sel.view(np.uint32), s1.view(np.uint32))
        k_ref, cu_ref = oracle.select_topk(s_sel, [0, n], [B])
        assert np.array_equal(kidx[:B], k_ref) and np.array_equal(cu, cu_ref)


def test_fp8_single_image_selected_in_the_launch(tsel):
    """E4M3 inputs take the same single-launch selection: keep_idx equals the
    oracle's selection on the same fp32 scores."""
    w = W.to_e4m3(W.make_segments([256], [256], 8, 4, 128, seed=1400, sink_counts=[3], hidden_dim=16))
    q, k = torch.from_numpy(w.q_bits).cuda(), torch.from_numpy(w.k_bits).cuda()
    ws = torch.zeros(tsel.tsel_score_select_workspace_size(1, 256, 256, 8, 1), dtype=torch.uint8,
                     device="cuda")
    s, _, kidx, cu = tsel.tsel_score_select(q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), 256, 256,
                                            i32([0, 256]), i32([100]), 100,
                                            softmax_scale=w.softmax_scale, workspace=ws)
    assert tsel.tsel_read_device_status(ws) == 0
    assert tsel.tsel_select_path_counts(ws) == [0, 0, 0, 0, 1]
    s = s.cpu().numpy()
    k_ref, cu_ref = oracle.select_topk(s, [0, 256], [100])
    assert np.array_equal(kidx.cpu().numpy(), k_ref) and np.array_equal(cu.cpu().numpy(), cu_ref)
    _, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k, w.softmax_scale,
                                 fmt="e4m3")
    assert max_rel_err(s, s_ref) <= REL_TOL
