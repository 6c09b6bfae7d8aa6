"""Pins for the fp64 oracle: facts fixed by the pages and by the mathematics.

Each test would fail on a plausible slip inside the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong normaliser or GQA mapping),
without re-deriving the oracle's own formula.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
from workloads import f32_to_bf16_bits, f32_to_e4m3_bits, make_segments

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _rand_case(rng, lq, lk, H, Hkv, d, std=1.0):
    q = rng.standard_normal((sum(lq), H, d)).astype(np.float32) * std
    k = rng.standard_normal((sum(lk), Hkv, d)).astype(np.float32) * std
    cu_q = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lk)]).astype(np.int32)
    return _bits(q), _bits(k), cu_q, cu_k


# ---------------------------------------------------------------------------
# Softmax and totals
# ---------------------------------------------------------------------------

def test_probability_rows_sum_to_one():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((37, 16)) * 3
    k = rng.standard_normal((53, 16)) * 3
    p, lse = oracle.attention_probabilities(q, k, 0.25)
    assert p.shape == (37, 53)
    assert np.all(p > 0)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    # The LSE is the natural-log normaliser: log sum_j exp(s_ij).
    s = 0.25 * (q @ k.T)
    np.testing.assert_allclose(lse, np.log(np.exp(s).sum(axis=1)), rtol=1e-12)


@pytest.mark.parametrize("lq,lk,H,Hkv", [([50, 7, 130], [50, 7, 130], 4, 4),
                                          ([142], [300], 8, 2),
                                          ([3, 90], [64, 1], 2, 1)])
def test_scores_are_a_mean_totals(lq, lk, H, Hkv):
    """Each query row spreads probability 1, so a segment's scores sum to 1
    (before averaging the total is heads x query rows)."""
    rng = np.random.default_rng(2)
    qb, kb, cu_q, cu_k = _rand_case(rng, lq, lk, H, Hkv, 32, std=2.0)
    lse, scores = oracle.importance(qb, kb, cu_q, cu_k)
    for g in range(len(lk)):
        seg = scores[cu_k[g]:cu_k[g + 1]]
        assert abs(seg.sum() - 1.0) < 1e-12
        assert abs(seg.sum() * H * lq[g] - H * lq[g]) < 1e-9
        assert np.all(seg > 0)
    assert lse.shape == (H, sum(lq))


def test_zero_queries_give_uniform_scores():
    rng = np.random.default_rng(3)
    lq, lk = [20, 5], [33, 17]
    _, kb, cu_q, cu_k = _rand_case(rng, lq, lk, 4, 4, 64)
    qb = np.zeros((sum(lq), 4, 64), np.uint16)
    lse, scores = oracle.importance(qb, kb, cu_q, cu_k)
    np.testing.assert_allclose(scores[:33], 1 / 33, rtol=1e-14)
    np.testing.assert_allclose(scores[33:], 1 / 17, rtol=1e-14)
    np.testing.assert_allclose(lse[:, :20], math.log(33), rtol=1e-14)


def test_identical_keys_give_uniform_scores():
    rng = np.random.default_rng(4)
    qb, kb, cu_q, cu_k = _rand_case(rng, [40], [25], 2, 2, 16)
    kb[:] = kb[0]
    _, scores = oracle.importance(qb, kb, cu_q, cu_k)
    np.testing.assert_allclose(scores, 1 / 25, rtol=1e-13)


@pytest.mark.parametrize("nk,alpha,d", [(7, 2.0, 64), (130, 1.5, 80), (2, 4.0, 128)])
def test_one_hot_closed_form(nk, alpha, d):
    """Q rows = alpha*e1, key j* = alpha*e1, other keys 0: with c = exp(alpha^2/sqrt(d)),
    p(j*) = c / (c + Nk - 1) and every other key gets 1 / (c + Nk - 1)."""
    nq, H = 9, 3
    q = np.zeros((nq, H, d), np.float32)
    q[:, :, 0] = alpha
    k = np.zeros((nk, H, d), np.float32)
    jstar = nk // 2
    k[jstar, :, 0] = alpha
    cu_q = np.array([0, nq], np.int32)
    cu_k = np.array([0, nk], np.int32)
    lse, scores = oracle.importance(_bits(q), _bits(k), cu_q, cu_k)
    c = math.exp(alpha * alpha / math.sqrt(d))
    expect = np.full(nk, 1.0 / (c + nk - 1))
    expect[jstar] = c / (c + nk - 1)
    np.testing.assert_allclose(scores, expect, rtol=1e-13)
    np.testing.assert_allclose(lse, math.log(c + nk - 1), rtol=1e-13)


def test_explicit_scale_matches_closed_form():
    nq, nk, d = 3, 5, 16
    q = np.zeros((nq, 1, d), np.float32)
    q[:, :, 1] = 1.0
    k = np.zeros((nk, 1, d), np.float32)
    k[0, :, 1] = 2.0
    cu = np.array([0, nq], np.int32), np.array([0, nk], np.int32)
    _, scores = oracle.importance(_bits(q), _bits(k), *cu, softmax_scale=0.7)
    c = math.exp(2.0 * 0.7)
    assert abs(scores[0] - c / (c + nk - 1)) < 1e-14


def test_single_key_segment_scores_one():
    rng = np.random.default_rng(5)
    qb, kb, cu_q, cu_k = _rand_case(rng, [13, 4], [1, 9], 2, 1, 32, std=3.0)
    _, scores = oracle.importance(qb, kb, cu_q, cu_k)
    assert scores[0] == pytest.approx(1.0, abs=1e-15)


def test_segment_without_queries_scores_zero():
    rng = np.random.default_rng(6)
    qb, kb, cu_q, cu_k = _rand_case(rng, [0, 5], [6, 4], 2, 2, 16)
    lse, scores = oracle.importance(qb, kb, cu_q, cu_k)
    assert np.all(scores[:6] == 0)
    assert abs(scores[6:].sum() - 1) < 1e-12


def test_segment_without_keys_lse_is_minus_inf():
    rng = np.random.default_rng(7)
    qb, kb, cu_q, cu_k = _rand_case(rng, [3, 5], [0, 4], 2, 2, 16)
    lse, scores = oracle.importance(qb, kb, cu_q, cu_k)
    assert np.all(np.isneginf(lse[:, :3]))
    assert np.all(np.isfinite(lse[:, 3:]))


# ---------------------------------------------------------------------------
# Symmetries
# ---------------------------------------------------------------------------

def test_key_permutation_permutes_scores_and_query_permutation_does_not_matter():
    rng = np.random.default_rng(8)
    qb, kb, cu_q, cu_k = _rand_case(rng, [31], [45], 4, 2, 32, std=2.0)
    _, base = oracle.importance(qb, kb, cu_q, cu_k)
    perm = rng.permutation(45)
    _, s_k = oracle.importance(qb, kb[perm], cu_q, cu_k)
    np.testing.assert_allclose(s_k, base[perm], rtol=1e-12)
    qperm = rng.permutation(31)
    lse0, _ = oracle.importance(qb, kb, cu_q, cu_k)
    lse1, s_q = oracle.importance(qb[qperm], kb, cu_q, cu_k)
    np.testing.assert_allclose(s_q, base, rtol=1e-12)
    np.testing.assert_allclose(lse1, lse0[:, qperm], rtol=1e-12)


def test_segments_are_independent():
    """Block-diagonal attention: one call over two segments equals two calls."""
    rng = np.random.default_rng(9)
    qb, kb, cu_q, cu_k = _rand_case(rng, [20, 35], [28, 11], 4, 4, 16, std=2.0)
    lse, scores = oracle.importance(qb, kb, cu_q, cu_k)
    l0, s0 = oracle.importance(qb[:20], kb[:28], [0, 20], [0, 28])
    l1, s1 = oracle.importance(qb[20:], kb[28:], [0, 35], [0, 11])
    np.testing.assert_allclose(scores, np.concatenate([s0, s1]), rtol=1e-13)
    np.testing.assert_allclose(lse, np.concatenate([l0, l1], axis=1), rtol=1e-13)


def test_gqa_equals_mha_with_replicated_kv_heads():
    """Query head h reads KV head h // (H / Hkv) (consecutive groups)."""
    rng = np.random.default_rng(10)
    H, Hkv = 8, 2
    qb, kb, cu_q, cu_k = _rand_case(rng, [17, 9], [23, 30], H, Hkv, 16, std=2.0)
    lse_g, s_g = oracle.importance(qb, kb, cu_q, cu_k)
    kb_mha = np.repeat(kb, H // Hkv, axis=1)     # head h <- kv head h // 4
    lse_m, s_m = oracle.importance(qb, kb_mha, cu_q, cu_k)
    np.testing.assert_allclose(s_g, s_m, rtol=1e-14)
    np.testing.assert_allclose(lse_g, lse_m, rtol=1e-14)
    # Tiling instead of repeating would map head h to kv head h % 2: different.
    _, s_t = oracle.importance(qb, np.tile(kb, (1, H // Hkv, 1)), cu_q, cu_k)
    assert np.max(np.abs(s_t - s_g)) > 1e-6


def test_sink_key_draws_the_most_attention():
    """A key scaled x4 (the workloads' 'sink' tokens) dominates the scores."""
    w = make_segments([64], [64], 2, 2, 32, seed=11, sink_counts=[1], hidden_dim=16)
    _, scores = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    sink = int(w.meta["sink_rows"][0])
    assert scores[sink] >= np.sort(scores)[-3]


# ---------------------------------------------------------------------------
# Budget (pinned by the pages' printed token counts)
# ---------------------------------------------------------------------------

def _golden_budget_rows():
    rows = []
    with open(os.path.join(GOLDEN, "budget_counts.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            a = line.split()
            rows.append(tuple(int(x) for x in a[:4]))
    return rows


def test_budget_counts_match_the_pages():
    rows = _golden_budget_rows()
    assert len(rows) == 5
    for visual, permille, text, total in rows:
        assert oracle.keep_count(visual, permille) + text == total


def test_budget_is_floor_not_round():
    # 0.3 * 3072 = 921.6 -> 921 (rounding would print 1064, the page prints 1063).
    assert oracle.keep_count(3072, 300) == 921
    assert oracle.keep_count(16384, 600) == 9830
    assert oracle.keep_count(16384, 800) == 13107
    assert oracle.keep_count(0, 500) == 0


# ---------------------------------------------------------------------------
# Top-B (brute force over tiny inputs with forced ties)
# ---------------------------------------------------------------------------

def _brute_keep(scores, B):
    """Token i is kept iff fewer than B tokens precede it in the total order
    (higher score, or equal score and lower index)."""
    n = len(scores)
    kept = []
    for i in range(n):
        before = sum(1 for j in range(n) if scores[j] > scores[i] or (scores[j] == scores[i] and j < i))
        if before < B:
            kept.append(i)
    return kept


def test_topk_brute_force_all_small_inputs():
    for n in range(0, 7):
        for vals in itertools.product([0.0, 1.0, 2.0], repeat=n):
            s = np.asarray(vals, np.float32)
            for B in range(0, n + 1):
                keep_idx, cu = oracle.select_topk(s, [0, n], [B])
                assert list(keep_idx) == _brute_keep(list(vals), B)
                assert list(cu) == [0, B]


def test_topk_pools_requests_independently_and_ascending():
    rng = np.random.default_rng(12)
    s = rng.integers(0, 5, size=40).astype(np.float32)
    off = [0, 10, 10, 31, 40]
    keep = [3, 0, 21, 4]
    keep_idx, cu = oracle.select_topk(s, off, keep)
    assert list(cu) == [0, 3, 3, 24, 28]
    for r in range(4):
        part = keep_idx[cu[r]:cu[r + 1]]
        assert np.all(np.diff(part) > 0)
        local = _brute_keep(list(s[off[r]:off[r + 1]]), keep[r])
        assert list(part - off[r]) == local


def test_topk_all_equal_keeps_lowest_indices():
    s = np.full(17, 0.25, np.float32)
    keep_idx, _ = oracle.select_topk(s, [0, 17], [5])
    assert list(keep_idx) == [0, 1, 2, 3, 4]


def test_topk_compares_in_the_given_precision():
    # Two values equal in fp32 but different in fp64 tie in fp32.
    a = np.float64(0.1)
    b = np.float64(np.nextafter(0.1, 1.0))
    assert np.float32(a) == np.float32(b)
    s64 = np.array([a, b])
    assert list(oracle.select_topk(s64, [0, 2], [1])[0]) == [1]
    assert list(oracle.select_topk(s64.astype(np.float32), [0, 2], [1])[0]) == [0]


# ---------------------------------------------------------------------------
# Compaction
# ---------------------------------------------------------------------------

def test_gather_compact_hand_example():
    hidden = np.arange(10 * 3, dtype=np.uint16).reshape(10, 3)
    pos = np.stack([np.arange(10), 100 + np.arange(10)], axis=1).astype(np.int32)
    cu = [0, 4, 4, 7, 10]            # images of 4, 0, 3, 3 tokens
    keep_idx = np.array([1, 3, 4, 8, 9], np.int32)
    oh, op, img, cuk = oracle.gather_compact(hidden, pos, cu, keep_idx)
    assert oh.tolist() == [[3, 4, 5], [9, 10, 11], [12, 13, 14], [24, 25, 26], [27, 28, 29]]
    assert op[:, 1].tolist() == [101, 103, 104, 108, 109]
    assert img.tolist() == [0, 0, 2, 3, 3]
    assert cuk.tolist() == [0, 2, 2, 3, 5]


def test_end_to_end_invariants():
    w = make_segments([40, 70, 18], [40, 70, 18], 4, 2, 32, seed=13, sink_counts=[2, 2, 1],
                      hidden_dim=24, pos_dim=3, keep_per_req=[60])
    out = oracle.prune(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k, w.req_tok_offsets,
                       w.keep_per_req, w.hidden_bits, w.pos)
    k = out["keep_idx"]
    assert k.shape == (60,) and np.all(np.diff(k) > 0)
    assert out["cu_seqlens_kept"][-1] == 60
    assert np.array_equal(out["hidden"], w.hidden_bits[k])
    # every kept score >= every dropped score
    s = out["scores"]
    dropped = np.setdiff1d(np.arange(128), k)
    assert s[k].min() >= s[dropped].max()


# ---------------------------------------------------------------------------
# FP8 E4M3 inputs (LiteVLM's FP8 deployment)
# ---------------------------------------------------------------------------

def test_e4m3_decode_known_codes():
    """Values fixed by the OCP FP8 E4M3 definition (bias 7, 3 mantissa bits,
    subnormals below 2^-6, max 448, S.1111.111 = NaN)."""
    codes = np.array([0x00, 0x38, 0x40, 0x7E, 0x01, 0x07, 0x08, 0x37, 0x80, 0xB8, 0xFE], np.uint8)
    expect = [0.0, 1.0, 2.0, 448.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 0.9375, -0.0, -1.0, -448.0]
    got = oracle.e4m3_bits_to_f64(codes)
    assert list(got) == expect
    assert np.isnan(oracle.e4m3_bits_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_is_monotone_with_one_ulp_steps():
    v = oracle.e4m3_bits_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)
    # within each binade of normals the spacing is 2^(e-10); subnormals step 2^-9
    steps = np.diff(v)
    for code in range(1, 0x7E):
        e = max(code >> 3, 1)
        assert steps[code] == 2.0 ** (e - 10) or (code & 7) == 7


def test_e4m3_quantiser_is_nearest_ties_even_and_saturating():
    rng = np.random.default_rng(20)
    x = np.concatenate([rng.normal(0, 50, 2000), [0.0, -0.0, 500.0, -1e9, 2.0 ** -10, 3 * 2.0 ** -11]])
    bits = f32_to_e4m3_bits(x)
    table = oracle.e4m3_bits_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    dec = oracle.e4m3_bits_to_f64(bits)
    for xi, di, bi in zip(x, dec, bits):
        a = min(abs(xi), 448.0)
        best = np.min(np.abs(table - a))
        assert abs(abs(di) - a) == best
        if best > 0 and np.sum(np.abs(table - a) == best) == 2:
            assert (int(bi) & 1) == 0          # tie -> even code
    assert dec[-4] == 448.0 and dec[-3] == -448.0


def test_importance_with_e4m3_inputs_one_hot_closed_form():
    nq, nk, d, H = 5, 40, 64, 2
    q = np.zeros((nq, H, d), np.uint8)
    q[:, :, 0] = 0x40            # 2.0
    k = np.zeros((nk, H, d), np.uint8)
    k[7, :, 0] = 0x40
    lse, scores = oracle.importance(q, k, [0, nq], [0, nk], fmt="e4m3")
    c = math.exp(4.0 / 8.0)
    assert abs(scores[7] - c / (c + nk - 1)) < 1e-13
    assert abs(scores[0] - 1 / (c + nk - 1)) < 1e-13
    np.testing.assert_allclose(lse, math.log(c + nk - 1), rtol=1e-13)


# ---------------------------------------------------------------------------
# SUM normalisation
# ---------------------------------------------------------------------------

def test_sum_normalisation_totals_heads_times_query_rows():
    """Total attention received: a segment's sums add up to H * Nq_g (each of
    its H * Nq_g query rows spreads probability 1), and a segment without
    query rows gets 0."""
    rng = np.random.default_rng(41)
    lq, lk, H, Hkv = [20, 0, 7], [33, 5, 64], 4, 2
    qb, kb, cu_q, cu_k = _rand_case(rng, lq, lk, H, Hkv, 32, std=2.0)
    _, s_sum = oracle.importance(qb, kb, cu_q, cu_k, norm="sum")
    for g in range(3):
        seg = s_sum[cu_k[g]:cu_k[g + 1]]
        assert abs(seg.sum() - H * lq[g]) < 1e-9 * max(1, H * lq[g])
    assert np.all(s_sum[cu_k[1]:cu_k[2]] == 0)
    # one-hot closed form in sum mode: the hot key collects c/(c+Nk-1) per row
    nq, nk, d, alpha = 6, 9, 16, 3.0
    q = np.zeros((nq, 1, d), np.float32)
    q[:, 0, 0] = alpha
    k = np.zeros((nk, 1, d), np.float32)
    k[4, 0, 0] = alpha
    _, s = oracle.importance(_bits(q), _bits(k), [0, nq], [0, nk], norm="sum")
    c = math.exp(alpha * alpha / math.sqrt(d))
    assert s[4] == pytest.approx(nq * c / (c + nk - 1), rel=1e-12)
    assert s[0] == pytest.approx(nq / (c + nk - 1), rel=1e-12)


# ---------------------------------------------------------------------------
# Dynamic keep ratio (mass budget)
# ---------------------------------------------------------------------------

def test_score_quanta_closed_forms():
    # max 1.0 lies in [2^0, 2^1): E = 1, quanta = s * 2^23
    assert oracle.score_quanta([1.0, 0.5, 0.25, 0.0]) == [1 << 23, 1 << 22, 1 << 21, 0]
    # max 0.75 lies in [2^-1, 2^0): E = 0, quanta = floor(s * 2^24)
    assert oracle.score_quanta([0.75, 1e-9, 0.3]) == [12582912, 0, int(math.floor(0.3 * 2 ** 24))]
    assert oracle.score_quanta([0.0, 0.0]) == [0, 0]
    assert oracle.score_quanta([]) == []
    # quanta never reach 2^24 and the largest is at least 2^23
    q = oracle.score_quanta(np.random.default_rng(5).random(1000).astype(np.float32))
    assert max(q) < 1 << 24 and max(q) >= 1 << 23


def _budget_brute(s, tau):
    """Smallest B whose top-B quanta reach ceil(tau * M / 1000), by trying every B."""
    q = oracle.score_quanta(s)
    M = sum(q)
    T = -(-M * tau // 1000)
    order = sorted(range(len(s)), key=lambda j: (-float(s[j]), j))
    for b in range(len(s) + 1):
        if sum(q[j] for j in order[:b]) >= T:
            return b
    raise AssertionError("unreachable")


def test_dynamic_budget_brute_force_small_inputs():
    vals = [0.0, 0.25, 0.5, 1.0]
    for n in range(0, 5):
        for combo in itertools.product(vals, repeat=n):
            s = np.asarray(combo, dtype=np.float32)
            for tau in (0, 1, 333, 500, 900, 1000):
                got = oracle.dynamic_budget(s, [0, n], tau, 0, 1000)
                assert got.tolist() == [_budget_brute(s, tau)], (combo, tau)


def test_dynamic_budget_closed_forms_and_bounds():
    # uniform scores: B = ceil(n * tau / 1000)
    for n, tau in [(7, 500), (1000, 900), (13, 1), (64, 1000)]:
        s = np.full(n, 0.01, np.float32)
        assert oracle.dynamic_budget(s, [0, n], tau, 0, 1000)[0] == -(-n * tau // 1000)
    # one token holding all the mass: B = 1 for any tau > 0
    s = np.zeros(50, np.float32)
    s[17] = 0.9
    assert oracle.dynamic_budget(s, [0, 50], 999, 0, 1000)[0] == 1
    # tau = 1000 keeps every token with a nonzero quantum
    s = np.asarray([0.5, 1e-12, 0.25, 0.0, 0.125], np.float32)
    assert oracle.dynamic_budget(s, [0, 5], 1000, 0, 1000)[0] == 3
    # floor and ceiling ratios
    assert oracle.dynamic_budget(np.full(100, 0.1, np.float32), [0, 100], 0, 200, 1000)[0] == 20
    assert oracle.dynamic_budget(np.full(100, 0.1, np.float32), [0, 100], 1000, 0, 750)[0] == 75
    # requests are independent; an empty request keeps 0
    s = np.concatenate([np.full(10, 0.2, np.float32), np.zeros(0, np.float32),
                        np.asarray([1.0, 0.0, 0.0], np.float32)])
    assert oracle.dynamic_budget(s, [0, 10, 10, 13], 500, 0, 1000).tolist() == [5, 0, 1]


def test_dynamic_budget_invariances():
    rng = np.random.default_rng(6)
    s = (rng.random(300) ** 4).astype(np.float32)
    b = oracle.dynamic_budget(s, [0, 300], 800, 0, 1000)[0]
    # scaling by a power of two leaves the quanta, hence B, unchanged
    assert oracle.dynamic_budget(s * np.float32(8.0), [0, 300], 800, 0, 1000)[0] == b
    # permuting the tokens leaves B unchanged
    assert oracle.dynamic_budget(s[rng.permutation(300)], [0, 300], 800, 0, 1000)[0] == b
    # concentrating the same ranking raises the top tokens' share: B cannot grow
    assert oracle.dynamic_budget(s ** 2, [0, 300], 800, 0, 1000)[0] <= b
