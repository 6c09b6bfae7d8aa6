"""Row-LSE pass, fixed reference and redo launch.

The row-LSE pass fixes each row's reference max on its first 64 keys; a row
whose later logits climb ~128 (log2) above it overflows the fp32 sum, and its
(head, 256-row query pair) is redone by a second launch with a moving
reference. These inputs put keys with a controlled logit gap into every
segment (gap ~128 nats: overflow; ~55 nats: large but finite terms) and check
the number of redone pairs exactly and the results against the fp64 oracle,
with and without key chunks, on bf16 and E4M3 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import REL_TOL, check_selection_exact, max_rel_err, run_path, to_device

pytestmark = pytest.mark.gpu

# keys at local position 100 (and 400 where a segment is that long): past the
# first 64 keys of the first tile, so the fixed reference never sees them
FAR = [100, 400]


@pytest.fixture(scope="module")
def tsel():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_score_vision_gb300 as t
    t.build()
    t.load_library()
    return t


def _expected_pairs(lengths, signs):
    """Pairs of every head whose queries see the far keys with a positive gap."""
    pairs = sum((int(n) + 255) // 256 for n in lengths if n > FAR[0])
    return pairs * sum(1 for s in signs if s > 0)


def _run(tsel, w, ws=None, flags=None):
    # these problems are below the size that picks the fixed reference by itself
    flags = tsel.TSEL_IMP_ROWREF_FIXED if flags is None else flags
    d = to_device(w)
    if ws is None:
        ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k,
                                                             w.num_heads), dtype=torch.uint8,
                         device="cuda")
    s, lse = tsel.tsel_importance(d["q"], d["k"], d["cu_q"], d["cu_k"], w.max_seqlen_q,
                                  w.max_seqlen_k, workspace=ws, flags=flags)
    torch.cuda.synchronize()
    return s.cpu().numpy(), lse.cpu().numpy(), tsel.tsel_importance_redo_pairs(ws), ws


def _check(w, s, lse, fmt="bf16"):
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                       w.softmax_scale, fmt=fmt)
    assert max_rel_err(s, s_ref) <= REL_TOL
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-5, atol=2e-4)


CASES = {
    # 16 heads over 9 query pairs: one key chunk per unit
    "whole_rows": dict(lengths=[300, 520, 129, 256, 295], H=16, Hkv=8, d=64,
                       signs=[1] * 8 + [-1] * 8),
    # 4 heads: key chunks (the 520-key segment in two), mixed with unsplit segments
    "key_chunks": dict(lengths=[300, 520, 129], H=4, Hkv=2, d=64, signs=[1, 1, -1, -1]),
    # one 2048-token segment, two heads on one KV head: eight key chunks (the
    # second head keeps every score above the fp32 normal range)
    "one_long": dict(lengths=[2048], H=2, Hkv=1, d=128, signs=[1, -1]),
}


def _case(name, gap_nats, seed):
    """Far keys whose logit stands about gap_nats above the rest (q_lead 4)."""
    c = CASES[name]
    far_value = gap_nats * np.sqrt(c["d"]) / 4.0
    return W.make_far_keys(c["lengths"], c["H"], c["Hkv"], c["d"], seed=seed, far_positions=FAR,
                           far_value=far_value, head_signs=c["signs"], name=name)


@pytest.mark.parametrize("name", sorted(CASES))
def test_overflowing_rows_are_redone(tsel, name):
    c = CASES[name]
    w = _case(name, 128.0, seed=900 + len(name))   # gap ~128 nats: 2^185 overflows
    s, lse, redo, _ = _run(tsel, w)
    assert redo == _expected_pairs(c["lengths"], c["signs"])
    _check(w, s, lse)


def test_overflow_redo_full_path(tsel):
    w = _case("key_chunks", 128.0, seed=911)
    out = run_path(tsel, w)
    assert out["status"] == 0
    check_selection_exact(w, out)


def test_large_finite_terms_need_no_redo(tsel):
    # an overflowing call first, then one with a ~55-nat gap (terms up to
    # 2^80) on the same workspace: the schedule stage resets the queue
    _, _, redo, ws = _run(tsel, _case("whole_rows", 128.0, seed=920))
    assert redo > 0
    w = _case("whole_rows", 55.0, seed=921)
    s, lse, redo, _ = _run(tsel, w, ws)
    assert redo == 0
    _check(w, s, lse)


def test_no_redo_on_seeded_workloads(tsel):
    for name in ("single_image_256", "six_views_1536", "text_query_3072"):
        w = W.make(name)
        _, _, redo, _ = _run(tsel, w)
        assert redo == 0, name


@pytest.mark.parametrize("name", sorted(CASES))
def test_moving_reference_needs_no_redo(tsel, name):
    # the one-launch mode handles the same gap by moving its reference
    w = _case(name, 128.0, seed=940 + len(name))
    s, lse, redo, _ = _run(tsel, w, flags=tsel.TSEL_IMP_ROWREF_MOVING)
    assert redo == 0
    _check(w, s, lse)


def test_fixed_and_moving_reference_agree(tsel):
    w = W.make("six_views_1536")
    s_f, lse_f, _, _ = _run(tsel, w, flags=tsel.TSEL_IMP_ROWREF_FIXED)
    s_m, lse_m, _, _ = _run(tsel, w, flags=tsel.TSEL_IMP_ROWREF_MOVING)
    np.testing.assert_allclose(lse_f, lse_m, rtol=1e-6, atol=1e-5)
    np.testing.assert_allclose(s_f, s_m, rtol=1e-4, atol=0)


def test_overflow_redo_e4m3(tsel):
    c = CASES["key_chunks"]
    w = W.to_e4m3(_case("key_chunks", 128.0, seed=930))
    q = torch.from_numpy(w.q_bits).cuda()
    k = torch.from_numpy(w.k_bits).cuda()
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k, w.num_heads),
                     dtype=torch.uint8, device="cuda")
    cq = torch.from_numpy(w.cu_seqlens_q).cuda()
    ck = torch.from_numpy(w.cu_seqlens_k).cuda()
    s, lse = tsel.tsel_importance(q, k, cq, ck, w.max_seqlen_q, w.max_seqlen_k,
                                  softmax_scale=w.softmax_scale, workspace=ws,
                                  flags=tsel.TSEL_IMP_ROWREF_FIXED)
    assert tsel.tsel_importance_redo_pairs(ws) == _expected_pairs(c["lengths"], c["signs"])
    assert tsel.tsel_read_device_status(ws) == 0
    _check(w, s.cpu().numpy(), lse.cpu().numpy(), fmt="e4m3")
