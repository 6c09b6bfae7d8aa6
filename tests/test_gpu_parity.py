"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Importance scores: max relative error <= 2e-3 (bf16 inputs, fp32 accumulate).
Top-B and compaction: bit-exact when fed the same fp32 scores.
End to end: the keep set equals the oracle's except for tokens whose oracle
score lies within 2e-3 of the B-th score.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import (REL_TOL, check_keep_set_agreement, check_selection_exact, max_rel_err,
                      oracle_full, run_path, segment_slice, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsel():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_score_vision_gb300 as t
    t.build()
    t.load_library()
    return t


@pytest.mark.parametrize("name", ["single_image_256", "six_views_1536", "text_query_3072"])
def test_small_workloads_full_oracle(tsel, name):
    w = W.make(name)
    out = run_path(tsel, w)
    assert out["status"] == 0
    lse_ref, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    err = max_rel_err(out["scores"], s_ref)
    assert err <= REL_TOL, err
    np.testing.assert_allclose(out["lse"], lse_ref, rtol=1e-5, atol=1e-4)
    check_selection_exact(w, out)
    check_keep_set_agreement(w, out, s_ref)


@pytest.mark.parametrize("name", ["thirty_images", "batch_8x16x1024"])
def test_full_size_workloads_sampled(tsel, name):
    """Full size, in the launch configuration the benchmark times; the oracle
    recomputes a sample of whole images (attention is block-diagonal, so one
    image's scores depend on that image alone)."""
    w = W.make(name)
    out = run_path(tsel, w)
    assert out["status"] == 0
    s = out["scores"]
    assert np.all(np.isfinite(s)) and np.all(s > 0)
    lens = np.diff(w.cu_seqlens_k)
    # every segment's scores sum to 1 (total importance = heads x query rows)
    for g in range(w.num_seg):
        tot = s[w.cu_seqlens_k[g]:w.cu_seqlens_k[g + 1]].astype(np.float64).sum()
        assert abs(tot - 1.0) <= REL_TOL, (g, tot)
    rng = np.random.default_rng(7)
    sample = sorted({int(np.argmin(lens)), int(np.argmax(lens)), *rng.choice(w.num_seg, 2, replace=False).tolist()})
    for g in sample:
        qb, kb, cq, ck, (q0, q1, k0, k1) = segment_slice(w, g)
        lse_ref, s_ref = oracle.importance(qb, kb, cq, ck)
        err = max_rel_err(s[k0:k1], s_ref)
        assert err <= REL_TOL, (g, err)
        np.testing.assert_allclose(out["lse"][:, q0:q1], lse_ref, rtol=1e-5, atol=1e-4)
    check_selection_exact(w, out)


@pytest.mark.parametrize("name", ["thirty_images", "batch_8x16x1024"])
def test_full_size_workloads_full_oracle_keep_set(tsel, name):
    """Full size against the oracle over every image (segments spread over
    host processes): every score within 2e-3, and the end-to-end keep set
    equal to the oracle's except for tokens within 2e-3 of a request's B-th
    oracle score (the 8-request batch: every request's pool)."""
    w = W.make(name)
    out = run_path(tsel, w)
    assert out["status"] == 0
    lse_ref, s_ref = oracle_full(name)
    assert max_rel_err(out["scores"], s_ref) <= REL_TOL
    np.testing.assert_allclose(out["lse"], lse_ref, rtol=1e-5, atol=1e-4)
    check_selection_exact(w, out)
    check_keep_set_agreement(w, out, s_ref)


def test_varlen_pool_end_to_end(tsel):
    """Images of very different sizes share one budget (unified candidate pool)."""
    L = [1, 127, 128, 129, 300, 700, 1000, 64]
    w = W.make_segments(L, L, 8, 8, 80, seed=101, sink_counts=[0, 2, 3, 3, 6, 14, 20, 1],
                        key_scales=[1, 0.5, 2, 1, 1.5, 0.7, 1, 1.2], hidden_dim=1280, pos_dim=3,
                        keep_per_req=[W.keep_floor(sum(L), 600)])
    out = run_path(tsel, w)
    assert out["status"] == 0
    _, s_ref = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(out["scores"], s_ref) <= REL_TOL
    check_selection_exact(w, out)
    check_keep_set_agreement(w, out, s_ref)


def test_determinism_bitwise(tsel):
    w = W.make("six_views_1536")
    dev = to_device(w)
    a = run_path(tsel, w, dev)
    for _ in range(3):
        b = run_path(tsel, w, dev)
        assert np.array_equal(a["scores"].view(np.uint32), b["scores"].view(np.uint32))
        assert np.array_equal(a["keep_idx"], b["keep_idx"])


@pytest.mark.parametrize("flags_name", ["TSEL_IMP_ROWREF_FIXED", "TSEL_IMP_ROWREF_MOVING"])
def test_determinism_bitwise_uneven_units(tsel, flags_name):
    """Images of 256..4096 tokens give units with odd B-tile counts, so which
    epilogue warpgroup takes the even tiles of a unit changes with the
    scheduling history of its CTA; the row LSE and the scores must not."""
    w = W.make("thirty_images")
    dev = to_device(w)
    flags = getattr(tsel, flags_name)
    ws = torch.zeros(tsel.tsel_importance_workspace_size(w.num_seg, w.total_q, w.total_k,
                                                         w.num_heads), dtype=torch.uint8,
                     device="cuda")
    ref = None
    for _ in range(4):
        s, lse = tsel.tsel_importance(dev["q"], dev["k"], dev["cu_q"], dev["cu_k"], w.max_seqlen_q,
                                      w.max_seqlen_k, flags=flags, workspace=ws)
        got = (s.view(torch.int32).cpu().numpy(), lse.view(torch.int32).cpu().numpy())
        if ref is None:
            ref = got
        else:
            assert np.array_equal(ref[0], got[0])
            assert np.array_equal(ref[1], got[1])
    assert tsel.tsel_read_device_status(ws) == 0
