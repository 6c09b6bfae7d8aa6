"""tsel_importance_noalloc: importance scores for callers that cannot
allocate device memory (an engine plugin whose memory pool already owns all
of HBM, or an embedded stack that forbids allocation after start-up) and so
cannot lend a workspace either. Its scratch is a static device array inside
the library.

The entry point is called through the C ABI (ctypes, raw device pointers)
and compared with tsel_importance on two different problems in a row, so a
second call must not be disturbed by what the first one left in the shared
array. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import REL_TOL, bits_to_bf16, i32, max_rel_err


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_score_vision_gb300 as tsel
    tsel.build()
    return tsel.load_library()


def _regular(w):
    import attention_score_vision_gb300 as tsel
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    s, lse = tsel.tsel_importance(q, k, i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), w.max_seqlen_q,
                                  w.max_seqlen_k)
    return s.cpu().numpy(), lse.cpu().numpy()


def _noalloc(lib, w):
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    cu_q, cu_k = i32(w.cu_seqlens_q), i32(w.cu_seqlens_k)
    scores = torch.full((w.total_k,), -1.0, dtype=torch.float32, device="cuda")
    lse = torch.full((w.num_heads, w.total_q), -1.0, dtype=torch.float32, device="cuda")
    status = torch.full((1,), 0xFF, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.tsel_importance_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_int64(0), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_int64(0), ctypes.c_void_p(cu_q.data_ptr()), ctypes.c_void_p(cu_k.data_ptr()),
        w.num_seg, w.total_q, w.total_k, w.max_seqlen_q, w.max_seqlen_k, w.num_heads,
        w.num_kv_heads, w.head_dim, ctypes.c_float(0.0), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(scores.data_ptr()), ctypes.c_void_p(status.data_ptr()),
        ctypes.c_void_p(stream))
    torch.cuda.synchronize()
    return st, scores.cpu().numpy(), lse.cpu().numpy(), int(status.item())


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point_twice_in_a_row(lib):
    first = W.make("thirty_images")              # the 30-image request (about 4.3 MB scratch)
    second = W.make_segments([300, 1, 129, 1024], [77, 5, 129, 1024], 8, 2, 128, seed=404,
                             sink_counts=[3, 0, 2, 20], hidden_dim=16)
    for w in (first, second):
        st, s, lse, status = _noalloc(lib, w)
        assert st == 0, lib.tsel_last_error().decode()
        assert status == 0
        s_ref, lse_ref = _regular(w)
        assert max_rel_err(s, s_ref.astype(np.float64)) <= REL_TOL
        fin = np.isfinite(lse_ref)
        np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=1e-6, atol=1e-6)
        assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_the_static_scratch(lib):
    # 64 heads over 262144 query tokens needs far more than 16 MiB of scratch;
    # the check happens on the host before any pointer is touched.
    st = lib.tsel_importance_noalloc(ctypes.c_void_p(16), ctypes.c_int64(0), ctypes.c_void_p(16),
                                     ctypes.c_int64(0), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                     1, 262144, 262144, 262144, 262144, 64, 64, 64,
                                     ctypes.c_float(0.0), None, ctypes.c_void_p(16), None, None)
    assert st == 3
    assert "static" in lib.tsel_last_error().decode()
