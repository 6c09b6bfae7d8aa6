"""tsel_importance_noalloc: importance scores for callers that cannot
allocate device memory (an engine plugin whose memory pool already owns all
of HBM, or an embedded stack that forbids allocation after start-up) and so
cannot lend a workspace either. Its scratch is a static device array inside
the library.

The entry point is called through the C ABI (ctypes, raw device pointers)
and compared with tsel_importance and with the fp64 oracle on two different
problems in a row, so a second call must not be disturbed by what the first
one left in the shared array. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_util import REL_TOL, bits_to_bf16, i32, max_rel_err, segment_slice


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


def _noalloc(lib, w, cu_k=None, with_status=True):
    q, k = bits_to_bf16(w.q_bits), bits_to_bf16(w.k_bits)
    cu_q = i32(w.cu_seqlens_q)
    cu_k = i32(w.cu_seqlens_k if cu_k is None else cu_k)
    scores = torch.full((w.total_k,), -1.0, dtype=torch.float32, device="cuda")
    lse = torch.full((w.num_heads, w.total_q), -1.0, dtype=torch.float32, device="cuda")
    status = torch.full((1,), 0xFF, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = lib.tsel_importance_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_int64(0), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_int64(0), ctypes.c_void_p(cu_q.data_ptr()), ctypes.c_void_p(cu_k.data_ptr()),
        w.num_seg, w.total_q, w.total_k, w.max_seqlen_q, w.max_seqlen_k, w.num_heads,
        w.num_kv_heads, w.head_dim, ctypes.c_float(0.0), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(scores.data_ptr()),
        ctypes.c_void_p(status.data_ptr()) if with_status else None, ctypes.c_void_p(stream))
    torch.cuda.synchronize()
    return st, scores.cpu().numpy(), lse.cpu().numpy(), int(status.item())


def _mixed():
    return W.make_segments([300, 1, 129, 1024], [77, 5, 129, 1024], 8, 2, 128, seed=404,
                           sink_counts=[3, 0, 2, 20], hidden_dim=16)


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point_and_oracle_twice_in_a_row(lib):
    first = W.make("thirty_images")              # the 30-image request (about 6 MB of scratch)
    second = _mixed()
    for w in (first, second):
        st, s, lse, status = _noalloc(lib, w)
        assert st == 0, lib.tsel_last_error().decode()
        assert status == 0
        s_ref, lse_ref = _regular(w)
        assert max_rel_err(s, s_ref.astype(np.float64)) <= REL_TOL
        fin = np.isfinite(lse_ref)
        np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=1e-6, atol=1e-6)
        assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
        # against the fp64 oracle: whole images (attention is block-diagonal,
        # so an image's scores depend on that image alone)
        lens = np.diff(w.cu_seqlens_k)
        sample = sorted({int(np.argmin(lens)), int(np.argmax(lens)), w.num_seg // 2})
        for g in sample:
            qb, kb, cq, ck, (q0, q1, k0, k1) = segment_slice(w, g)
            lse_o, s_o = oracle.importance(qb, kb, cq, ck)
            assert max_rel_err(s[k0:k1], s_o) <= REL_TOL, g
            fin = np.isfinite(lse_o)
            np.testing.assert_allclose(lse[:, q0:q1][fin], lse_o[fin], rtol=1e-5, atol=1e-4)


@pytest.mark.gpu
def test_noalloc_status_word_belongs_to_each_call(lib):
    """The shared array's status word is cleared at the start of every call:
    a malformed call reports its bit, the clean call after it reports none,
    and a call without a status output still computes the scores."""
    w = _mixed()
    bad = np.array(w.cu_seqlens_k, dtype=np.int64)
    bad[1], bad[2] = bad[2], bad[1]                     # not monotone
    st, _, _, status = _noalloc(lib, w, cu_k=bad)
    assert st == 0
    assert status & 0x1                                 # TSEL_DEV_SEQLENS
    st, s, _, status = _noalloc(lib, w)
    assert st == 0 and status == 0
    st, s2, _, status = _noalloc(lib, w, with_status=False)
    assert st == 0
    assert status == 0xFF                               # untouched: no status pointer passed
    assert np.array_equal(s.view(np.uint32), s2.view(np.uint32))
    _, s_o = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k)
    assert max_rel_err(s2, s_o) <= REL_TOL


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


class _FakeCudaTensor:
    """Just enough of a CUDA tensor for the binding's input checks (no GPU)."""

    def __init__(self, shape, dtype, strides=None):
        self.shape = tuple(shape)
        self.dtype = dtype
        self.is_cuda = True
        self.device = torch.device("cuda", 0)
        if strides is None:
            strides, acc = [], 1
            for n in reversed(self.shape):
                strides.insert(0, acc)
                acc *= n
        self._strides = tuple(strides)

    def dim(self):
        return len(self.shape)

    def stride(self, i):
        return self._strides[i]

    def numel(self):
        return int(np.prod(self.shape))


def test_binding_rejects_int64_seqlens_and_transposed_heads():
    import attention_score_vision_gb300 as tsel
    q = _FakeCudaTensor((10, 2, 64), torch.bfloat16)
    cu32 = _FakeCudaTensor((3,), torch.int32)
    cu64 = _FakeCudaTensor((3,), torch.int64)
    qt = _FakeCudaTensor((10, 2, 64), torch.bfloat16, strides=(128, 1, 2))   # heads innermost
    for fn in (tsel.tsel_importance, tsel.tsel_importance_noalloc):
        with pytest.raises(TypeError):
            fn(q, q, cu64, cu32, 8, 8)
        with pytest.raises(TypeError):
            fn(q, q, cu32, cu64, 8, 8)
        with pytest.raises(ValueError):
            fn(qt, q, cu32, cu32, 8, 8)
        with pytest.raises(ValueError):
            fn(q, qt, cu32, cu32, 8, 8)
