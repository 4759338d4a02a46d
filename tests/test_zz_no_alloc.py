"""satk_dcp_rescue_select_noalloc against satk_dcp_rescue_select.

The no-allocation variant is for callers that cannot hand the library a
scratch buffer (they only hold pointers to their own inputs and outputs, or
may not call an allocator where they run): its scratch is a fixed array in
the library's device memory.  Its results must be those of the ordinary
entry point, which takes the scratch from the caller.  Two calls in a row
check that a call is not disturbed by what the previous one left in the
shared array.  Called through the C ABI with ctypes.

This file is named to be collected last, and must pass both alone in a
fresh process and after the other tests.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import sparse_attention_indexer_radix_gb300 as satk
from sparse_attention_indexer_radix_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MAX_WORDS = 2 * 1024 * 1024  # SATK_RESCUE_NOALLOC_MAX_WORDS


def _lib():
    from sparse_attention_indexer_radix_gb300 import build as satk_build
    satk_build.build()
    L = binding.lib()
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f = L.satk_dcp_rescue_select_noalloc
    f.argtypes = [vp, i32, i64, i32, i32, vp, i64, i64, vp, vp, vp, i64, vp, vp]
    f.restype = ctypes.c_int
    return L


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _round1(W, T, S, n, k, skew_count, seed):
    lg, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=skew_count,
                                   seed=seed, device=DEV)
    local = satk.topk_rows(lg.view(W * T, S), n)
    packed = satk.dcp_pack(lg.view(W * T, S), local).view(W, T, n + n // 32)
    sat = torch.zeros(T, dtype=torch.int32, device=DEV)
    ids1 = satk.dcp_merge_select(packed, k, packed=True, sat_word=sat)
    return lg, packed, sat, ids1


@pytest.mark.parametrize("W,T,S,n,k,skew", [(4, 12, 3000, 64, 512, 120),
                                            (8, 128, 65536, 384, 2048, 600)])
def test_noalloc_matches_rescue_with_caller_scratch(W, T, S, n, k, skew):
    L = _lib()
    lg, packed, sat, ids1 = _round1(W, T, S, n, k, skew, seed=1237)
    assert satk.rescue_recv_words(T, n, k) <= MAX_WORDS
    assert int(((sat >> 16) != 0).sum()) > 0, "the workload must exercise the rescue"
    # the ordinary entry point, scratch from the caller
    want = ids1.clone()
    st_want = torch.zeros(1, dtype=torch.int32, device=DEV)
    satk.dcp_rescue_select(packed, lg, sat, want, k, status=st_want)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        got = ids1.clone()
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        rc = L.satk_dcp_rescue_select_noalloc(_p(packed), W, T, n, k, _p(lg), S, S, None,
                                              _p(sat), _p(got), k, _p(st), stream)
        assert rc == 0, f"call {call}: rc {rc}"
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"call {call}: ids differ from the ordinary entry point"
        assert int(st.item()) == int(st_want.item())
    assert not torch.equal(want, ids1), "the rescue changed no row"


def test_noalloc_rejects_requests_beyond_its_scratch():
    L = _lib()
    T, n, k = 1_000_000, 64, 512  # T * 7 * 528 words: far beyond the array
    assert satk.rescue_recv_words(T, n, k) > MAX_WORDS
    dummy = torch.zeros(16, dtype=torch.int32, device=DEV)
    rc = L.satk_dcp_rescue_select_noalloc(_p(dummy), 8, T, n, k, _p(dummy), 100, 100, None,
                                          _p(dummy), _p(dummy), k, None, None)
    assert rc == -2  # SATK_EUNSUPPORTED, nothing launched
    torch.cuda.synchronize()
    assert np.all(dummy.cpu().numpy() == 0)
