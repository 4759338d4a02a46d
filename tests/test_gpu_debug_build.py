"""The bounds-checking debug build on the GPU.

libsatk_debug.so is built from the same sources with -DSATK_DEBUG: before
every shared-memory list index, output position, histogram bin and scratch
index that the kernels rely on an invariant for, a check records a failure
in a device word (read by satk_debug_flags) and skips the access, instead
of trapping.  These tests route the same calls the other GPU tests make to
the debug library, check every result against the oracle and every output
buffer's guard canaries, and require the debug word to stay 0.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_radix_gb300 as satk
from guards import guarded
from sparse_attention_indexer_radix_gb300 import binding, inputs
from sparse_attention_indexer_radix_gb300 import build as satk_build

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dbg():
    L = binding.load(satk_build.build(debug=True))
    oracle.build()
    assert L.satk_debug_flags(1) != 0xFFFFFFFF
    return L


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _topk_case(x, k, ends, what, sorted=False):
    rows = x.shape[0]
    out, guard = guarded((rows, k + 3), fill=-7)
    satk.topk_rows(x.to(DEV), k, row_ends=None if ends is None else ends.to(DEV), out=out,
                   sorted=sorted)
    guard(what)
    host = _bits(x) if x.dtype == torch.bfloat16 else x.numpy()
    want = np.full((rows, k + 3), -7, dtype=np.int32)
    oracle.topk_rows(host, k, row_ends=None if ends is None else ends.numpy(), out=want,
                     sorted=sorted)
    assert np.array_equal(out.cpu().numpy(), want), what


def test_debug_build_row_paths(dbg):
    """Every row path (one warp, one CTA of 128 and of 256 threads, clusters,
    the score-sorted kernel), fp32 and bf16, with the exact fallback forced
    by few-level rows."""
    with binding.routed_to(dbg):
        x, ends = inputs.prefill(rows=64, cols=4096, seed=1235)
        _topk_case(x, 512, ends, "prefill smoke (warp rows)")
        x, ends = inputs.prefill(rows=48, cols=12000, seed=3)
        x[5] = torch.randint(0, 3, (12000,)).float()        # exact path
        _topk_case(x, 512, ends, "128-thread rows")
        x, ends = inputs.prefill(rows=40, cols=40000, seed=4)
        _topk_case(x, 2048, ends, "256-thread rows")
        x, _ = inputs.prefill(rows=4, cols=300000, seed=5, causal=False, dtype=torch.bfloat16)
        _topk_case(x, 384, None, "clustered rows")
        x, ends = inputs.prefill(rows=12, cols=9000, seed=6)
        _topk_case(x, 1000, ends, "score-sorted", sorted=True)
        x, ends = inputs.prefill(rows=40, cols=4096, seed=8)
        x[3] = torch.randint(0, 3, (4096,)).float()          # ties in the sort
        _topk_case(x, 512, ends, "score-sorted warp rows", sorted=True)
        _topk_case(x.to(torch.bfloat16), 100, ends, "score-sorted warp rows bf16", sorted=True)
        x, ends, _ = inputs.adversarial(rows=24, cols=20000, seed=7)
        _topk_case(x, 2048, ends, "adversarial bf16")
        torch.cuda.synchronize()
    assert dbg.satk_debug_flags(1) == 0


def test_debug_build_decode_pipeline(dbg):
    """The decode step (fused top-n pack, round-1 merge, rescue on both push
    kernels, emit_rows) and the pairs merge through the debug library."""
    with binding.routed_to(dbg):
        for S, ld_pad in ((65536, 0), (9000, 3)):
            W, T, n, k = 4, 16, 128, 1024
            lg, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_frac=0.5,
                                           skew_count=3 * n, seed=S)
            buf = torch.zeros((W, T, S + ld_pad), dtype=torch.bfloat16, device=DEV)
            buf[:, :, :S] = lg.to(DEV)
            flat = buf.view(W * T, S + ld_pad)[:, :S]
            packed, g_p = guarded((W, T, n + n // 32))
            satk.dcp_topk_pack(flat, n, out=packed.view(W * T, -1))
            sat, g_s = guarded((T,), fill=0)
            ids, g_i = guarded((T, k))
            st = torch.zeros(1, dtype=torch.int32, device=DEV)
            satk.dcp_merge_select(packed, k, packed=True, ids_out=ids, sat_word=sat, status=st)
            recv, g_r = guarded((satk.rescue_recv_words(T, n, k),), fill=0)
            satk.dcp_rescue_select(packed, buf[:, :, :S], sat, ids, k, recv=recv, status=st)
            table = torch.arange(T * (S // 64 + 1), dtype=torch.int32,
                                 device=DEV).view(T, -1)
            req = torch.arange(T, dtype=torch.int32, device=DEV)
            rows_out, g_ro = guarded((T, k))
            valid, g_v = guarded((T,))
            satk.dcp_emit_rows(ids, W, 1, req, table, 64, 64, rows_out=rows_out, valid_out=valid)
            torch.cuda.synchronize()
            for chk, what in ((g_p, "packed"), (g_s, "sat_word"), (g_i, "ids"), (g_r, "recv"),
                              (g_ro, "rows_out"), (g_v, "valid_out")):
                chk(what)
            bits = _bits(lg)
            o_local = oracle.topk_rows(bits.reshape(W * T, S), n)
            o_packed = oracle.dcp_pack(bits.reshape(W * T, S), o_local).reshape(W, T, -1)
            o_ids, o_sat, _ = oracle.merge_packed(o_packed, k)
            o_ids, _, _ = oracle.rescue(o_packed, k, bits, o_sat, o_ids)
            assert np.array_equal(packed.cpu().numpy(), o_packed)
            assert np.array_equal(sat.cpu().numpy(), o_sat)
            assert np.array_equal(ids.cpu().numpy(), o_ids)
            o_rows, o_valid, _ = oracle.emit_rows(o_ids, W, 1, req.cpu().numpy(),
                                                  table.cpu().numpy(), 64, 64)
            assert np.array_equal(rows_out.cpu().numpy(), o_rows)
            assert np.array_equal(valid.cpu().numpy(), o_valid)
        cand = inputs.pairs_merge(W=8, rows=24, k=2048, local=8192, seed=9, device=DEV)
        ids, g = guarded((24, 2048))
        satk.dcp_merge_select(cand, 2048, packed=False, ids_out=ids)
        torch.cuda.synchronize()
        g("pairs ids")
        assert np.array_equal(ids.cpu().numpy(), oracle.merge_pairs(cand.cpu().numpy(), 2048))
    assert dbg.satk_debug_flags(1) == 0
