"""The entry points on side streams and inside CUDA graphs.

No entry point allocates, copies or synchronises, so every call captures
into a CUDA graph: the three row paths (one warp per row, one CTA per row,
a cluster per row, plus the score-sorted variant) and a whole decode step
(local top-N, pack, merge, rescue, emit_rows).  Replays must match the
oracle bit for bit, and must follow new input data written in place into
the captured buffers between replays."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_radix_gb300 as satk
from sparse_attention_indexer_radix_gb300 import inputs
from test_gpu_parity import (CANARY, DEV, _compare_decode, _decode_oracle, assert_rows_equal,
                             bits_of, host_view)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_indexer_radix_gb300 import build as satk_build
    satk_build.build()
    oracle.build()


# (rows, cols, dtype, k, sorted): 9000 fp32 columns take one warp per row,
# 16000 bf16 columns one CTA per row, 8 rows of 300000 a cluster per row;
# score-sorted: 20001 columns on the CTA path, 8192 on the warp path
ROW_CASES = [(64, 9000, torch.float32, 512, False), (16, 16000, torch.bfloat16, 512, False),
             (8, 300000, torch.float32, 512, False), (12, 20001, torch.float32, 1000, True),
             (24, 8192, torch.float32, 512, True)]


def _row_inputs(seed):
    xs, ends = [], []
    for j, (rows, cols, dtype, _, _) in enumerate(ROW_CASES):
        x, e = inputs.prefill(rows=rows, cols=cols, seed=seed + j, dtype=torch.float32)
        g = torch.Generator().manual_seed(seed + j)
        e = torch.randint(0, cols + 1, (rows,), generator=g, dtype=torch.int32)
        e[0] = cols
        x[1, ::3] = float("nan")
        xs.append(x.to(dtype))
        ends.append(e)
    return xs, ends


def _check_rows(xs, ends, outs, what):
    for (rows, cols, dtype, k, srt), x, e, o in zip(ROW_CASES, xs, ends, outs):
        want = np.full(tuple(o.shape), CANARY, dtype=np.int32)
        oracle.topk_rows(host_view(x), k, row_ends=e.numpy(), out=want, sorted=srt)
        assert_rows_equal(o.cpu().numpy(), want, f"{what} {rows}x{cols} {dtype} sorted={srt}")


def test_topk_rows_side_stream_and_graph():
    xs, ends = _row_inputs(500)
    xd = [x.to(DEV) for x in xs]
    ed = [e.to(DEV) for e in ends]
    outs = [torch.full((c[0], c[3] + 3), CANARY, dtype=torch.int32, device=DEV)
            for c in ROW_CASES]

    def step():
        for c, x, e, o in zip(ROW_CASES, xd, ed, outs):
            satk.topk_rows(x, c[3], row_ends=e, out=o, sorted=c[4])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    side.synchronize()
    _check_rows(xs, ends, outs, "side stream")

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for o in outs:
        o.fill_(CANARY)
    graph.replay()
    torch.cuda.synchronize()
    _check_rows(xs, ends, outs, "graph replay")

    xs2, ends2 = _row_inputs(900)  # new data in the captured buffers
    for x, e, x2, e2 in zip(xd, ed, xs2, ends2):
        x.copy_(x2)
        e.copy_(e2)
    for o in outs:
        o.fill_(CANARY)
    graph.replay()
    torch.cuda.synchronize()
    _check_rows(xs2, ends2, outs, "graph replay on new data")


def test_decode_step_in_one_graph():
    W, T, S, n, k = 4, 16, 20000, 128, 512
    slots = (k - 1) // n
    lg_a, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=300, seed=61)
    lg_b, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=300, seed=62)
    g = lg_a.to(DEV)
    local = torch.empty((W * T, n), dtype=torch.int32, device=DEV)
    packed = torch.empty((W, T, n + n // 32), dtype=torch.int32, device=DEV)
    sat = torch.empty(T, dtype=torch.int32, device=DEV)
    status = torch.empty(1, dtype=torch.int32, device=DEV)
    ids1 = torch.empty((T, k), dtype=torch.int32, device=DEV)
    ids2 = torch.empty((T, k), dtype=torch.int32, device=DEV)
    recv = torch.empty(T * slots * (k + k // 32), dtype=torch.int32, device=DEV)
    B = 64
    width = (S + B - 1) // B
    rng = np.random.default_rng(8)
    table = torch.from_numpy(rng.permutation(T * width).astype(np.int32).reshape(T, width))
    req = torch.from_numpy(rng.permutation(T).astype(np.int32))
    table_d, req_d = table.to(DEV), req.to(DEV)
    rows_out = torch.empty((T, k), dtype=torch.int32, device=DEV)
    valid = torch.empty(T, dtype=torch.int32, device=DEV)
    emit_status = torch.empty(1, dtype=torch.int32, device=DEV)
    rank = 1

    def step():
        status.zero_()
        emit_status.zero_()
        recv.fill_(123)
        satk.topk_rows(g.view(W * T, S), n, out=local)
        satk.dcp_pack(g.view(W * T, S), local, out=packed.view(W * T, -1))
        satk.dcp_merge_select(packed, k, packed=True, ids_out=ids1, sat_word=sat, status=status)
        ids2.copy_(ids1)
        satk.dcp_rescue_select(packed, g, sat, ids2, k, recv=recv, status=status)
        satk.dcp_emit_rows(ids2, W, rank, req_d, table_d, B, B, rows_out=rows_out,
                           valid_out=valid, status=emit_status)

    step()  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for lg, what in ((lg_a, "graph decode"), (lg_b, "graph decode on new data")):
        g.copy_(lg.to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        got = dict(local=local.cpu().numpy(), packed=packed.cpu().numpy(),
                   ids1=ids1.cpu().numpy(), sat=sat.cpu().numpy(), ids2=ids2.cpu().numpy(),
                   recv=recv.cpu().numpy().reshape(T, slots, k + k // 32),
                   status=int(status.item()))
        want = _decode_oracle(lg, n, k)
        _compare_decode(got, want, what)
        want_rows, want_valid, st = oracle.emit_rows(want["ids2"], W, rank, req.numpy(),
                                                     table.numpy(), B, B)
        assert_rows_equal(rows_out.cpu().numpy(), want_rows, f"{what}: emit_rows")
        assert np.array_equal(valid.cpu().numpy(), want_valid)
        assert int(emit_status.item()) == st
    assert bits_of(lg_a).tobytes() != bits_of(lg_b).tobytes()
