"""Pins of the CPU oracle against facts fixed outside the oracle itself.

* brute force on tiny rows: every subset of the right size is tried and the
  one that dominates the rest under (score desc, column asc) must be the
  oracle's (a different mechanism from the oracle's full sort);
* the score-multiset property on realistic rows (numpy sort of reals);
* the hand-worked B' pack table (tests/golden/pack_example.txt);
* the closed form of the pairs merge: the top-K of the union of every rank's
  logits (the merge only sees each rank's top-K list);
* hand-worked saturation / rescue example;
* the decode-merge exactness invariant and the saturation rows of a skewed
  workload;
* the checkers bite: corrupted outputs fail them.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from checks import (bf16_bits_to_f32, check_decode_merge_row, check_topk_layout,
                    check_topk_row, order_key, packed_contract)
from sparse_attention_indexer_radix_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

ALPHABET = [math.nan, -math.inf, -1.0, -0.0, 0.0, 1.0, math.inf]


def brute_topk(vals, end, k):
    """All subsets of size min(k, n_valid): the answer is the one whose
    every member strictly precedes every non-member under (score desc,
    column asc).  Laid out as [> K-th, by column][== K-th, by column]; a
    short row is all valid columns by column."""
    valid = [c for c in range(end) if not math.isnan(vals[c])]

    def before(a, b):  # a strictly precedes b
        ka, kb = order_key(vals[a]), order_key(vals[b])
        return ka > kb or (ka == kb and a < b)

    m = min(k, len(valid))
    winners = []
    for sub in itertools.combinations(valid, m):
        s = set(sub)
        if all(before(a, b) for a in sub for b in valid if b not in s):
            winners.append(sub)
    assert len(winners) == 1
    chosen = list(winners[0])
    if len(valid) < k:
        return sorted(chosen) + [-1] * (k - len(valid))
    kth = min((order_key(vals[c]) for c in chosen))
    gt = sorted(c for c in chosen if order_key(vals[c]) > kth)
    eq = sorted(c for c in chosen if order_key(vals[c]) == kth)
    return gt + eq


def test_topk_exhaustive_tiny_alphabet():
    L = 4
    rows = np.array(list(itertools.product(ALPHABET, repeat=L)), dtype=np.float32)
    for k in range(1, L + 2):
        for end in range(0, L + 1):
            ends = np.full(len(rows), end, dtype=np.int32)
            got = oracle.topk_rows(rows, k, row_ends=ends)
            for i in range(len(rows)):
                want = brute_topk(rows[i].tolist(), end, k)
                assert got[i].tolist() == want, (rows[i], end, k, got[i], want)


def test_topk_random_small_rows_few_levels():
    rng = np.random.default_rng(7)
    levels = np.array([math.nan, -math.inf, -2.5, -1.0, -0.0, 0.0, 0.5, 1.0, 3.0,
                       math.inf], dtype=np.float32)
    for cols in (5, 8, 12):
        x = levels[rng.integers(0, len(levels), size=(300, cols))]
        ends = rng.integers(-2, cols + 3, size=300).astype(np.int32)
        for k in (1, 2, 3, cols // 2, cols, cols + 1):
            got = oracle.topk_rows(x, k, row_ends=ends)
            for i in range(len(x)):
                e = max(0, min(int(ends[i]), cols))
                assert got[i].tolist() == brute_topk(x[i].tolist(), e, k)


def test_topk_signed_zero_and_infinities():
    x = np.array([[-0.0, 0.0], [0.0, -0.0]], dtype=np.float32)
    assert oracle.topk_rows(x, 1).tolist() == [[1], [0]]
    assert oracle.topk_rows(x, 2).tolist() == [[1, 0], [0, 1]]
    y = np.array([[-math.inf, math.nan, math.inf, 5.0, -math.inf]], dtype=np.float32)
    assert oracle.topk_rows(y, 2).tolist() == [[2, 3]]
    assert oracle.topk_rows(y, 4).tolist() == [[2, 3, 0, 4]]
    assert oracle.topk_rows(y, 3).tolist() == [[2, 3, 0]]
    allnan = np.full((1, 9), math.nan, dtype=np.float32)
    assert oracle.topk_rows(allnan, 4).tolist() == [[-1, -1, -1, -1]]


def test_topk_prefill_smoke_shape_scores_and_layout():
    x, ends = inputs.prefill(rows=64, cols=4096, seed=1235)
    x, ends = x.numpy(), ends.numpy()
    out = np.full((64, 640), -7, dtype=np.int32)
    oracle.topk_rows(x, 512, row_ends=ends, out=out)
    for i in range(64):
        e = int(ends[i])
        check_topk_row(x[i], e, 512, out[i], ld_canary=-7, where=f"row {i}")
        check_topk_layout(x[i], e, 512, out[i], where=f"row {i}")
        # N(0,1) fp32 rows have no ties at the cut: the set is argsort's
        want = set(np.argsort(-x[i, :e], kind="stable")[:512].tolist())
        assert set(out[i, :512].tolist()) == want


def test_topk_bf16_agrees_with_widened_f32():
    x, ends, _ = inputs.adversarial(rows=12, cols=3000, seed=99)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    f = bf16_bits_to_f32(bits)
    e = ends.numpy()
    for k in (1, 17, 600, 2048):
        a = oracle.topk_rows(bits, k, row_ends=e)
        b = oracle.topk_rows(f, k, row_ends=e)
        assert np.array_equal(a, b)
        for i in range(12):
            end = max(0, min(int(e[i]), 3000))
            check_topk_row(f[i], end, k, a[i], where=f"k={k} row {i}")
            check_topk_layout(f[i], end, k, a[i], where=f"k={k} row {i}")


def test_topk_short_rows_tails_and_padding():
    x, _ = inputs.prefill(rows=8, cols=100, seed=5)
    x = x.numpy()
    ends = np.array([0, 1, 5, 31, 32, 33, 100, 1000], dtype=np.int32)
    out = np.full((8, 48), 12345, dtype=np.int32)
    oracle.topk_rows(x, 32, row_ends=ends, out=out)
    for i in range(8):
        e = max(0, min(int(ends[i]), 100))
        check_topk_row(x[i], e, 32, out[i], ld_canary=12345)
        n = min(32, e)
        assert np.all(out[i, n:32] == -1)


# ------------------------------------------------------------------ pack --

def _load_pack_golden():
    rows = []
    with open(os.path.join(GOLDEN, "pack_example.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            j, bits, local, whex, wint, plane, gid = line.split()
            rows.append(dict(j=int(j), bits=None if bits == "-" else int(bits, 16),
                             local=int(local), word=int(wint), plane=int(plane),
                             gid=None if gid == "-" else int(gid)))
    return rows


def _pack_golden_inputs():
    g = _load_pack_golden()
    S = (1 << 17) + 1
    logits = np.zeros((1, S), dtype=np.uint16)
    idx = np.full((1, 32), -1, dtype=np.int32)
    for e in g:
        idx[0, e["j"]] = e["local"]
        if e["bits"] is not None:
            logits[0, e["local"]] = e["bits"]
    return g, logits, idx, S


def test_pack_hand_worked_example():
    g, logits, idx, S = _pack_golden_inputs()
    packed = oracle.dcp_pack(logits, idx, row_ends=np.array([S], dtype=np.int32))
    want = np.zeros(33, dtype=np.int32)
    for e in g:
        want[e["j"]] = e["word"]
    want[32] = 0x22
    assert packed[0].tolist() == want.tolist()
    # decode through the merge: owner rank 3 of W = 8, others empty
    W, k = 8, 64
    gathered = np.zeros((W, 1, 33), dtype=np.int32)
    gathered[3, 0] = packed[0]
    ids, sat, status = oracle.merge_packed(gathered, k)
    chosen = [e["gid"] for e in g if e["gid"] is not None]
    assert ids[0, :len(chosen)].tolist() == chosen
    assert np.all(ids[0, len(chosen):] == -1)


def test_bf16_order_chain_through_pack():
    """-inf < -max < -1 < -0 < +0 < 1 < max < +inf, through the words."""
    chain = [0xFF80, 0xFF7F, 0xBF80, 0x8000, 0x0000, 0x3F80, 0x7F7F, 0x7F80]
    want_ord = [0x007F, 0x0080, 0x407F, 0x7FFF, 0x8000, 0xBF80, 0xFF7F, 0xFF80]
    logits = np.array([chain], dtype=np.uint16)
    idx = np.array([list(range(8)) + [-1] * 24], dtype=np.int32)
    w = oracle.dcp_pack(logits, idx)[0, :8].astype(np.int64) & 0xFFFFFFFF
    assert (w >> 16).tolist() == want_ord
    assert ((0xFFFF - (w & 0xFFFF))).tolist() == list(range(8))


def test_pack_contract_on_local_topn():
    lg, _, _ = inputs.decode_merge(W=2, rows=6, S=3000, n=64, k=256, skew_count=80, seed=3)
    bits = lg.view(torch.int16).numpy().view(np.uint16).reshape(12, 3000)
    ends = np.array([3000, 10, 64, 65, 2999, 0] * 2, dtype=np.int32)
    local = oracle.topk_rows(bits, 64, row_ends=ends)
    packed = oracle.dcp_pack(bits, local, row_ends=ends)
    packed_contract(packed, bits, ends, 64)


def test_pack_drops_out_of_range_and_nan():
    S = 100
    logits = np.full((1, S), 0x3F80, dtype=np.uint16)
    logits[0, 4] = 0x7FC1
    idx = np.array([[-5, 0, 4, 99, 100, 50, 2**17, 7] + [-1] * 24], dtype=np.int32)
    p = oracle.dcp_pack(logits, idx, row_ends=np.array([60], dtype=np.int32))
    nz = (p[0, :32] != 0).tolist()
    assert nz[:8] == [False, True, False, False, False, True, False, True]


# ----------------------------------------------------------------- merges --

def test_pairs_merge_equals_union_topk():
    W, R, k, local = 8, 24, 256, 2048
    cand, logits = inputs.pairs_merge(W=W, rows=R, k=k, local=local, seed=11, keep_logits=True)
    cand_np = cand.numpy()
    ids = oracle.merge_pairs(cand_np, k)
    lg = logits.numpy()
    for t in range(R):
        scores = lg[:, t, :].reshape(-1)           # [W * local], rank-major
        r = np.repeat(np.arange(W), local)
        loc = np.tile(np.arange(local), W)
        gid = loc * W + r
        order = np.lexsort((gid, -scores))
        want = set(gid[order[:k]].tolist())
        assert set(ids[t].tolist()) == want
        # flat-order layout: chosen positions ascend in the rank-major buffer
        flat_of = {}
        for rr in range(W):
            for j in range(k):
                flat_of[int(cand_np[rr, t, j, 1])] = rr * k + j
        pos = [flat_of[g] for g in ids[t].tolist()]
        assert pos == sorted(pos)


def test_pairs_merge_empty_entries_and_short():
    W, k, n = 2, 8, 4
    cand = np.zeros((W, 1, n, 2), dtype=np.int32)
    sc = np.array([[3.0, np.nan, 1.0, 2.0], [5.0, 0.5, -1.0, 7.0]], dtype=np.float32)
    gid = np.array([[0, 2, -1, 6], [1, 3, 5, 7]], dtype=np.int32)
    cand[:, 0, :, 0] = sc.view(np.int32)
    cand[:, 0, :, 1] = gid
    ids = oracle.merge_pairs(cand, k)
    # valid: (3,0) (2,6) (5,1) (0.5,3) (-1,5) (7,7); fewer than k -> all, flat order
    assert ids[0].tolist() == [0, 6, 1, 3, 5, 7, -1, -1]
    ids3 = oracle.merge_pairs(cand, 3)
    assert ids3[0].tolist() == [0, 1, 7]


def _hand_rescue_case():
    """W=2, n=32, K=64, S=64.  Rank 0 scores 200-l, rank 1 scores 100-l
    (exact in bf16).  Round 1 sees rank 0's top-32 and rank 1's top-32; the
    K-th is 69, rank 0 is saturated, the rescue must return rank 0's 64."""
    W, T, S, n, k = 2, 1, 64, 32, 64
    vals = np.zeros((W, T, S), dtype=np.float32)
    vals[0, 0] = 200.0 - np.arange(S)
    vals[1, 0] = 100.0 - np.arange(S)
    bits = (vals.view(np.uint32) >> 16).astype(np.uint16)
    return W, T, S, n, k, bits


def test_rescue_hand_worked_example():
    W, T, S, n, k, bits = _hand_rescue_case()
    local = oracle.topk_rows(bits.reshape(W * T, S), n)
    packed = oracle.dcp_pack(bits.reshape(W * T, S), local).reshape(W, T, n + n // 32)
    ids, sat, status = oracle.merge_packed(packed, k)
    assert status == 0
    # round 1: rank 0 locals 0..31 (gid 2l), rank 1 locals 0..31 (gid 2l+1)
    assert ids[0].tolist() == [2 * l for l in range(32)] + [2 * l + 1 for l in range(32)]
    assert sat[0] == (1 << 16) | 0xC28A  # mask 0b01, tau16 = ord16(bf16 69.0)
    ids2, recv, status = oracle.rescue(packed, k, bits, sat, ids.copy())
    assert status == 0
    assert ids2[0].tolist() == [2 * l for l in range(64)]
    words = recv[0, 0, :64].astype(np.int64) & 0xFFFFFFFF
    assert ((0xFFFF - (words & 0xFFFF))).tolist() == list(range(64))
    check_decode_merge_row(ids2[0], bits, 0, k)


def _decode_pipeline(W, T, S, n, k, skew_count, seed):
    lg, skewed, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=skew_count,
                                        seed=seed)
    bits = lg.view(torch.int16).numpy().view(np.uint16)
    flat = bits.reshape(W * T, S)
    local = oracle.topk_rows(flat, n)
    packed = oracle.dcp_pack(flat, local).reshape(W, T, n + n // 32)
    ids1, sat, status = oracle.merge_packed(packed, k)
    ids2, recv, status2 = oracle.rescue(packed, k, bits, sat, ids1.copy())
    return bits, skewed.numpy(), packed, ids1, sat, ids2, recv, status | status2


def test_decode_merge_exact_and_saturation_rows():
    W, T, S, n, k = 8, 16, 4096, 96, 512
    bits, skewed, packed, ids1, sat, ids2, recv, status = _decode_pipeline(
        W, T, S, n, k, skew_count=150, seed=21)
    assert status == 0
    mask = (sat.astype(np.int64) & 0xFFFFFFFF) >> 16
    assert np.array_equal(mask != 0, skewed), (mask, skewed)
    for t in range(T):
        check_decode_merge_row(ids2[t], bits, t, k, where="rescued")
    bitten = 0
    for t in np.nonzero(skewed)[0]:
        try:
            check_decode_merge_row(ids1[t], bits, t, k)
        except AssertionError:
            bitten += 1
    assert bitten >= 1, "round 1 alone should miss tokens on a skewed row"
    for t in np.nonzero(~skewed)[0]:
        assert np.array_equal(ids1[t], ids2[t])


def test_decode_merge_deterministic():
    a = _decode_pipeline(4, 6, 2048, 64, 256, skew_count=80, seed=5)
    b = _decode_pipeline(4, 6, 2048, 64, 256, skew_count=80, seed=5)
    for x, y in zip(a[2:7], b[2:7]):
        assert np.array_equal(x, y)


def test_packed_merge_duplicate_words_out_of_contract():
    """A producer that repeats a word (a NaN row's arbitrary ids, on the
    page) is outside the contract: the select keeps fewer than K rather than
    reading past, reports it, and tau16 falls to 0."""
    W, n, k = 1, 32, 4
    packed = np.zeros((W, 1, 33), dtype=np.int32)
    w = (0xBF80 << 16) | (0xFFFF - 3)
    packed[0, 0, :6] = np.array([w, w, w, w, w, w], dtype=np.uint32).view(np.int32)
    ids, sat, status = oracle.merge_packed(packed, k)
    assert status & 2
    assert ids[0].tolist() == [-1, -1, -1, -1]
    assert (int(sat[0]) & 0xFFFF) == 0


# ------------------------------------------------------- checkers bite --

def test_checkers_reject_corrupted_outputs():
    x, ends = inputs.prefill(rows=4, cols=600, seed=8)
    x, ends = x.numpy(), ends.numpy()
    out = oracle.topk_rows(x, 64, row_ends=ends)
    e = int(ends[0])
    bad = out[0].copy()
    # swap a chosen id for an unchosen lower-scoring column
    unchosen = [c for c in np.argsort(x[0, :e]) if c not in set(bad.tolist())]
    bad[5] = unchosen[0]
    with pytest.raises(AssertionError):
        check_topk_row(x[0], e, 64, bad)
    bad = out[0].copy()
    bad[[3, 4]] = bad[[4, 3]]
    with pytest.raises(AssertionError):
        check_topk_layout(x[0], e, 64, bad)
    bad = out[0].copy()
    bad[10] = bad[11]
    with pytest.raises(AssertionError):
        check_topk_row(x[0], e, 64, bad)


def test_contract_checker_bites():
    lg, _, _ = inputs.decode_merge(W=1, rows=2, S=500, n=32, k=64, skew_count=10, seed=4)
    bits = lg.view(torch.int16).numpy().view(np.uint16).reshape(2, 500)
    local = oracle.topk_rows(bits, 32)
    worst = np.argsort(bf16_bits_to_f32(bits[0]))[0]
    local[0, 0] = worst  # a sent token below an unsent one
    packed = oracle.dcp_pack(bits, local)
    with pytest.raises(AssertionError):
        packed_contract(packed, bits, None, 32)


# ------------------------------------------------------------- emit_rows --

def _emit_rows_golden():
    path = os.path.join(os.path.dirname(__file__), "golden", "emit_rows_example.txt")
    g = {"table": [], "ids": [], "rows": []}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        vals = [int(v) for v in vals]
        if key in g:
            g[key].append(vals)
        else:
            g[key] = vals if len(vals) > 1 else vals[0]
    return g


def test_emit_rows_hand_worked_example():
    g = _emit_rows_golden()
    rows, valid, status = oracle.emit_rows(
        np.array(g["ids"], dtype=np.int32), g["W"], g["rank"],
        np.array(g["req"], dtype=np.int32), np.array(g["table"], dtype=np.int32),
        g["block_size"], g["stride_rows"], ld_rows=10)
    assert rows[:, :8].tolist() == g["rows"]
    assert np.all(rows[:, 8:] == -7)  # columns past k never written
    assert valid.tolist() == g["valid"]
    assert status == g["status"]


def test_emit_rows_identity_table_gives_local_ids():
    """block_table[r][b] = b and stride_rows = B make every physical row the
    token's own local index gid // W: the owned subsequence, in order."""
    rng = np.random.default_rng(11)
    W, B, k, T = 8, 64, 256, 12
    width = 40
    ids = rng.integers(-1, W * B * width + 3 * W * B, size=(T, k)).astype(np.int32)
    table = np.tile(np.arange(width, dtype=np.int32), (3, 1))
    req = rng.integers(0, 3, size=T).astype(np.int32)
    for rank in range(W):
        rows, valid, status = oracle.emit_rows(ids, W, rank, req, table, B, B)
        assert status == 0
        for t in range(T):
            want = [g // W for g in ids[t].tolist()
                    if g >= 0 and g % W == rank and g // W // B < width]
            assert valid[t] == len(want)
            assert rows[t, :len(want)].tolist() == want
            assert np.all(rows[t, len(want):] == -1)


def test_emit_rows_ranks_partition_the_selection():
    """Over all ranks every selected id in the table's range is emitted
    exactly once, and dropped blocks by none."""
    lg, _, _ = inputs.decode_merge(W=4, rows=6, S=3000, n=64, k=256, skew_count=0, seed=9)
    bits = lg.view(torch.int16).numpy().view(np.uint16).reshape(24, 3000)
    packed = oracle.dcp_pack(bits, oracle.topk_rows(bits, 64)).reshape(4, 6, 66)
    ids, _, _ = oracle.merge_packed(packed, 256)
    W, B, width = 4, 16, 40  # local < 3000 -> blocks up to 187; half dropped
    table = (np.arange(6 * width, dtype=np.int32).reshape(6, width) * 3 + 1)
    req = np.arange(6, dtype=np.int32)[::-1].copy()
    total = np.zeros(6, dtype=np.int64)
    for rank in range(W):
        rows, valid, _ = oracle.emit_rows(ids, W, rank, req, table, B, 2 * B)
        total += valid
        for t in range(6):
            got = rows[t, :valid[t]]
            assert len(set(got.tolist())) == len(got)  # distinct tokens, distinct rows
    in_range = ((ids >= 0) & ((ids // W) // B < width)).sum(axis=1)
    assert total.tolist() == in_range.tolist()
    assert 0 < in_range.sum() < (ids >= 0).sum()


def test_emit_rows_max_blocks_and_bad_requests():
    ids = np.array([[1, 5, 9, 13, 17]], dtype=np.int32)  # rank 1 of W=4: locals 0..4
    table = np.array([[10, 20, 30]], dtype=np.int32)
    rows, valid, status = oracle.emit_rows(ids, 4, 1, np.array([0], np.int32), table, 2, 100,
                                           max_blocks=2)
    assert rows[0].tolist() == [1000, 1001, 2000, 2001, -1] and valid[0] == 4 and status == 0
    rows, valid, status = oracle.emit_rows(ids, 4, 1, np.array([-1], np.int32), table, 2, 100)
    assert rows[0].tolist() == [-1] * 5 and valid[0] == 0 and status == 4


# ------------------------------------------------------- sorted top-K --

def test_topk_sorted_exhaustive_tiny_alphabet():
    """Score-sorted output: brute force over every row of 4 values from
    {NaN, -inf, -1, -0, +0, 1, +inf} (with repeats) against Python's sorted()
    on (-ordered key, column), for every K and row end."""
    alphabet = [float("nan"), float("-inf"), -1.0, -0.0, 0.0, 1.0, float("inf")]

    def okey(v):  # -0.0 below +0.0
        return (v, math.copysign(1.0, v))
    for vals in itertools.product(alphabet, repeat=4):
        x = np.array([vals], dtype=np.float32)
        for end in range(5):
            for k in (1, 2, 3, 4, 5):
                got = oracle.topk_rows(x, k, row_ends=np.array([end], np.int32), sorted=True)[0]
                valid = [c for c in range(end) if not math.isnan(vals[c])]
                order = sorted(valid, key=lambda c: (tuple(-t for t in okey(vals[c])), c))
                want = order[:k] + [-1] * (k - min(k, len(order)))
                assert got.tolist() == want, (vals, end, k, got.tolist(), want)


def test_topk_sorted_is_the_unsorted_set():
    x, ends = inputs.prefill(rows=12, cols=3000, seed=5)
    x, ends = x.numpy(), ends.numpy()
    x[3, ::7] = x[3, 1]  # ties
    for k in (1, 64, 512, 4000):
        a = oracle.topk_rows(x, k, row_ends=ends)
        b = oracle.topk_rows(x, k, row_ends=ends, sorted=True)
        for i in range(12):
            assert sorted(a[i].tolist()) == sorted(b[i].tolist())
            ids = b[i][b[i] >= 0]
            s = x[i, ids]
            assert np.all(s[:-1] >= s[1:])  # non-increasing scores


# ------------------------------------------- hand-worked decode examples --

def _load_golden_cases(name):
    """Header keys (`key v ...`), `word r j hex` input words and `case K`
    blocks (ids / sat / status) of a hand-worked merge example."""
    head, words, cases = {}, [], []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        vals = [int(v, 0) for v in vals]
        if key == "word":
            words.append(vals)
        elif key == "case":
            cases.append({"K": vals[0]})
        elif cases:
            cases[-1][key] = vals if key == "ids" else vals[0]
        else:
            head[key] = vals if len(vals) > 1 else vals[0]
    return head, words, cases


def golden_packed_buffer(name):
    """The [W, 1, N + N/32] B' buffer of a hand-worked example, and its cases."""
    head, words, cases = _load_golden_cases(name)
    W, n = head["W"], head["N"]
    p = np.zeros((W, 1, n + n // 32), dtype=np.uint32)
    for r, j, w in words:
        p[r, 0, j] = w
    return p.view(np.int32), cases


def _u32(v):
    return int(v) & 0xFFFFFFFF


@pytest.mark.parametrize("name", ["decode_zero_score_example.txt",
                                  "slots_exceeded_example.txt"])
def test_packed_merge_hand_worked_examples(name):
    """Words with a zero score field are candidates below every other score
    (the page's _decode_key); a mask with more saturated ranks than slots,
    which only repeated keys produce, is cleared with status bit 1."""
    packed, cases = golden_packed_buffer(name)
    for c in cases:
        ids, sat, status = oracle.merge_packed(packed, c["K"])
        assert ids[0].tolist() == c["ids"], (name, c["K"])
        assert _u32(sat[0]) == c["sat"], (name, c["K"], hex(_u32(sat[0])))
        assert status == c["status"], (name, c["K"], status)


def load_rescue_plane_golden():
    """Inputs and expected outputs of tests/golden/rescue_plane_example.txt:
    logits bits [W, T, S] and a dict of the expected arrays."""
    g = {}
    cols = {}
    for line in open(os.path.join(GOLDEN, "rescue_plane_example.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        vals = [int(v, 0) for v in vals]
        if key == "cols":
            cols[vals[0]] = (vals[1], vals[2:])
        elif key in ("local", "packed"):
            g.setdefault(key, {})[vals[0]] = vals[1:]
        else:
            g[key] = vals if len(vals) > 1 else vals[0]
    W, T, S = g["W"], g["T"], g["S"]
    bits = np.full((W, T, S), g["nan_bits"], dtype=np.uint16)
    for r, (val, cs) in cols.items():
        bits[r, 0, cs] = val
    return bits, g


def test_rescue_plane_hand_worked_example():
    """Pushed local ids at and above 2**16 set their plane bits, a column at
    2**17 is not pushed, and the re-select decodes the plane bits back into
    distinct global ids (hand-worked table)."""
    bits, g = load_rescue_plane_golden()
    W, T, S, n, k = g["W"], g["T"], g["S"], g["N"], g["K"]
    flat = bits.reshape(W * T, S)
    local = oracle.topk_rows(flat, n)
    for r in range(W):
        assert local[r].tolist() == g["local"][r]
    packed = oracle.dcp_pack(flat, local).reshape(W, T, n + n // 32)
    for r in range(W):
        assert [_u32(v) for v in packed[r, 0]] == g["packed"][r]
    ids1, sat, st1 = oracle.merge_packed(packed, k)
    assert ids1[0].tolist() == g["ids1"]
    assert _u32(sat[0]) == g["sat"] and st1 == 0
    ids2, recv, st2 = oracle.rescue(packed, k, bits, sat, ids1.copy())
    assert [_u32(v) for v in recv[0, 0]] == g["recv"]
    assert ids2[0].tolist() == g["ids2"]
    assert st2 == g["status"]
    assert len(set(g["ids2"])) == k  # the plane keeps the gids distinct
