"""Randomised pins of the oracle (hypothesis, CPU): rows of up to 160
columns, any row end and any K, against a counting formulation that shares
nothing with the oracle's sort -- a column is chosen exactly when fewer than
K valid columns precede it under (score desc, column asc).  The same for the score-sorted layout and for the pairs merge
(a candidate is chosen when fewer than K non-empty candidates precede it
under (score desc, gid asc))."""
from __future__ import annotations

import math

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
from checks import bf16_bits_to_f32, order_key  # noqa: E402

SPECIALS = [math.nan, -math.inf, math.inf, -0.0, 0.0]


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _values(draw, n):
    """Scores with many ties (small integers), special values and reals."""
    reals = st.floats(-1e30, 1e30, allow_nan=False).map(lambda v: float(np.float32(v)))
    pool = st.one_of(st.sampled_from(SPECIALS), st.integers(-3, 3).map(float), reals)
    return [draw(pool) for _ in range(n)]


def _chosen(vals, end, k):
    """Columns preceded by fewer than k valid columns, counted pairwise."""
    valid = [c for c in range(end) if not math.isnan(vals[c])]
    keys = {c: order_key(vals[c]) for c in valid}
    out = []
    for a in valid:
        ahead = sum(1 for b in valid if keys[b] > keys[a] or (keys[b] == keys[a] and b < a))
        if ahead < k:
            out.append(a)
    return out, keys, valid


def _layout(vals, end, k):
    chosen, keys, valid = _chosen(vals, end, k)
    if len(valid) < k:
        return sorted(chosen) + [-1] * (k - len(valid))
    kth = min(keys[c] for c in chosen)
    return (sorted(c for c in chosen if keys[c] > kth) +
            sorted(c for c in chosen if keys[c] == kth))


def _sorted_layout(vals, end, k):
    chosen, keys, _ = _chosen(vals, end, k)
    order = sorted(chosen, key=lambda c: (tuple(-v for v in keys[c]), c))
    return order + [-1] * (k - len(order))


@st.composite
def topk_case(draw):
    cols = draw(st.integers(1, 160))
    rows = draw(st.integers(1, 4))
    x = np.array([_values(draw, cols) for _ in range(rows)], dtype=np.float32)
    ends = np.array([draw(st.integers(-3, cols + 3)) for _ in range(rows)], dtype=np.int32)
    k = draw(st.integers(1, cols + 4))
    return x, ends, k


@settings(max_examples=150, deadline=None)
@given(topk_case())
def test_topk_rows_against_counting(case):
    x, ends, k = case
    got = oracle.topk_rows(x, k, row_ends=ends)
    srt = oracle.topk_rows(x, k, row_ends=ends, sorted=True)
    for i in range(len(x)):
        e = max(0, min(int(ends[i]), x.shape[1]))
        vals = x[i].tolist()
        assert got[i].tolist() == _layout(vals, e, k)
        assert srt[i].tolist() == _sorted_layout(vals, e, k)


@settings(max_examples=100, deadline=None)
@given(topk_case())
def test_topk_rows_bf16_against_counting(case):
    x, ends, k = case
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16 patterns
    got = oracle.topk_rows(bits, k, row_ends=ends)
    vals = bf16_bits_to_f32(bits)
    for i in range(len(x)):
        e = max(0, min(int(ends[i]), x.shape[1]))
        assert got[i].tolist() == _layout(vals[i].tolist(), e, k)


@st.composite
def pairs_case(draw):
    W = draw(st.integers(1, 4))
    T = draw(st.integers(1, 3))
    n = draw(st.integers(1, 12))
    k = draw(st.integers(1, W * n + 3))
    scores = np.array([[_values(draw, n) for _ in range(T)] for _ in range(W)],
                      dtype=np.float32)
    gid = np.empty((W, T, n), dtype=np.int64)
    for t in range(T):  # distinct gids per row, some negative (empty)
        ids = draw(st.lists(st.integers(-2, 200), min_size=W * n, max_size=W * n,
                            unique=True))
        gid[:, t, :] = np.array(ids).reshape(W, n)
    return scores, gid, k


@settings(max_examples=150, deadline=None)
@given(pairs_case())
def test_pairs_merge_against_counting(case):
    scores, gid, k = case
    W, T, n = scores.shape
    cand = np.empty((W, T, n, 2), dtype=np.int32)
    cand[..., 0] = scores.view(np.int32)
    cand[..., 1] = gid.astype(np.int32)
    got = oracle.merge_pairs(cand, k)
    for t in range(T):
        ent = [(r * n + j, float(scores[r, t, j]), int(gid[r, t, j]))
               for r in range(W) for j in range(n)
               if gid[r, t, j] >= 0 and not math.isnan(scores[r, t, j])]
        chosen = []
        for f, s, g in ent:
            ks = order_key(s)
            ahead = sum(1 for _, s2, g2 in ent
                        if order_key(s2) > ks or (order_key(s2) == ks and g2 < g))
            if ahead < k:
                chosen.append((f, g))
        want = [g for _, g in sorted(chosen)] + [-1] * (k - len(chosen))
        assert got[t].tolist() == want


@st.composite
def decode_case(draw):
    W = draw(st.integers(2, 4))
    T = draw(st.integers(1, 3))
    S = draw(st.integers(40, 400))
    n = draw(st.sampled_from([32, 64]))
    k = n * draw(st.integers(2, 4))
    rng = np.random.default_rng(draw(st.integers(0, 2**31 - 1)))
    levels = draw(st.sampled_from([0, 3, 40]))  # 0: bf16 of N(0,1); else few levels
    if levels:
        table = (rng.standard_normal(levels).astype(np.float32).view(np.uint32) >> 16)
        bits = table[rng.integers(0, levels, size=(W, T, S))].astype(np.uint16)
    else:
        bits = (rng.standard_normal((W, T, S)).astype(np.float32).view(np.uint32)
                >> 16).astype(np.uint16)
    bits[rng.random((W, T, S)) < 0.02] = 0x7FC0                    # NaN
    bits[rng.random((W, T, S)) < 0.01] = 0xFF80                    # -inf
    for t in range(T):                                             # one skewed rank
        if rng.random() < 0.6:
            r = int(rng.integers(0, W))
            pos = rng.choice(S, size=min(S, int(rng.integers(n, 2 * n + 1))), replace=False)
            big = (3.0 + rng.random(len(pos))).astype(np.float32)
            bits[r, t, pos] = (big.view(np.uint32) >> 16).astype(np.uint16)
    ends = None
    if draw(st.booleans()):
        ends = rng.integers(0, S + 5, size=(W, T)).astype(np.int32)
    return bits, n, k, ends


@settings(max_examples=60, deadline=None)
@given(decode_case())
def test_decode_merge_exact_whenever_the_slots_suffice(case):
    """The packed merge and its rescue, step by step in the oracle, end
    with the top-k scores of the union of all ranks on every row.  A
    producer that sends distinct keys never saturates more ranks than there
    are rescue slots (N saturated words per rank all sit strictly above the
    K-th key, so at most (K-1)//N ranks), so no status bit is ever raised."""
    from checks import check_decode_merge_row
    bits, n, k, ends = case
    W, T, S = bits.shape
    flat = bits.reshape(W * T, S)
    fe = None if ends is None else ends.reshape(-1)
    local = oracle.topk_rows(flat, n, row_ends=fe)
    packed = oracle.dcp_pack(flat, local, row_ends=fe).reshape(W, T, n + n // 32)
    ids1, sat, st1 = oracle.merge_packed(packed, k)
    ids2, _, st2 = oracle.rescue(packed, k, bits, sat, ids1.copy(), row_ends=ends)
    assert (st1 | st2) == 0
    for t in range(T):
        check_decode_merge_row(ids2[t], bits, t, k, row_ends=ends)


@st.composite
def pack_case(draw):
    rows = draw(st.integers(1, 4))
    S = draw(st.sampled_from([50, 70000, 131072, 140000]))
    n = draw(st.sampled_from([32, 64, 96]))
    rng = np.random.default_rng(draw(st.integers(0, 2**31 - 1)))
    bits = rng.integers(0, 1 << 16, size=(rows, S), dtype=np.int64).astype(np.uint16)
    edges = np.array([-1, 0, 1, 65535, 65536, 65537, 131071, 131072, S - 1, S, S + 3])
    local = np.where(rng.random((rows, n)) < 0.3, rng.choice(edges, size=(rows, n)),
                     rng.integers(-2, S + 2, size=(rows, n))).astype(np.int32)
    ends = None
    if draw(st.booleans()):
        ends = rng.integers(-1, S + 3, size=rows).astype(np.int32)
    return bits, local, ends


@settings(max_examples=80, deadline=None)
@given(pack_case())
def test_pack_words_decode_back(case):
    """Each non-zero word gives back its slot's local id (low 16 bits
    complemented, bit 16 from the plane) and score bits (the inverse of the
    order-preserving ord16 map); zero words, with a clear plane bit, sit
    exactly on the slots that cannot be packed (local outside [0, min(end,
    S, 2**17)) or a NaN score)."""
    bits, local, ends = case
    rows, S = bits.shape
    n = local.shape[1]
    packed = oracle.dcp_pack(bits, local, row_ends=ends)
    assert packed.shape == (rows, n + n // 32)
    words = packed.view(np.uint32)
    for i in range(rows):
        lim = min(S, 1 << 17) if ends is None else min(max(int(ends[i]), 0), S, 1 << 17)
        for j in range(n):
            w = int(words[i, j])
            plane = (int(words[i, n + j // 32]) >> (j % 32)) & 1
            loc = int(local[i, j])
            ok = 0 <= loc < lim
            if ok:
                h = int(bits[i, loc])
                ok = not ((h & 0x7FFF) > 0x7F80)  # NaN
            if not ok:
                assert w == 0 and plane == 0, (i, j, loc)
                continue
            assert (0xFFFF - (w & 0xFFFF)) | (plane << 16) == loc
            o = w >> 16
            h_back = (o & 0x7FFF) if (o & 0x8000) else (~o & 0xFFFF)
            assert h_back == int(bits[i, loc]), (i, j, hex(o), hex(int(bits[i, loc])))
