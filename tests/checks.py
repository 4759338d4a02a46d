"""Property checks shared by the oracle pins and the GPU parity tests.

These restate what the pages fix about a correct answer -- not how the
oracle computes it -- so that they can catch a mistake in either side:

* the chosen scores of a row, as a multiset of reals, are the K largest
  non-NaN scores of the row ([Perf][DSA] Use DeepSelect for eligible
  sparse-indexer prefill chunks, Test Plan and Test Result: selected-score
  equality, valid/unique indices, short-row tails);
* ids are unique, in range, never NaN, with -1 tails and untouched padding
  (same page, Test Plan);
* the packed producer contract (vLLM API page
  vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels,
  assert_packed_merge_contract), restated from its description;
* the exactness of the decode merge: the selected scores equal, as a
  multiset, the top-K of the union of all ranks' bf16 logits (same page,
  module docstring).
"""
from __future__ import annotations

import math

import numpy as np


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 patterns -> float32 values (bf16 is the top half of a
    binary32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def row_end(ends, i, cols):
    if ends is None:
        return cols
    return max(0, min(int(ends[i]), cols))


def check_topk_row(vals: np.ndarray, end: int, k: int, out_row: np.ndarray,
                   ld_canary=None, where: str = ""):
    """vals: float32 scores of one row (all columns); out_row: the full
    output row (length ld_out).  Raises AssertionError on a violation."""
    v = vals[:end]
    valid = ~np.isnan(v)
    n_valid = int(valid.sum())
    n_sel = min(k, n_valid)
    ids = out_row[:k]
    assert np.all(ids[n_sel:] == -1), f"{where}: -1 tail must start at {n_sel}"
    sel = ids[:n_sel]
    assert np.all((sel >= 0) & (sel < end)), f"{where}: id out of [0, {end})"
    assert len(np.unique(sel)) == n_sel, f"{where}: repeated id"
    assert not np.any(np.isnan(v[sel])), f"{where}: NaN chosen"
    want = np.sort(v[valid])[::-1][:n_sel]
    got = np.sort(v[sel])[::-1]
    assert np.array_equal(want, got), f"{where}: chosen scores are not the top-{k}"
    if ld_canary is not None and len(out_row) > k:
        assert np.all(out_row[k:] == ld_canary), f"{where}: padding past K written"


def check_topk_layout(vals: np.ndarray, end: int, k: int, out_row: np.ndarray,
                      where: str = ""):
    """The documented layout: strictly-above-the-K-th ids in ascending column
    order, then the ids tied with the K-th in ascending column order (and
    those are the lowest columns of the tie); a short row lists all its
    valid columns in ascending order."""
    v = vals[:end]
    valid_cols = np.nonzero(~np.isnan(v))[0]
    if len(valid_cols) < k:
        assert np.array_equal(out_row[:len(valid_cols)], valid_cols), f"{where}: short row order"
        return
    ids = out_row[:k]
    s = v[ids]
    kth = total_order_min(s)
    above = np.array([rank_gt(x, kth) for x in s])
    n_gt = int(above.sum())
    assert np.all(above[:n_gt]) and not np.any(above[n_gt:]), f"{where}: [>v][==v] split"
    assert np.all(np.diff(ids[:n_gt]) > 0), f"{where}: >v part not ascending"
    assert np.all(np.diff(ids[n_gt:]) > 0), f"{where}: ==v part not ascending"
    tied = [c for c in valid_cols if same_rank(v[c], kth)]
    assert list(ids[n_gt:]) == tied[:k - n_gt], f"{where}: tie not broken toward low columns"


def order_key(x: float):
    """The total order on non-NaN scores used by every path: real order,
    and -0.0 just below +0.0."""
    return (float(x), math.copysign(1.0, float(x)))


def rank_gt(a, b) -> bool:
    return order_key(a) > order_key(b)


def same_rank(a, b) -> bool:
    return order_key(a) == order_key(b)


def total_order_min(vals):
    return min(vals, key=order_key)


def packed_contract(packed: np.ndarray, logits_bits: np.ndarray, row_ends, n: int,
                    where: str = ""):
    """Producer contract of a packed merge input, restated from the page's
    description of assert_packed_merge_contract: per row exactly min(N, v)
    non-empty words (v = non-NaN tokens below the row end), distinct local
    ids below the row end, no NaN sent, each word's score the logit's bits,
    and no unsent non-NaN token scoring above the lowest sent one."""
    rows, S = logits_bits.shape
    words = packed[:, :n].astype(np.int64) & 0xFFFFFFFF
    plane = packed[:, n:].astype(np.int64) & 0xFFFFFFFF
    j = np.arange(n)
    local = (0xFFFF - (words & 0xFFFF)) | (((plane[:, j // 32] >> (j % 32)) & 1) << 16)
    vals = bf16_bits_to_f32(logits_bits)
    for t in range(rows):
        end = row_end(row_ends, t, S)
        sent = words[t] != 0
        ids = local[t][sent]
        valid = ~np.isnan(vals[t, :end])
        nv = int(valid.sum())
        assert len(ids) == min(n, nv), f"{where} row {t}: {len(ids)} words, want {min(n, nv)}"
        if len(ids) == 0:
            continue
        assert ids.max() < end, f"{where} row {t}: local id past row end"
        assert len(np.unique(ids)) == len(ids), f"{where} row {t}: repeated ids"
        assert not np.any(np.isnan(vals[t, ids])), f"{where} row {t}: NaN sent"
        # a word's score field holds the logit's bf16 bits under the pack's
        # order-preserving map; compare through the value it orders
        sent_scores = vals[t, ids]
        unsent = valid.copy()
        unsent[ids] = False
        if unsent.any():
            assert vals[t, :end][unsent].max() <= sent_scores.min(), \
                f"{where} row {t}: not a top-{n} by score"


def union_topk_scores(logits_bits: np.ndarray, t: int, k: int, row_ends=None):
    """Top-k bf16 scores (as float32, descending) of row t over all ranks'
    logits [W, T, S], NaN dropped."""
    W, T, S = logits_bits.shape
    vals = []
    for r in range(W):
        end = S if row_ends is None else max(0, min(int(row_ends[r, t]), S))
        v = bf16_bits_to_f32(logits_bits[r, t, :end])
        vals.append(v[~np.isnan(v)])
    allv = np.concatenate(vals)
    return np.sort(allv)[::-1][:k]


def check_decode_merge_row(ids_row: np.ndarray, logits_bits: np.ndarray, t: int, k: int,
                           row_ends=None, where: str = ""):
    """Exactness of the decode merge for row t: the chosen global ids are
    unique, in range, and their scores are the top-k of the union."""
    W, T, S = logits_bits.shape
    want = union_topk_scores(logits_bits, t, k, row_ends)
    n_sel = len(want)
    assert np.all(ids_row[n_sel:k] == -1), f"{where} row {t}: -1 tail"
    sel = ids_row[:n_sel].astype(np.int64)
    assert np.all((sel >= 0) & (sel < W * S)), f"{where} row {t}: gid out of range"
    assert len(np.unique(sel)) == n_sel, f"{where} row {t}: repeated gid"
    r, local = sel % W, sel // W
    got = np.sort(bf16_bits_to_f32(logits_bits[r, t, local]))[::-1]
    assert np.array_equal(got, want), f"{where} row {t}: scores differ from the union's top-{k}"
