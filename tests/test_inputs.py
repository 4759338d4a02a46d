"""The seeded input generators against the recipes they state: shapes,
causal row ends, the distribution ablation, each rank's list being its own
top-k, the skewed decode rows, the adversarial mix, and determinism."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from sparse_attention_indexer_radix_gb300 import inputs


def test_bf16_bit_patterns_round_trip():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32)
    x = inputs.bits_to_bf16(bits)
    back = x.view(torch.int16).to(torch.int32) & 0xFFFF
    assert x.dtype == torch.bfloat16 and torch.equal(back, bits)


@pytest.mark.parametrize("rows,cols", [(64, 4096), (16, 10)])
def test_prefill_shape_causal_ends_and_seed(rows, cols):
    x, ends = inputs.prefill(rows=rows, cols=cols, seed=5)
    assert x.shape == (rows, cols) and x.dtype == torch.float32 and ends.dtype == torch.int32
    want = np.clip(np.arange(rows) + cols - rows + 1, 0, None)
    assert np.array_equal(ends.numpy(), want)          # more rows than columns: leading 0s
    x2, _ = inputs.prefill(rows=rows, cols=cols, seed=5)
    x3, _ = inputs.prefill(rows=rows, cols=cols, seed=6)
    assert torch.equal(x, x2) and not torch.equal(x, x3)
    _, full = inputs.prefill(rows=rows, cols=cols, seed=5, causal=False)
    assert bool((full == cols).all())
    xb, _ = inputs.prefill(rows=rows, cols=cols, seed=5, dtype=torch.bfloat16)
    assert torch.equal(xb, x.to(torch.bfloat16))


def test_prefill_is_standard_normal():
    x, _ = inputs.prefill(rows=256, cols=4096, seed=9)
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01


def test_prefill_shifted_ablation():
    base, ends = inputs.prefill(32, 512, seed=1240)
    plus, e1 = inputs.prefill_shifted(32, 512, "plus100")
    tiny, _ = inputs.prefill_shifted(32, 512, "times1e-8")
    same, _ = inputs.prefill_shifted(32, 512, "normal")
    assert torch.equal(plus, base + 100.0) and torch.equal(tiny, base * 1e-8)
    assert torch.equal(same, base) and torch.equal(e1, ends)
    with pytest.raises(ValueError):
        inputs.prefill_shifted(4, 8, "other")


def test_pairs_lists_are_each_ranks_top_k():
    W, R, k, local = 4, 6, 32, 300
    cand, logits = inputs.pairs_merge(W=W, rows=R, k=k, local=local, seed=3, keep_logits=True,
                                      chunk_rows=4)
    assert cand.shape == (W, R, k, 2) and cand.dtype == torch.int32
    scores = cand[..., 0].contiguous().view(torch.float32).numpy()
    gids = cand[..., 1].numpy()
    lg = logits.numpy()
    for r in range(W):
        for t in range(R):
            assert np.all(gids[r, t] % W == r)
            loc = gids[r, t] // W
            order = np.lexsort((np.arange(local), -lg[r, t]))[:k]  # score desc, id asc
            assert set(loc.tolist()) == set(order.tolist())
            assert np.array_equal(scores[r, t], lg[r, t][loc])
    again = inputs.pairs_merge(W=W, rows=R, k=k, local=local, seed=3, chunk_rows=4)
    assert torch.equal(again, cand)


def test_decode_merge_skewed_rows_overflow_one_rank():
    W, T, S, n, k = 4, 8, 4096, 192, 512  # n well above k / W = 128
    lg, skewed, skew_rank = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=200,
                                                seed=11)
    assert lg.shape == (W, T, S) and lg.dtype == torch.bfloat16
    assert int(skewed.sum()) == round(T * 0.25)
    assert torch.equal(skewed, skew_rank >= 0) and int(skew_rank.max()) < W
    x = lg.float().numpy()
    for t in range(T):
        union = x[:, t].reshape(-1)
        top = np.argsort(-union, kind="stable")[:k]
        per_rank = np.bincount(top // S, minlength=W)
        if bool(skewed[t]):
            assert per_rank[int(skew_rank[t])] > n   # the rank alone overflows its n slots
        else:
            assert per_rank.max() <= n


def test_adversarial_mix():
    rows, cols = 24, 20000
    x, ends, nan_row = inputs.adversarial(rows=rows, cols=cols, seed=7)
    bits = x.view(torch.int16).to(torch.int32).numpy() & 0xFFFF
    assert x.dtype == torch.bfloat16 and ends.dtype == torch.int32
    is_nan = ((bits & 0x7FFF) > 0x7F80)
    assert not is_nan[np.arange(rows) != nan_row].any()
    assert 0.4 < is_nan[nan_row].mean() < 0.6
    rest = bits[np.arange(rows) != nan_row]
    assert abs((rest == 0xFF80).mean() - 0.01) < 0.002          # -inf
    assert abs((rest == 0x7F80).mean() - 0.001) < 0.0005        # +inf
    finite = set(np.unique(rest[(rest != 0xFF80) & (rest != 0x7F80)]).tolist())
    assert len(finite) == 64 and {0x0000, 0x8000} <= finite     # 64 levels, both zeros
    assert ends[1:6].tolist() == [0, 1, 2047, 2048, 2049]
    assert int(ends.min()) >= 0 and int(ends.max()) <= cols
