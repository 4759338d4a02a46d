"""CUDA path against the CPU oracle, element by element, through the C ABI.

Integer outputs (ids, packed words, saturation words, rescue lists, status
bits) must match bit for bit.  Cases span several tiles and ragged tails of
both row paths (register-resident and streaming), fp32 and bf16, aligned and
unaligned rows, the edge cases of the pages' test plans (empty and short
rows, rows around K, full rows, strided output with untouched padding, -1
tails, NaN rows, infinities, signed zeros, massive ties), and the workloads
at their full sizes (every row)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_radix_gb300 as satk
from checks import check_decode_merge_row, check_topk_layout, check_topk_row, packed_contract
from guards import guarded
from sparse_attention_indexer_radix_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
CANARY = -7


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_indexer_radix_gb300 import build as satk_build
    satk_build.build()
    oracle.build()


def bits_of(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 numpy bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_view(x: torch.Tensor) -> np.ndarray:
    return bits_of(x) if x.dtype == torch.bfloat16 else x.cpu().numpy()


def run_topk(x: torch.Tensor, k: int, ends: torch.Tensor | None, ld_out: int, ld_x=None,
             sorted=False):
    """GPU and oracle outputs for x ([rows, cols], CPU tensor)."""
    rows, cols = x.shape
    if ld_x is not None and ld_x != cols:
        buf = torch.zeros((rows, ld_x), dtype=x.dtype, device=DEV)
        buf[:, :cols] = x.to(DEV)
        xg = buf[:, :cols]
    else:
        xg = x.to(DEV)
    out, guard = guarded((rows, ld_out), fill=CANARY)
    satk.topk_rows(xg, k, row_ends=None if ends is None else ends.to(DEV), out=out, sorted=sorted)
    guard("topk_rows out")
    want = np.full((rows, ld_out), CANARY, dtype=np.int32)
    oracle.topk_rows(host_view(x), k, row_ends=None if ends is None else ends.numpy(), out=want,
                     sorted=sorted)
    return out.cpu().numpy(), want


def assert_rows_equal(got, want, what=""):
    if not np.array_equal(got, want):
        bad = np.nonzero((got != want).any(axis=1))[0]
        r = int(bad[0])
        c = np.nonzero(got[r] != want[r])[0][:8]
        raise AssertionError(f"{what}: {len(bad)} rows differ; row {r} cols {c.tolist()} "
                             f"got {got[r, c].tolist()} want {want[r, c].tolist()}")


# ------------------------------------------------------------- topk_rows --

def test_prefill_smoke_workload():
    x, ends = inputs.prefill(rows=64, cols=4096, seed=1235)
    got, want = run_topk(x, 512, ends, 640)
    assert_rows_equal(got, want, "64x4096 fp32 K=512")
    for i in range(64):
        check_topk_row(x[i].numpy(), int(ends[i]), 512, got[i], ld_canary=CANARY)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cols", [37, 1000, 2048, 2049, 4100, 8191, 8192, 9000, 16390, 22528,
                                  24576, 40000])
def test_topk_shapes_both_paths(dtype, cols):
    rows = 24
    x, _ = inputs.prefill(rows=rows, cols=cols, seed=cols, dtype=dtype)
    g = torch.Generator().manual_seed(cols)
    ends = torch.randint(-3, cols + 5, (rows,), generator=g, dtype=torch.int32)
    ends[:6] = torch.tensor([0, 1, 511, 512, 513, cols], dtype=torch.int32)
    for k in (1, 33, 512):
        got, want = run_topk(x, k, ends, k + 9)
        assert_rows_equal(got, want, f"{dtype} cols={cols} k={k}")


@pytest.mark.parametrize("dtype,cols", [(torch.float32, 20480), (torch.bfloat16, 30720)])
def test_topk_short_cta_wide_rows_full_wave(dtype, cols):
    """Rows of 16K-45K columns in a batch that fills a wave of CTAs take the
    128-thread CTA (its list-fit rule); every row against the oracle."""
    rows = 1024
    x, ends = inputs.prefill(rows=rows, cols=cols, seed=cols + 11, dtype=dtype)
    ends[:3] = torch.tensor([0, 700, cols], dtype=torch.int32)
    got, want = run_topk(x, 512, ends, 512 + 7)
    assert_rows_equal(got, want, f"{dtype} {rows}x{cols}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cols,ld", [(3001, 3003), (20001, 20005), (777, 777)])
def test_topk_unaligned_rows(dtype, cols, ld):
    x, ends = inputs.prefill(rows=16, cols=cols, seed=7, dtype=dtype)
    got, want = run_topk(x, 300, ends, 300, ld_x=ld)
    assert_rows_equal(got, want, f"unaligned {dtype} cols={cols} ld={ld}")


@pytest.mark.parametrize("k", [1, 2047, 2048, 2049, 4096])
def test_topk_large_k_and_no_row_ends(k):
    x, _ = inputs.prefill(rows=8, cols=70000, seed=k)
    got, want = run_topk(x, k, None, k)
    assert_rows_equal(got, want, f"k={k}")


def test_topk_special_values_and_ties():
    rows, cols = 12, 6000
    g = torch.Generator().manual_seed(3)
    levels = torch.tensor([float("-inf"), -2.0, -0.0, 0.0, 1.5, float("inf"), float("nan")])
    x = levels[torch.randint(0, len(levels), (rows, cols), generator=g)]
    x[0] = float("nan")                          # all-NaN row
    x[1] = 1.0                                   # one value everywhere
    x[2, :] = -0.0
    x[2, 100:110] = 0.0
    ends = torch.full((rows,), cols, dtype=torch.int32)
    for k in (1, 10, 11, 512, 4096):
        got, want = run_topk(x, k, ends, k + 3)
        assert_rows_equal(got, want, f"specials k={k}")
        xb = x.to(torch.bfloat16)
        got, want = run_topk(xb, k, ends, k + 3)
        assert_rows_equal(got, want, f"specials bf16 k={k}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("ld", [8192, 8195])
def test_topk_warp_rows_edges(dtype, ld):
    """Rows short enough for one warp per row: row ends around the list
    size and the sample's run layout, a clustered top block the sample can
    miss, and few-level rows whose list overflows (the exact path)."""
    rows, cols = 40, 8192
    x, _ = inputs.prefill(rows=rows, cols=cols, seed=ld, dtype=torch.float32)
    g = torch.Generator().manual_seed(ld)
    x[30, 3000:3600] = 10.0 + torch.rand(600, generator=g)   # clustered top block
    x[31, 5000:5300] = 7.0                                   # clustered, tied
    x[32] = torch.randint(0, 3, (cols,), generator=g).float()  # three levels
    x[33] = torch.randint(0, 40, (cols,), generator=g).float()
    x[34, ::3] = float("nan")
    ends = torch.full((rows,), cols, dtype=torch.int32)
    ends[:12] = torch.tensor([0, 31, 32, 511, 1024, 1025, 1046, 1100, 1535, 1536, 1537, 4097],
                             dtype=torch.int32)
    x = x.to(dtype)
    for k in (1, 100, 512):
        got, want = run_topk(x, k, ends, k + 5, ld_x=ld)
        assert_rows_equal(got, want, f"warp rows {dtype} ld={ld} k={k}")


@pytest.mark.parametrize("rows,dtype,ld", [(8, torch.float32, 70000), (200, torch.bfloat16, 70000),
                                           (600, torch.float32, 70000),
                                           (1000, torch.float32, 70004),
                                           (600, torch.bfloat16, 70001)])
def test_topk_few_long_rows(rows, dtype, ld):
    """Few long rows: rows that fill less than a wave of resident CTAs take
    a cluster per row, the smallest of 2, 4, 8 CTAs whose clusters fill one
    (8 rows: eight; 200: four; 600: two at K <= 1024, where 608 CTAs are
    resident, one CTA per row at K = 2048), more rows one CTA per row (1000).
    Random row ends around the slice and list sizes, NaN, constant and
    few-level rows (the exact path), fp32 and bf16, aligned and unaligned
    rows; sampled rows against the oracle."""
    cols = 70000
    x, _ = inputs.prefill(rows=rows, cols=cols, seed=rows + ld, dtype=torch.float32)
    g = torch.Generator().manual_seed(rows)
    ends = torch.randint(0, cols + 1, (rows,), generator=g, dtype=torch.int32)
    special = {0: 0, 1: cols, 2: 4000, 3: 16352, 4: 16353, 5: 32704, 6: 32705, 7: 65535}
    for r, e in special.items():
        ends[r] = e
    x[1] = float("nan")
    x[2, ::2] = float("nan")
    if rows == 8:  # the cluster threshold's ordered-key fallback on eight-CTA clusters
        x[6, ::97] = float("inf")                             # an infinity in the range
        x[7] = 0.5                                            # a single value
    if rows > 8:
        for r, e in enumerate((8176, 8177, 16368, 16369, 32736, 65472, 65473), start=11):
            ends[r] = e                                       # list-size boundaries
        x[8] = 0.5                                            # one value
        x[9] = torch.randint(0, 4, (cols,), generator=g).float()  # four levels
        x[10, 100:700] = 9.0                                  # a clustered tied top block
    x = x.to(dtype)
    sample = sorted(set(range(min(rows, 18))) |
                    set(np.random.default_rng(rows).integers(0, rows, 24).tolist()))
    buf = torch.zeros((rows, ld), dtype=dtype, device=DEV)
    buf[:, :cols] = x.to(DEV)
    for k in (1, 512, 2048):
        out = torch.full((rows, k + 3), CANARY, dtype=torch.int32, device=DEV)
        satk.topk_rows(buf[:, :cols], k, row_ends=ends.to(DEV), out=out)
        got = out.cpu().numpy()[sample]
        want = np.full((len(sample), k + 3), CANARY, dtype=np.int32)
        oracle.topk_rows(host_view(x[sample]), k, row_ends=ends[sample].numpy(), out=want)
        assert_rows_equal(got, want, f"few long rows={rows} {dtype} k={k}")


@pytest.mark.parametrize("rows,cols,dtype", [(700, 40000, torch.float32),
                                             (64, 12000, torch.float32),
                                             (64, 12000, torch.bfloat16)])
def test_topk_sample_defeating_rows(rows, cols, dtype):
    """Rows shaped against a sampled threshold, on the CTA-per-row paths
    (700 x 40000: 256 threads per row; 64 x 12000: 128): a hidden block of
    large values, a sparse periodic top, ramps both ways, a tie exactly at
    the K-th value, a top block at the row's end, half the row -inf, and a
    huge dynamic range.  Each must come out as the oracle's."""
    x, _ = inputs.prefill(rows=rows, cols=cols, seed=cols + rows, dtype=torch.float32)
    g = torch.Generator().manual_seed(rows + cols)
    ends = torch.randint(0, cols + 1, (rows,), generator=g, dtype=torch.int32)
    ends[:8] = cols
    off = int(torch.randint(0, cols - 600, (1,), generator=g))
    x[0, off:off + 600] = 10.0 + torch.rand(600, generator=g)      # hidden block
    x[1, 7::61] = 5.0 + torch.rand(len(range(7, cols, 61)), generator=g)  # sparse period
    x[2] = torch.arange(cols, dtype=torch.float32)                  # ascending ramp
    x[3] = -torch.arange(cols, dtype=torch.float32)                 # descending ramp
    x[4] = 1.0
    x[4, torch.randperm(cols, generator=g)[:511]] = 3.0             # K-th value tied
    x[5] = 1.0
    x[5, cols - 513:] = 2.0                                         # top block at the end
    x[6, : cols // 2] = float("-inf")
    x[7] = x[7] * torch.where(torch.rand(cols, generator=g) < 0.5, 1e30, 1e-30)
    x = x.to(dtype)
    sample = sorted(set(range(12)) | set(np.random.default_rng(cols).integers(0, rows, 12).tolist()))
    xd = x.to(DEV)
    for k in (1, 512, 2048):
        out = torch.full((rows, k + 3), CANARY, dtype=torch.int32, device=DEV)
        satk.topk_rows(xd, k, row_ends=ends.to(DEV), out=out)
        got = out.cpu().numpy()[sample]
        want = np.full((len(sample), k + 3), CANARY, dtype=np.int32)
        oracle.topk_rows(host_view(x[sample]), k, row_ends=ends[sample].numpy(), out=want)
        assert_rows_equal(got, want, f"sample-defeating {rows}x{cols} {dtype} k={k}")


def test_topk_decode_shaped_few_rows():
    """A handful of very long bf16 rows (the benchmark's 4 x 524288 case and
    shorter row ends), K = 384 and 2048."""
    x, _ = inputs.prefill(rows=5, cols=524288, seed=1260, causal=False, dtype=torch.bfloat16)
    ends = torch.tensor([524288, 524287, 300001, 70000, 5], dtype=torch.int32)
    for k in (384, 2048):
        got, want = run_topk(x, k, ends, k)
        assert_rows_equal(got, want, f"few rows k={k}")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("cols,ld", [(3000, 3000), (20001, 20003), (70000, 70000)])
def test_topk_sorted(dtype, cols, ld):
    """Score-sorted output: every K class (sort widths 512 to 4096), short
    rows, ties, NaN and signed zeros, aligned and unaligned rows."""
    rows = 12
    x, _ = inputs.prefill(rows=rows, cols=cols, seed=cols + 3, dtype=torch.float32)
    g = torch.Generator().manual_seed(cols)
    ends = torch.randint(0, cols + 1, (rows,), generator=g, dtype=torch.int32)
    ends[:4] = torch.tensor([0, 5, 600, cols], dtype=torch.int32)
    x[4] = torch.randint(0, 3, (cols,), generator=g).float()  # three levels
    x[5, ::2] = float("nan")
    x[6, :] = -0.0
    x[6, 1::3] = 0.0
    x = x.to(dtype)
    for k in (1, 300, 512, 1000, 2048, 4096):
        got, want = run_topk(x, k, ends, k + 2, ld_x=ld, sorted=True)
        assert_rows_equal(got, want, f"sorted {dtype} cols={cols} k={k}")


@pytest.mark.parametrize("mode", ["plus100", "times1e-8"])
def test_topk_concentrated_distributions(mode):
    x, ends = inputs.prefill_shifted(64, 8192, mode)
    got, want = run_topk(x, 512, ends, 512)
    assert_rows_equal(got, want, mode)
    x, ends = inputs.prefill_shifted(16, 51200, mode)
    got, want = run_topk(x, 512, ends, 512)
    assert_rows_equal(got, want, mode + " long")


def test_adversarial_workload_full():
    x, ends, nan_row = inputs.adversarial(seed=1239)  # 256 x 131072 bf16, K=2048
    got, want = run_topk(x, 2048, ends, 2048 + 64)
    assert_rows_equal(got, want, "adversarial")
    xb = bits_of(x)
    f = (xb.astype(np.uint32) << 16).view(np.float32)
    for i in [0, 1, 2, 3, 4, 5, nan_row]:
        e = max(0, min(int(ends[i]), xb.shape[1]))
        check_topk_row(f[i], e, 2048, got[i], ld_canary=CANARY)
        check_topk_layout(f[i], e, 2048, got[i])


@pytest.mark.parametrize("cols", inputs.PREFILL_COLS)
def test_prefill_full_size_every_row(cols):
    """The prefill workload at full size (4096 rows, K = 512, strided
    output), in the launch configuration the benchmark times: every row
    against the oracle, canaries past K intact."""
    x, ends = inputs.prefill(rows=inputs.PREFILL_ROWS, cols=cols, seed=1236, device=DEV)
    check_full_size(x, ends, inputs.PREFILL_LD_OUT, what=f"prefill {cols}")


def test_prefill_sorted_full_size_every_row():
    """The score-sorted option on the prefill 8192-column width at full size
    (4096 rows, K = 512, the benchmark's workload; one warp per row and the
    bucket sort): every row against the oracle's score order."""
    x, ends = inputs.prefill(rows=inputs.PREFILL_ROWS, cols=8192, seed=1236, device=DEV)
    check_full_size(x, ends, inputs.PREFILL_LD_OUT, what="sorted 8192", sorted=True)


@pytest.mark.parametrize("rows,cols", [(8192, 4096), (8192, 8192), (2048, 25600), (2048, 51200),
                                       (1310, 102400)])
def test_prefill_page_shapes_every_row(rows, cols):
    """The other query-row x column shapes the benchmark reports, at full
    size, every row against the oracle."""
    x, ends = inputs.prefill(rows=rows, cols=cols, seed=1250, device=DEV)
    check_full_size(x, ends, inputs.PREFILL_K, what=f"{rows}x{cols}")


@pytest.mark.parametrize("mode", ["plus100", "times1e-8"])
def test_prefill_shifted_full_size_every_row(mode):
    """The distribution ablation the benchmark reports, 8192 x 8192, at full
    size, every row against the oracle."""
    x, ends = inputs.prefill_shifted(8192, 8192, mode, device=DEV)
    check_full_size(x, ends, inputs.PREFILL_K, what=mode)


def check_full_size(x, ends, ld_out, what, chunk=1024, sorted=False):
    """Every row of a full-size launch against the oracle, canaries past K
    included (the oracle runs in row chunks to bound host memory)."""
    rows, k = x.shape[0], inputs.PREFILL_K
    out = torch.full((rows, ld_out), CANARY, dtype=torch.int32, device=DEV)
    satk.topk_rows(x, k, row_ends=ends, out=out, sorted=sorted)
    got = out.cpu().numpy()
    ends_h = ends.cpu().numpy()
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        want = np.full((r1 - r0, ld_out), CANARY, dtype=np.int32)
        oracle.topk_rows(x[r0:r1].cpu().numpy(), k, row_ends=ends_h[r0:r1], out=want,
                         sorted=sorted)
        assert_rows_equal(got[r0:r1], want, f"{what} rows {r0}..{r1}")
    # every row (N(0,1): no NaN): min(end, k) ids in [0, end), unique, then
    # -1, canaries intact
    assert np.all(got[:, k:] == CANARY)
    e = np.clip(ends.cpu().numpy().astype(np.int64), 0, x.shape[1])
    nsel = np.minimum(e, k)
    pos = np.arange(k)[None, :]
    ids = got[:, :k]
    sel = pos < nsel[:, None]
    assert np.all(np.where(sel, (ids >= 0) & (ids < e[:, None]), ids == -1))
    srt = np.sort(np.where(sel, ids, -1 - pos), axis=1)
    assert np.all(srt[:, 1:] != srt[:, :-1])


# ------------------------------------------------------------------ pack --

def test_pack_matches_oracle():
    W, T, S, n = 4, 16, 5000, 128
    lg, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=512, skew_count=50, seed=9)
    x = lg.view(W * T, S)
    xb = bits_of(x)
    g = torch.Generator().manual_seed(1)
    local = torch.randint(-3, S + 3, (W * T, n), generator=g, dtype=torch.int32)
    local[0] = torch.arange(n)
    ends = torch.randint(0, S + 10, (W * T,), generator=g, dtype=torch.int32)
    xb[3, :] = 0x7FC1  # a NaN row
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16)
    got = satk.dcp_pack(x.to(DEV), local.to(DEV), row_ends=ends.to(DEV)).cpu().numpy()
    want = oracle.dcp_pack(xb, local.numpy(), row_ends=ends.numpy())
    assert_rows_equal(got, want, "pack")


def test_pack_hand_worked_example_on_gpu():
    from test_oracle_pins import _pack_golden_inputs
    g, logits, idx, S = _pack_golden_inputs()
    x = torch.from_numpy(logits.view(np.int16)).view(torch.bfloat16).to(DEV)
    got = satk.dcp_pack(x, torch.from_numpy(idx).to(DEV),
                        row_ends=torch.tensor([S], dtype=torch.int32, device=DEV)).cpu().numpy()
    want = np.zeros(33, dtype=np.int32)
    for e in g:
        want[e["j"]] = e["word"]
    want[32] = 0x22
    assert got[0].tolist() == want.tolist()


# ----------------------------------------------------------------- merges --

@pytest.mark.parametrize("W,R,k,local", [(8, 48, 2048, 16384), (2, 20, 512, 4096),
                                         (4, 9, 1024, 3000), (16, 6, 2048, 4096)])
def test_pairs_merge_matches_oracle(W, R, k, local):
    cand = inputs.pairs_merge(W=W, rows=R, k=k, local=local, seed=W * R)
    got = satk.dcp_merge_select(cand.to(DEV), k, packed=False).cpu().numpy()
    want = oracle.merge_pairs(cand.numpy(), k)
    assert_rows_equal(got, want, f"pairs W={W}")


def test_pairs_merge_ties_empties_and_short_rows():
    W, T, n, k = 4, 6, 64, 96
    g = torch.Generator().manual_seed(5)
    sc = torch.tensor([1.0, 2.0, -0.0, 0.0, float("inf"), float("nan")])[
        torch.randint(0, 6, (W, T, n), generator=g)]
    gid = torch.randperm(W * T * n, generator=g).view(W, T, n).to(torch.int32)
    gid[:, 1, ::3] = -1                                   # empties
    gid[:, 2, 5:] = -1                                    # a short row
    cand = torch.stack([sc.contiguous().view(torch.int32), gid], dim=-1).contiguous()
    for kk in (1, 7, k, W * n, W * n + 5):
        got = satk.dcp_merge_select(cand.to(DEV), kk, packed=False).cpu().numpy()
        want = oracle.merge_pairs(cand.numpy(), kk)
        assert_rows_equal(got, want, f"pairs ties k={kk}")


def test_pairs_merge_sampled_threshold_edge_ranges():
    """Rows with more candidates than the list holds take the sampled
    value threshold; these rows give it the ranges it must not trust or
    must refine: an infinity among the scores, a single score value, a few
    levels (a crowded histogram bin), an overflowing span (-3e38 .. 3e38),
    mostly empty pairs (fewer valid samples than the rank), and signed
    zeros with NaN."""
    W, T, n = 8, 8, 2048
    g = torch.Generator().manual_seed(77)
    sc = torch.randn((W, T, n), generator=g)
    sc[:, 0, ::97] = float("inf")
    sc[:, 1] = 1.5
    sc[:, 2] = torch.randint(0, 4, (W, n), generator=g).float()
    sc[:, 3, ::2] = 3e38
    sc[:, 3, 1::2] = -3e38
    sc[:, 5] = torch.tensor([-0.0, 0.0, float("nan"), 1e-30])[
        torch.randint(0, 4, (W, n), generator=g)]
    sc[:, 6, ::5] = float("-inf")
    gid = torch.randperm(W * T * n, generator=g).view(W, T, n).to(torch.int32)
    gid[:, 4, 7:] = -1                                    # mostly empty
    gid[:, 7, ::2] = -1                                   # half empty
    cand = torch.stack([sc.contiguous().view(torch.int32), gid], dim=-1).contiguous()
    for kk in (1, 100, 2048, 3000):
        got = satk.dcp_merge_select(cand.to(DEV), kk, packed=False).cpu().numpy()
        want = oracle.merge_pairs(cand.numpy(), kk)
        assert_rows_equal(got, want, f"pairs edge ranges k={kk}")


@pytest.mark.parametrize("W,n", [(2, 32), (8, 2048)])
def test_merges_exactly_k_equal_candidates(W, n):
    """Rows that hold exactly K non-empty candidates, all with the same
    score (K = 1: a single candidate): nothing is tied beyond the K-th, so
    every candidate is chosen -- on the pairs merge (the list path below
    the list's capacity, the sampled path above it) and on the packed list
    engine."""
    T = 6
    g = torch.Generator().manual_seed(W * n)
    for kk in (1, 3):
        sc = torch.full((W, T, n), 0.75)
        gid = torch.full((W, T, n), -1, dtype=torch.int32)
        for t in range(T):
            slots = torch.randperm(W * n, generator=g)[:kk]
            for f in slots.tolist():
                gid[f // n, t, f % n] = torch.randint(0, 1 << 20, (1,), generator=g).item() * W
        cand = torch.stack([sc.contiguous().view(torch.int32), gid], dim=-1).contiguous()
        got = satk.dcp_merge_select(cand.to(DEV), kk, packed=False).cpu().numpy()
        want = oracle.merge_pairs(cand.numpy(), kk)
        assert (want >= 0).all()
        assert_rows_equal(got, want, f"pairs exactly {kk} W={W} n={n}")
    if W * n > 4096:
        return
    words = n + n // 32
    for kk in (1, 3):
        packed = torch.zeros((W, T, words), dtype=torch.int32)
        for t in range(T):
            for f in torch.randperm(W * n, generator=g)[:kk].tolist():
                packed[f // n, t, f % n] = (0x4100 << 16) | (0xffff - (f % n) * 3)
        ids = satk.dcp_merge_select(packed.to(DEV), kk, packed=True).cpu().numpy()
        o_ids, _, _ = oracle.merge_packed(packed.numpy(), kk)
        assert (o_ids >= 0).all()
        assert_rows_equal(ids, o_ids, f"packed exactly {kk}")


def test_pairs_merge_full_size_every_row():
    """The rank-major merge workload at full size (W = 8, 6710 rows, 8 x
    2048 candidates per row, K = 2048): every row against the oracle."""
    W, R, k = 8, 6710, 2048
    cand = inputs.pairs_merge(W=W, rows=R, k=k, local=16384, seed=1236, device=DEV)
    ids, guard = guarded((R, k))
    satk.dcp_merge_select(cand, k, packed=False, ids_out=ids)
    guard("pairs ids")
    got = ids.cpu().numpy()
    want = oracle.merge_pairs(cand.cpu().numpy(), k)
    assert_rows_equal(got, want, "pairs full size")


@pytest.mark.parametrize("k", [2049, 3000, 4096])
def test_pairs_merge_k_above_2048(k):
    """K above 2048 takes the wider list (8 warps x 1024 entries); 8 ranks
    of 2048 candidates exceed it, so the sampled threshold runs too."""
    W, R, n = 8, 24, 2048
    cand = inputs.pairs_merge(W=W, rows=R, k=n, local=8192, seed=k, device=DEV)
    got = satk.dcp_merge_select(cand, k, packed=False).cpu().numpy()
    want = oracle.merge_pairs(cand.cpu().numpy(), k)
    assert_rows_equal(got, want, f"pairs k={k}")


@pytest.mark.parametrize("k", [512, 3000])
def test_pairs_merge_16_byte_aligned_buffer(k):
    """A pairs buffer that starts 16 bytes past a 32-byte boundary (two
    pairs into an allocation) takes the 128-bit load path."""
    W, R, n = 4, 20, 2048
    cand = inputs.pairs_merge(W=W, rows=R, k=n, local=8192, seed=k + 1, device=DEV)
    flat = torch.zeros(cand.numel() + 8, dtype=torch.int32, device=DEV)
    view = flat[4:4 + cand.numel()].view(cand.shape)
    view.copy_(cand)
    assert view.data_ptr() % 32 == 16
    got = satk.dcp_merge_select(view, k, packed=False).cpu().numpy()
    want = oracle.merge_pairs(cand.cpu().numpy(), k)
    assert_rows_equal(got, want, f"pairs 16-byte aligned k={k}")


def _decode_gpu(lg, n, k, row_ends=None):
    W, T, S = lg.shape
    g = lg.to(DEV)
    re = None if row_ends is None else row_ends.to(DEV)
    local, g_local = guarded((W * T, n))
    satk.topk_rows(g.view(W * T, S), n, row_ends=None if re is None else re.view(-1), out=local)
    packed, g_packed = guarded((W, T, n + n // 32))
    satk.dcp_pack(g.view(W * T, S), local, row_ends=None if re is None else re.view(-1),
                  out=packed.view(W * T, n + n // 32))
    sat, g_sat = guarded((T,), fill=0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids1, g_ids1 = guarded((T, k))
    satk.dcp_merge_select(packed, k, packed=True, ids_out=ids1, sat_word=sat, status=status)
    slots = (k - 1) // n
    recv, g_recv = guarded((T * slots * (k + k // 32),), fill=123)
    ids2, g_ids2 = guarded((T, k))
    ids2.copy_(ids1)
    satk.dcp_rescue_select(packed, g, sat, ids2, k, recv=recv, row_ends=re, status=status)
    torch.cuda.synchronize()
    for chk, what in ((g_local, "local"), (g_packed, "packed"), (g_sat, "sat_word"),
                      (g_ids1, "round-1 ids"), (g_recv, "recv"), (g_ids2, "rescued ids")):
        chk(what)
    return dict(local=local.cpu().numpy(), packed=packed.cpu().numpy(), ids1=ids1.cpu().numpy(),
                sat=sat.cpu().numpy(), ids2=ids2.cpu().numpy(),
                recv=recv.cpu().numpy().reshape(T, slots, k + k // 32),
                status=int(status.item()))


def _decode_oracle(lg, n, k, row_ends=None):
    W, T, S = lg.shape
    bits = bits_of(lg)
    re = None if row_ends is None else row_ends.numpy()
    local = oracle.topk_rows(bits.reshape(W * T, S), n,
                             row_ends=None if re is None else re.reshape(-1))
    packed = oracle.dcp_pack(bits.reshape(W * T, S), local,
                             row_ends=None if re is None else re.reshape(-1)).reshape(
        W, T, n + n // 32)
    ids1, sat, st1 = oracle.merge_packed(packed, k)
    slots = (k - 1) // n
    recv = np.full((T, slots, k + k // 32), 123, dtype=np.int32)
    ids2, recv, st2 = oracle.rescue(packed, k, bits, sat, ids1.copy(), row_ends=re, recv=recv)
    return dict(local=local, packed=packed, ids1=ids1, sat=sat, ids2=ids2, recv=recv,
                status=st1 | st2)


def _compare_decode(got, want, what):
    for key in ("local", "packed", "ids1", "sat", "ids2", "recv"):
        a, b = got[key], want[key]
        a2 = a.reshape(a.shape[0], -1) if a.ndim > 2 else a.reshape(len(a), -1)
        b2 = b.reshape(b.shape[0], -1) if b.ndim > 2 else b.reshape(len(b), -1)
        assert_rows_equal(a2, b2, f"{what}: {key}")
    assert got["status"] == want["status"], f"{what}: status {got['status']} vs {want['status']}"


def test_decode_merge_full_workload():
    W, T, S, n, k = 8, 128, 65536, 384, 2048
    lg, skewed, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, seed=1237, device=DEV)
    lg = lg.cpu()
    got = _decode_gpu(lg, n, k)
    want = _decode_oracle(lg, n, k)
    _compare_decode(got, want, "decode full")
    mask = (want["sat"].astype(np.int64) & 0xFFFFFFFF) >> 16
    assert np.array_equal(mask != 0, skewed.cpu().numpy())
    bits = bits_of(lg)
    for t in range(T):
        check_decode_merge_row(got["ids2"][t], bits, t, k)
    packed_contract(got["packed"].reshape(W * T, -1), bits.reshape(W * T, S), None, n)


@pytest.mark.parametrize("k", [512, 2048])
def test_decode_merge_long_rank_rows(k):
    """Rank rows long enough for the clustered push: row ends around the
    cluster's slice and list sizes, a half-NaN rank row, a skewed rank."""
    W, T, S, n = 4, 16, 40000, 128
    lg, skewed, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=400, seed=k)
    bits = bits_of(lg)
    bits[1, 3, 1::2] = 0xFFC3
    lg = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    g = torch.Generator().manual_seed(k)
    ends = torch.randint(S // 2, S + 50, (W, T), generator=g, dtype=torch.int32)
    ends[:, 0] = torch.tensor([0, 10, 65472 // 8 * 8, S])[:W]
    ends[:, 1] = torch.tensor([32704, 32705, 32736, 32737])[:W]
    got = _decode_gpu(lg, n, k, row_ends=ends)
    want = _decode_oracle(lg, n, k, row_ends=ends)
    _compare_decode(got, want, f"decode long rank rows k={k}")


def test_decode_rescue_massive_ties():
    """Four saturated ranks whose pushed lists tie with the round-1 cut:
    every pushed word scores >= tau16, so the filtered rescue list overflows
    and the row takes the register select over every slot; the other ranks
    hold a single value.  Bit-exact against the oracle."""
    W, T, S, n, k = 8, 4, 5000, 256, 2048
    g = torch.Generator().manual_seed(31)
    x = torch.full((W, T, S), 0.5)
    for r in range(4):
        for t in range(T):
            pos = torch.randperm(S, generator=g)[:300]
            x[r, t, pos] = 4.0 + torch.rand(300, generator=g)
    lg = x.to(torch.bfloat16)
    got = _decode_gpu(lg, n, k)
    want = _decode_oracle(lg, n, k)
    _compare_decode(got, want, "decode massive ties")
    assert int(((want["sat"] >> 16) != 0).sum()) > 0, "the case must saturate"


def test_decode_merge_row_ends_nan_and_small():
    W, T, S, n, k = 4, 12, 3000, 64, 512
    lg, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=120, seed=77)
    bits = bits_of(lg)
    bits[2, 5, ::2] = 0xFFC3                 # half of a rank's row NaN
    lg = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    g = torch.Generator().manual_seed(2)
    ends = torch.randint(0, S + 50, (W, T), generator=g, dtype=torch.int32)
    ends[0, 0] = 0
    ends[1, 1] = 10
    got = _decode_gpu(lg, n, k, row_ends=ends)
    want = _decode_oracle(lg, n, k, row_ends=ends)
    _compare_decode(got, want, "decode small")


def test_packed_merge_wide():
    """W * n above the list engine's capacity: the register merge (16 ranks
    of 1024 candidates), ids, saturation words and status against the
    oracle."""
    W, T, S, n, k = 16, 4, 5000, 1024, 2048
    lg, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=1500, seed=41)
    bits = bits_of(lg)
    local = oracle.topk_rows(bits.reshape(W * T, S), n)
    packed = oracle.dcp_pack(bits.reshape(W * T, S), local).reshape(W, T, n + n // 32)
    sat = torch.zeros(T, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids = satk.dcp_merge_select(torch.from_numpy(packed).to(DEV), k, packed=True, sat_word=sat,
                                status=st)
    w_ids, w_sat, w_st = oracle.merge_packed(packed, k)
    assert_rows_equal(ids.cpu().numpy(), w_ids, "wide packed merge")
    assert np.array_equal(sat.cpu().numpy(), w_sat) and int(st.item()) == w_st


def test_packed_merge_out_of_contract_words():
    """Repeated words (a NaN row's arbitrary ids on the page) and more
    saturated ranks than slots: bit-exact status, ids and sat_word.  Row 0
    repeats one word per rank, so the repeated key straddles the cut at
    k = 48: fewer than k are chosen, tau16 falls to 0 and all four full
    ranks count as saturated, more than the one rescue slot."""
    W, T, n, k = 4, 3, 32, 48
    words = n + n // 32
    p = np.zeros((W, T, words), dtype=np.int32)
    hi = np.uint32((0xBF80 << 16) | (0xFFFF - 3))
    p[:, 0, :n] = np.array([hi] * n, dtype=np.uint32).view(np.int32)     # duplicates
    rng = np.random.default_rng(0)
    for r in range(W):  # every rank full and high: 4 saturated ranks, 1 slot
        sc = rng.integers(0xC000, 0xF000, size=n).astype(np.uint32)
        p[r, 1, :n] = ((sc << 16) | (0xFFFF - np.arange(n, dtype=np.uint32))).view(np.int32)
    p[:, 2, :n] = np.int32(5)                                          # zero score field
    got_sat = torch.zeros(T, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids = satk.dcp_merge_select(torch.from_numpy(p).to(DEV), k, packed=True, sat_word=got_sat,
                                status=st)
    w_ids, w_sat, w_st = oracle.merge_packed(p, k)
    assert_rows_equal(ids.cpu().numpy(), w_ids, "out of contract ids")
    assert got_sat.cpu().numpy().tolist() == w_sat.tolist()
    assert int(st.item()) == w_st


# -------------------------------------------------------------- ABI edges --

def test_abi_rejects_with_real_buffers():
    x = torch.zeros((4, 100), device=DEV)
    out = torch.zeros((4, 8), dtype=torch.int32, device=DEV)
    L = binding.lib()
    import ctypes
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert L.satk_topk_rows(p(x), 0, 4, 100, 99, None, 8, p(out), 8, None) == -1
    assert L.satk_topk_rows(p(x), 0, 4, 100, 100, None, 9, p(out), 8, None) == -1
    assert L.satk_topk_rows(p(x), 5, 4, 100, 100, None, 8, p(out), 8, None) == -1
    assert L.satk_dcp_merge_select(p(out), 1, 17, 1, 32, 8, p(out), 8, None, None, None) == -1
    assert L.satk_dcp_merge_select(p(out), 0, 1, 1, 48, 8, p(out), 8, None, None, None) == -1
    torch.cuda.synchronize()
    assert np.all(out.cpu().numpy() == 0)  # nothing was launched


def test_empty_batches_are_no_ops():
    """Zero rows (torch hands out a null data pointer for them): every entry
    point returns at once with nothing written and nothing raised."""
    W, n, k, S = 4, 64, 512, 1000
    x = torch.empty((0, 5000), device=DEV)
    assert satk.topk_rows(x, 512).shape == (0, 512)
    assert satk.topk_rows(x, 512, row_ends=torch.empty(0, dtype=torch.int32, device=DEV),
                          sorted=True).shape == (0, 512)
    lg = torch.empty((0, S), dtype=torch.bfloat16, device=DEV)
    local = torch.empty((0, n), dtype=torch.int32, device=DEV)
    assert satk.dcp_pack(lg, local).shape == (0, n + n // 32)
    packed = torch.empty((W, 0, n + n // 32), dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sat = torch.empty(0, dtype=torch.int32, device=DEV)
    ids = satk.dcp_merge_select(packed, k, packed=True, sat_word=sat, status=status)
    assert ids.shape == (0, k)
    pairs = torch.empty((W, 0, 256, 2), dtype=torch.int32, device=DEV)
    assert satk.dcp_merge_select(pairs, 256, packed=False).shape == (0, 256)
    logits = torch.empty((W, 0, S), dtype=torch.bfloat16, device=DEV)
    satk.dcp_rescue_select(packed, logits, sat, ids, k, status=status)
    table = torch.zeros((3, 16), dtype=torch.int32, device=DEV)
    rows, valid = satk.dcp_emit_rows(ids, W, 0, torch.empty(0, dtype=torch.int32, device=DEV),
                                     table, 64, 64, status=status)
    assert rows.shape == (0, k) and valid.shape == (0,)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


# ------------------------------------------------------------- emit_rows --

def run_emit_rows(ids, W, rank, req, table, B, stride, max_blocks=None, ld_rows=None):
    """GPU (through the C ABI) and oracle outputs for host int32 arrays."""
    T, k = ids.shape
    ld_rows = k if ld_rows is None else ld_rows
    rows, g_rows = guarded((T, ld_rows), fill=CANARY)
    valid, g_valid = guarded((T,), fill=CANARY)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    satk.dcp_emit_rows(torch.from_numpy(ids).to(DEV), W, rank, torch.from_numpy(req).to(DEV),
                       torch.from_numpy(table).to(DEV), B, stride, max_blocks=max_blocks,
                       rows_out=rows[:, :k] if ld_rows != k else rows, valid_out=valid,
                       status=st)
    g_rows("rows_out")
    g_valid("valid_out")
    want_rows, want_valid, want_st = oracle.emit_rows(ids, W, rank, req, table, B, stride,
                                                      max_blocks=max_blocks, ld_rows=ld_rows)
    return (rows.cpu().numpy(), valid.cpu().numpy(), int(st.item())), \
        (want_rows, want_valid, want_st)


def test_emit_rows_hand_worked_example_on_gpu():
    import test_oracle_pins as pins
    g = pins._emit_rows_golden()
    got, want = run_emit_rows(np.array(g["ids"], np.int32), g["W"], g["rank"],
                              np.array(g["req"], np.int32), np.array(g["table"], np.int32),
                              g["block_size"], g["stride_rows"], ld_rows=10)
    assert got[0][:, :8].tolist() == g["rows"]
    assert np.all(got[0][:, 8:] == CANARY)
    assert got[1].tolist() == g["valid"] and got[2] == g["status"]


@pytest.mark.parametrize("k,ld_rows", [(2048, 2048), (64, 70), (13, 13), (5000, 5003)])
def test_emit_rows_matches_oracle(k, ld_rows):
    rng = np.random.default_rng(k)
    T, W, B, width, R = 37, 8, 64, 50, 5
    ids = rng.integers(-3, W * B * width * 5 // 4, size=(T, k)).astype(np.int32)
    ids[3] = -1                                     # an empty row
    table = rng.integers(0, 1 << 20, size=(R, width)).astype(np.int32)
    table[1, 7] = 40_000_000                        # wraps at stride 64
    req = rng.integers(0, R, size=T).astype(np.int32)
    req[5], req[6] = -1, R                          # bad requests
    for rank in (0, 3, 7):
        for max_blocks in (None, 0, 17):
            got, want = run_emit_rows(ids, W, rank, req, table, B, 64, max_blocks=max_blocks,
                                      ld_rows=ld_rows)
            assert_rows_equal(got[0], want[0], f"emit_rows k={k} rank={rank} mb={max_blocks}")
            assert np.array_equal(got[1], want[1]) and got[2] == want[2] == 4


def test_emit_rows_after_the_decode_merge():
    """The decode pipeline's final ids (merge and rescue) to each rank's rows."""
    W, T, S, n, k = 8, 32, 20000, 128, 1024
    lg, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=300, seed=21,
                                   device=DEV)
    local = satk.topk_rows(lg.view(W * T, S), n)
    packed = satk.dcp_pack(lg.view(W * T, S), local).view(W, T, n + n // 32)
    sat = torch.zeros(T, dtype=torch.int32, device=DEV)
    ids = satk.dcp_merge_select(packed, k, packed=True, sat_word=sat)
    satk.dcp_rescue_select(packed, lg, sat, ids, k)
    B = 64
    width = (S + B - 1) // B
    rng = np.random.default_rng(5)
    table = rng.permutation(T * width).astype(np.int32).reshape(T, width)
    req = rng.permutation(T).astype(np.int32)
    ids_h = ids.cpu().numpy()
    total = np.zeros(T, dtype=np.int64)
    for rank in range(W):
        got, want = run_emit_rows(ids_h, W, rank, req, table, B, B)
        assert_rows_equal(got[0], want[0], f"decode emit_rows rank={rank}")
        assert np.array_equal(got[1], want[1]) and got[2] == 0
        total += got[1]
    assert np.array_equal(total, (ids_h >= 0).sum(axis=1))  # every token owned once
