"""Seeded synthetic inputs for the exact per-row top-K path.

This module only draws numbers: it holds none of the selection, packing or
merging arithmetic, so the CUDA path and the CPU oracle can both be fed from
it without sharing any of the method.  Every generator takes an explicit
seed and device and returns plain tensors; shapes default to the workloads
the pages measure or describe, and can be shrunk for tests.

Workloads (pages cited by title and section):
  * prefill top-K -- [Perf][DSA] Use DeepSelect for eligible sparse-indexer
    prefill chunks (vLLM PR #57206), "Synthetic controls": fp32 N(0,1)
    logits, 4096 query rows, causal row ends, K=512, preallocated output.
  * rank-major pairs merge -- vLLM PR #65178, "Overview"/"Claims": W=8,
    6710 rows, top-2048 per rank, (score, global id) pairs, rank-major
    [W, R, K, 2].
  * one-round decode merge -- vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge
    .kernels, module docstring: bf16 logits per rank, local top-N packed,
    saturated ranks rescued.
  * adversarial top-K -- the distribution ablation of PR #57206
    ("Synthetic controls") pushed further: few distinct levels, infinities,
    a NaN row and short rows.
"""
from __future__ import annotations

import torch

PREFILL_ROWS = 4096
PREFILL_COLS = (8192, 51200, 102400)
PREFILL_K = 512
PREFILL_LD_OUT = 640  # strided output: [rows, 640] buffer, top-K in [:, :512]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def bits_to_bf16(bits: torch.Tensor) -> torch.Tensor:
    """int32 tensor of 16-bit patterns (0..65535) -> bf16 tensor with those
    exact bits."""
    signed = bits - ((bits >> 15) & 1) * 0x10000
    return signed.to(torch.int16).view(torch.bfloat16)


def prefill(rows: int = 64, cols: int = 4096, seed: int = 1235, device="cpu",
            causal: bool = True, dtype=torch.float32):
    """fp32 (or bf16) N(0,1) logits [rows, cols] and causal row ends
    ``row_end[i] = cols - rows + i + 1`` (clamped to >= 0), int32."""
    g = _gen(seed, device)
    x = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32)
    if dtype != torch.float32:
        x = x.to(dtype)
    if causal:
        ends = torch.arange(rows, device=device, dtype=torch.int64) + (cols - rows + 1)
        ends = ends.clamp_(min=0).to(torch.int32)
    else:
        ends = torch.full((rows,), cols, device=device, dtype=torch.int32)
    return x, ends


def prefill_shifted(rows: int, cols: int, mode: str, seed: int = 1240, device="cpu"):
    """The distribution ablation of the prefill page: N(0,1), the same
    values + 100, or the same values * 1e-8."""
    x, ends = prefill(rows, cols, seed=seed, device=device)
    if mode == "plus100":
        x = x + 100.0
    elif mode == "times1e-8":
        x = x * 1e-8
    elif mode != "normal":
        raise ValueError(mode)
    return x, ends


def pairs_merge(W: int = 8, rows: int = 6710, k: int = 2048, local: int = 16384,
                seed: int = 1236, device="cpu", keep_logits: bool = False,
                chunk_rows: int = 256):
    """Rank-major candidate pairs [W, rows, k, 2] int32 (element 0 holds the
    float32 score's bits, element 1 the global id ``local_id * W + r``).

    Rank r's list for a row is the k best of its own ``local`` N(0,1) logits
    (score descending, lower local id first among equal scores), stored in a
    seeded random order.  With ``keep_logits`` the per-rank logits
    [W, rows, local] are returned too (for small cases)."""
    g = _gen(seed, device)
    cand = torch.empty((W, rows, k, 2), dtype=torch.int32, device=device)
    logits_all = (torch.empty((W, rows, local), dtype=torch.float32, device=device)
                  if keep_logits else None)
    for t0 in range(0, rows, chunk_rows):
        t1 = min(rows, t0 + chunk_rows)
        lg = torch.randn((W, t1 - t0, local), generator=g, device=device)
        if keep_logits:
            logits_all[:, t0:t1] = lg
        vals, idx = torch.sort(lg, dim=-1, descending=True, stable=True)
        vals, idx = vals[..., :k], idx[..., :k]
        order = torch.argsort(torch.rand((W, t1 - t0, k), generator=g, device=device), dim=-1)
        vals = torch.gather(vals, -1, order)
        idx = torch.gather(idx, -1, order)
        rank = torch.arange(W, device=device, dtype=torch.int64).view(W, 1, 1)
        gid = idx * W + rank
        cand[:, t0:t1, :, 0] = vals.contiguous().view(torch.int32)
        cand[:, t0:t1, :, 1] = gid.to(torch.int32)
    return (cand, logits_all) if keep_logits else cand


def decode_merge(W: int = 8, rows: int = 128, S: int = 65536, n: int = 384,
                 k: int = 2048, skew_frac: float = 0.25, skew_count: int = 600,
                 seed: int = 1237, device="cpu", skew_from: int = 0):
    """bf16 logits [W, rows, S] ~ bf16(N(0,1)); on a seeded quarter of the
    rows one seeded rank gets ``skew_count`` seeded positions (drawn from
    columns [skew_from, S)) set to bf16(N(3.5, 0.25)), so that rank alone
    holds more than n of the row's top-k.  Returns (logits, skewed_rows
    [bool rows], skew_rank [rows] (-1 where not skewed))."""
    g = _gen(seed, device)
    lg = torch.randn((W, rows, S), generator=g, device=device).to(torch.bfloat16)
    n_skew = int(round(rows * skew_frac))
    skew_rows = torch.randperm(rows, generator=g, device=device)[:n_skew]
    skew_rank = torch.full((rows,), -1, dtype=torch.int64, device=device)
    ranks = torch.randint(0, W, (n_skew,), generator=g, device=device)
    skew_rank[skew_rows] = ranks
    for i in range(n_skew):
        t = int(skew_rows[i])
        r = int(ranks[i])
        pos = skew_from + torch.randperm(S - skew_from, generator=g, device=device)[:skew_count]
        vals = (torch.randn((skew_count,), generator=g, device=device) * 0.25 + 3.5)
        lg[r, t, pos] = vals.to(torch.bfloat16)
    skewed = skew_rank >= 0
    return lg, skewed, skew_rank


_NAN_PATTERNS = (0x7FC0, 0x7F81, 0x7FFF, 0xFFC0, 0xFF81, 0xFFFF, 0x7FA5, 0xFFD3)


def adversarial(rows: int = 256, cols: int = 131072, levels: int = 64,
                seed: int = 1239, device="cpu", nan_row: int | None = None,
                short_rows=(0, 1, 2047, 2048, 2049)):
    """bf16 logits [rows, cols] drawn from ``levels`` distinct bf16 values
    (two of them +0.0 and -0.0), ~1% -inf, ~0.1% +inf; one seeded row holds
    NaN (mixed sign and payload) at half its positions; row ends uniform in
    [0, cols] with rows 1..len(short_rows) forced to ``short_rows``.
    Returns (x bf16, row_ends int32, nan_row)."""
    g = _gen(seed, device)
    base = (torch.randn((4 * levels,), generator=g, device=device) * 4).to(torch.bfloat16)
    bits = base.view(torch.int16).to(torch.int32) & 0xFFFF
    uniq = []
    for b in bits.tolist():
        if b not in uniq and b not in (0x0000, 0x8000):
            uniq.append(b)
        if len(uniq) == levels - 2:
            break
    table = torch.tensor(uniq + [0x0000, 0x8000], dtype=torch.int32, device=device)
    pick = torch.randint(0, levels, (rows, cols), generator=g, device=device)
    xb = table[pick]
    u = torch.rand((rows, cols), generator=g, device=device)
    xb = torch.where(u < 0.01, torch.full_like(xb, 0xFF80), xb)
    xb = torch.where((u >= 0.01) & (u < 0.011), torch.full_like(xb, 0x7F80), xb)
    if nan_row is None:
        nan_row = int(torch.randint(len(short_rows) + 1, rows, (1,), generator=g, device=device)) \
            if rows > len(short_rows) + 1 else rows - 1
    nan_sel = torch.rand((cols,), generator=g, device=device) < 0.5
    pats = torch.tensor(_NAN_PATTERNS, dtype=torch.int32, device=device)
    nan_vals = pats[torch.randint(0, len(_NAN_PATTERNS), (cols,), generator=g, device=device)]
    xb[nan_row] = torch.where(nan_sel, nan_vals, xb[nan_row])
    x = bits_to_bf16(xb)
    ends = torch.randint(0, cols + 1, (rows,), generator=g, device=device, dtype=torch.int64)
    for i, e in enumerate(short_rows):
        if 1 + i < rows:
            ends[1 + i] = min(e, cols)
    return x, ends.to(torch.int32), nan_row


def flush_buffer(device, nbytes: int | None = None) -> torch.Tensor:
    """A scratch buffer twice the size of L2 (or ``nbytes``), written between
    timed repetitions so every one starts with a cold L2."""
    if nbytes is None:
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        nbytes = 2 * int(l2)
    return torch.empty(nbytes // 4, dtype=torch.int32, device=device)
