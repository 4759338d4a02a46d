"""Packed B' words on the GPU, bit for bit against the oracle.

* The hand-worked tables of tests/golden/ through the C ABI: words whose
  score field is 0 (candidates below every other score, as the vLLM API
  page vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels, section
  _decode_key, keys them), a mask with more saturated ranks than slots, and
  a rescue whose pushed list holds local ids at and above 2**16.
* The local[16] bit plane through the whole decode pipeline (local top-n,
  pack, merge, push, re-select) on rank rows longer than 2**16 columns,
  with the skewed rank's large values at columns >= 2**16, on both push
  kernels (aligned rows take the clustered push, unaligned rows the
  one-CTA push).
* Zero-score words on both merge engines (the shared-memory list engine and
  the register engine for more than 8192 candidates), and a saturation word
  whose mask names a rank at or above W.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_indexer_radix_gb300 as satk
from guards import guarded
from test_oracle_pins import golden_packed_buffer, load_rescue_plane_golden

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from sparse_attention_indexer_radix_gb300 import build as satk_build
    satk_build.build()
    oracle.build()


def _u32(a):
    return (np.asarray(a).astype(np.int64) & 0xFFFFFFFF).tolist()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _assert_equal(got, want, what):
    got, want = np.asarray(got), np.asarray(want)
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)[:6].tolist()
        raise AssertionError(f"{what}: differ at {bad}: got {[got[tuple(i)] for i in bad]} "
                             f"want {[want[tuple(i)] for i in bad]}")


def _merge_gpu(packed: np.ndarray, k: int):
    T = packed.shape[1]
    sat, g_sat = guarded((T,), fill=77)
    ids, g_ids = guarded((T, k))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    satk.dcp_merge_select(torch.from_numpy(packed).to(DEV), k, packed=True, ids_out=ids,
                          sat_word=sat, status=st)
    g_sat("sat_word")
    g_ids("ids")
    return ids.cpu().numpy(), sat.cpu().numpy(), int(st.item())


# ----------------------------------------------------- hand-worked tables --

@pytest.mark.parametrize("name", ["decode_zero_score_example.txt",
                                  "slots_exceeded_example.txt"])
def test_packed_merge_hand_worked_examples_on_gpu(name):
    packed, cases = golden_packed_buffer(name)
    for c in cases:
        ids, sat, status = _merge_gpu(packed, c["K"])
        assert ids[0].tolist() == c["ids"], (name, c["K"], ids[0].tolist())
        assert _u32(sat)[0] == c["sat"], (name, c["K"], hex(_u32(sat)[0]))
        assert status == c["status"], (name, c["K"], status)


@pytest.mark.parametrize("pad", [0, 7])
def test_rescue_plane_hand_worked_example_on_gpu(pad):
    """The hand-worked rescue with local ids >= 2**16: rows of 2**17 + 1
    columns (pad 0: unaligned rows, the one-CTA push) or padded to a 16-byte
    row stride (pad 7: the clustered push).  Every intermediate is checked."""
    bits, g = load_rescue_plane_golden()
    W, T, S, n, k = g["W"], g["T"], g["S"], g["N"], g["K"]
    ld = S + pad
    host = np.zeros((W, T, ld), dtype=np.uint16)
    host[:, :, :S] = bits
    buf = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).to(DEV)
    lg = buf[:, :, :S]
    flat = buf.view(W * T, ld)[:, :S]
    local = satk.topk_rows(flat, n)
    for r in range(W):
        assert local[r].cpu().tolist() == g["local"][r]
    packed = satk.dcp_pack(flat, local).view(W, T, n + n // 32)
    for r in range(W):
        assert _u32(packed[r, 0].cpu().numpy()) == g["packed"][r], f"packed rank {r}"
    sat = torch.zeros(T, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids = satk.dcp_merge_select(packed, k, packed=True, sat_word=sat, status=st)
    assert ids[0].cpu().tolist() == g["ids1"]
    assert _u32(sat.cpu().numpy())[0] == g["sat"]
    recv = torch.full((T * ((k - 1) // n) * (k + k // 32),), 555, dtype=torch.int32, device=DEV)
    satk.dcp_rescue_select(packed, lg, sat, ids, k, recv=recv, status=st)
    assert _u32(recv.cpu().numpy()) == g["recv"]
    assert ids[0].cpu().tolist() == g["ids2"]
    assert int(st.item()) == g["status"]


# ------------------------------------------------- local[16] end to end --

def _pipeline_gpu(lg_host: torch.Tensor, n: int, k: int, ld: int, row_ends=None):
    W, T, S = lg_host.shape
    buf = torch.zeros((W, T, ld), dtype=torch.bfloat16, device=DEV)
    buf[:, :, :S] = lg_host.to(DEV)
    lg = buf[:, :, :S]
    flat = buf.view(W * T, ld)[:, :S]
    re = None if row_ends is None else row_ends.to(DEV)
    local, g_local = guarded((W * T, n))
    satk.topk_rows(flat, n, row_ends=None if re is None else re.view(-1), out=local)
    packed, g_packed = guarded((W, T, n + n // 32))
    satk.dcp_pack(flat, local, row_ends=None if re is None else re.view(-1),
                  out=packed.view(W * T, n + n // 32))
    fused, g_fused = guarded((W * T, n + n // 32))
    satk.dcp_topk_pack(flat, n, row_ends=None if re is None else re.view(-1), out=fused)
    sat, g_sat = guarded((T,), fill=0)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ids1, g_ids1 = guarded((T, k))
    satk.dcp_merge_select(packed, k, packed=True, ids_out=ids1, sat_word=sat, status=st)
    slots = (k - 1) // n
    recv, g_recv = guarded((T * slots * (k + k // 32),), fill=123)
    ids2, g_ids2 = guarded((T, k))
    ids2.copy_(ids1)
    satk.dcp_rescue_select(packed, lg, sat, ids2, k, recv=recv, row_ends=re, status=st)
    torch.cuda.synchronize()
    for chk, what in ((g_local, "local"), (g_packed, "packed"), (g_fused, "fused pack"),
                      (g_sat, "sat_word"), (g_ids1, "round-1 ids"), (g_recv, "recv"),
                      (g_ids2, "rescued ids")):
        chk(what)
    assert torch.equal(fused.view(W, T, -1), packed), "fused top-n pack differs from the pack"
    return dict(local=local.cpu().numpy(), packed=packed.cpu().numpy(), ids1=ids1.cpu().numpy(),
                sat=sat.cpu().numpy(), ids2=ids2.cpu().numpy(),
                recv=recv.cpu().numpy().reshape(T, slots, k + k // 32), status=int(st.item()))


def _pipeline_oracle(bits: np.ndarray, n: int, k: int, row_ends=None):
    W, T, S = bits.shape
    re = None if row_ends is None else row_ends.numpy()
    flat = bits.reshape(W * T, S)
    fe = None if re is None else re.reshape(-1)
    local = oracle.topk_rows(flat, n, row_ends=fe)
    packed = oracle.dcp_pack(flat, local, row_ends=fe).reshape(W, T, n + n // 32)
    ids1, sat, st1 = oracle.merge_packed(packed, k)
    slots = (k - 1) // n
    recv = np.full((T, slots, k + k // 32), 123, dtype=np.int32)
    ids2, recv, st2 = oracle.rescue(packed, k, bits, sat, ids1.copy(), row_ends=re, recv=recv)
    return dict(local=local, packed=packed, ids1=ids1, sat=sat, ids2=ids2, recv=recv,
                status=st1 | st2)


@pytest.mark.parametrize("W,T,S,n,k,pad,ends", [
    (4, 16, 131072, 384, 2048, 0, False),   # aligned rows: clustered push
    (2, 16, 100000, 128, 512, 0, True),     # aligned, row ends
    (2, 16, 100001, 128, 512, 0, False),    # unaligned rows: one-CTA push
    (4, 12, 140000, 384, 2048, 3, True),    # S above 2**17, unaligned stride
    (3, 8, 131077, 256, 1024, 0, False),    # W not a power of two
])
def test_decode_pipeline_local_plane_bit(W, T, S, n, k, pad, ends):
    """The local[16] plane bit through the decode pipeline: half the rows
    skewed, their large values at columns >= 2**16, so pushed lists and
    round-1 words carry local ids above 2**16 on both push kernels; local
    top-n, packed words, ids of both rounds, sat_word, recv and status
    bit-exact against the oracle."""
    from sparse_attention_indexer_radix_gb300 import inputs
    lg, skewed, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_frac=0.5,
                                        skew_count=3 * n, seed=S + k, skew_from=1 << 16)
    row_ends = None
    if ends:
        g = torch.Generator().manual_seed(S)
        row_ends = torch.randint(70000, S + 40, (W, T), generator=g, dtype=torch.int32)
        row_ends[:, 0] = S                     # one row untouched
    got = _pipeline_gpu(lg, n, k, S + pad, row_ends)
    want = _pipeline_oracle(_bits(lg), n, k, row_ends)
    for key in ("local", "packed", "ids1", "sat", "ids2", "recv"):
        a, b = got[key], want[key]
        _assert_equal(a.reshape(a.shape[0], -1), b.reshape(b.shape[0], -1), key)
    assert got["status"] == want["status"]
    mask = (want["sat"].astype(np.int64) & 0xFFFFFFFF) >> 16
    assert (mask != 0).sum() >= 2, "the case must saturate"
    # the plane bits are exercised: set in round-1 words and in pushed lists
    words = n + n // 32
    assert np.any(want["packed"][:, :, n:words] != 0)
    pushed = want["recv"][(mask != 0)][:, 0, k:]
    assert np.any(pushed != 0), "no pushed local id at or above 2**16"


# ------------------------------------------------ zero-score words, wide --

@pytest.mark.parametrize("W,n", [(4, 512), (16, 1024)])
def test_packed_merge_zero_score_words_both_engines(W, n):
    """Random B' rows with non-zero words whose score field is 0 (and
    plane bits, empty slots, ties): the list engine (W*n <= 8192) and the
    register engine (16 x 1024) against the oracle, several K."""
    T = 6
    rng = np.random.default_rng(W * n)
    words = n + n // 32
    p = np.zeros((W, T, words), dtype=np.uint32)
    for t in range(T):
        score = rng.choice(np.array([0, 0x3F80, 0x4000, 0x8000, 0x7FFF, 0xC000], np.uint32),
                           size=(W, n), p=[0.3, 0.2, 0.2, 0.1, 0.1, 0.1])
        if t == 1:
            score[:] = 0                              # every word scores 0
        if t == 2:
            score[0] = 0xC000                         # a full rank, tau16 0
        low = rng.integers(0, 1 << 16, size=(W, n)).astype(np.uint32)
        w = (score << 16) | low
        w[rng.random((W, n)) < 0.1] = 0               # empty slots
        if t == 3:
            w[:, n // 2:] = 0
        p[:, t, :n] = w
        p[:, t, n:] = rng.integers(0, 1 << 32, size=(W, n // 32), dtype=np.uint64).astype(
            np.uint32)
    packed = p.view(np.int32)
    for k in (1, 37, n, 2048, W * n // 2 + 3, W * n):
        ids, sat, st = _merge_gpu(packed, k)
        w_ids, w_sat, w_st = oracle.merge_packed(packed, k)
        _assert_equal(ids, w_ids, f"ids W={W} n={n} k={k}")
        _assert_equal(sat, w_sat, f"sat_word W={W} n={n} k={k}")
        assert st == w_st, (k, st, w_st)


def test_rescue_mask_bit_at_or_above_W():
    """A saturation word naming a rank at or above W is outside the
    contract: the row keeps its ids and status bit 1 is raised (as a mask
    with more bits than slots)."""
    W, T, S, n, k = 4, 3, 3000, 64, 512
    from sparse_attention_indexer_radix_gb300 import inputs
    lg, _, _ = inputs.decode_merge(W=W, rows=T, S=S, n=n, k=k, skew_count=200, seed=3)
    bits = _bits(lg)
    local = oracle.topk_rows(bits.reshape(W * T, S), n)
    packed = oracle.dcp_pack(bits.reshape(W * T, S), local).reshape(W, T, n + n // 32)
    ids, sat, _ = oracle.merge_packed(packed, k)
    sat = sat.copy()
    sat[1] = (1 << (16 + W)) | 0x8000                 # bit W of the mask
    sat[2] = (1 << (16 + W + 3)) | (1 << 16) | 0x8000
    w_ids, _, w_st = oracle.rescue(packed, k, bits, sat, ids.copy())
    g_ids = torch.from_numpy(ids.copy()).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    satk.dcp_rescue_select(torch.from_numpy(packed).to(DEV), lg.to(DEV),
                           torch.from_numpy(sat).to(DEV), g_ids, k, status=st)
    _assert_equal(g_ids.cpu().numpy(), w_ids, "ids")
    assert int(st.item()) == w_st and (w_st & 1)
    assert np.array_equal(w_ids[1:], ids[1:])


# ------------------------------------------------ fused local top-n pack --

@pytest.mark.parametrize("rows,S,n,ld_pad,ends", [
    (40, 6000, 128, 0, True),        # one warp per row
    (24, 40000, 384, 0, True),       # one CTA per row
    (1024, 65536, 384, 0, False),    # the decode workload's local top-n
    (6, 140000, 384, 0, True),       # few long rows (clusters), S above 2**17
    (12, 20001, 256, 3, True),       # unaligned rows
    (10, 3000, 2048, 0, False),      # n above the row length: zero words after
])
def test_topk_pack_matches_pack_of_topk(rows, S, n, ld_pad, ends):
    """satk_dcp_topk_pack is dcp_pack(topk_rows(x, n)): every word and plane
    word against the oracle's composition, on every row path (warp, CTA,
    cluster), aligned and unaligned rows, row ends, NaN, ties, local ids at
    and above 2**16 and 2**17."""
    from sparse_attention_indexer_radix_gb300 import inputs
    x, _ = inputs.prefill(rows=rows, cols=S, seed=S + n, causal=False, dtype=torch.bfloat16)
    bits = _bits(x).copy()
    bits[1, ::3] = 0x7FC0                          # NaN columns
    bits[2, : S // 2] = 0x3F80                     # ties at 1.0
    if S > (1 << 17):
        bits[3, (1 << 17) - 5:(1 << 17) + 5] = 0x4300   # 128.0 around 2**17
    re = None
    if ends:
        g = torch.Generator().manual_seed(S)
        re = torch.randint(0, S + 10, (rows,), generator=g, dtype=torch.int32)
        re[0] = S
        re[4] = n // 2 if rows > 4 else re[4]
    host = np.zeros((rows, S + ld_pad), dtype=np.uint16)
    host[:, :S] = bits
    buf = torch.from_numpy(host.view(np.int16)).view(torch.bfloat16).to(DEV)
    got, guard = guarded((rows, n + n // 32))
    satk.dcp_topk_pack(buf[:, :S], n, row_ends=None if re is None else re.to(DEV), out=got)
    guard("topk_pack out")
    rn = None if re is None else re.numpy()
    local = oracle.topk_rows(bits, n, row_ends=rn)
    want = oracle.dcp_pack(bits, local, row_ends=rn)
    _assert_equal(got.cpu().numpy(), want, f"topk_pack rows={rows} S={S} n={n}")
