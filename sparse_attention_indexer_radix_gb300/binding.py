"""Thin ctypes binding of libsatk.so (include/satk.h).

Argument marshalling only: every function checks dtypes and shapes of the
torch tensors it is handed, passes their device pointers, sizes and strides
to the C entry point of the same name on the current CUDA stream, and raises
on a non-zero return.  No computation happens here and there is no fallback:
without the compiled library every call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsatk.so")

SATK_F32, SATK_BF16 = 0, 1
SATK_PAIRS_F32, SATK_PACKED_BF16 = 0, 1
STATUS_SLOTS_EXCEEDED = 1
STATUS_DUPLICATE_KEYS = 2
STATUS_BAD_REQUEST = 4
TOPK_MAX_K = 4096
MERGE_MAX_CANDIDATES = 32768

EXPORTS = ("satk_topk_rows", "satk_dcp_pack", "satk_dcp_merge_select",
           "satk_dcp_rescue_select", "satk_rescue_recv_words", "satk_status_string",
           "satk_dcp_emit_rows", "satk_topk_rows_sorted", "topk_rows", "topk_rows_sorted",
           "dcp_pack", "dcp_merge_select", "dcp_rescue_select", "dcp_emit_rows",
           "satk_dcp_topk_pack", "dcp_topk_pack", "satk_debug_flags")

_lock = threading.Lock()
_lib = None


class SatkError(RuntimeError):
    pass


def load(path: str) -> ctypes.CDLL:
    """Loads a build of the library at `path` and declares the signatures of
    its entry points (include/satk.h)."""
    if not os.path.exists(path):
        raise SatkError(f"{path} is missing: build it with "
                        "`python -m sparse_attention_indexer_radix_gb300.build`")
    L = ctypes.CDLL(path)
    vp, i32, i64, c_int = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
    sigs = {
        "satk_topk_rows": [vp, c_int, i64, i64, i64, vp, i32, vp, i64, vp],
        "satk_topk_rows_sorted": [vp, c_int, i64, i64, i64, vp, i32, vp, i64, vp],
        "satk_dcp_pack": [vp, i64, i64, i64, vp, i64, i32, vp, vp, vp],
        "satk_dcp_topk_pack": [vp, i64, i64, i64, vp, i32, vp, vp],
        "satk_dcp_merge_select": [vp, c_int, i32, i64, i32, i32, vp, i64, vp, vp, vp],
        "satk_dcp_rescue_select": [vp, i32, i64, i32, i32, vp, i64, i64, vp, vp, vp, vp,
                                   i64, vp, vp],
        "satk_dcp_emit_rows": [vp, i64, i32, i64, i32, i32, vp, vp, i64, i64, i32, i32,
                               i64, vp, i64, vp, vp, vp],
    }
    for name, args in sigs.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = c_int
    L.satk_rescue_recv_words.argtypes = [i64, i32, i32]
    L.satk_rescue_recv_words.restype = ctypes.c_size_t
    L.satk_status_string.argtypes = [c_int]
    L.satk_status_string.restype = ctypes.c_char_p
    L.satk_debug_flags.argtypes = [c_int]
    L.satk_debug_flags.restype = ctypes.c_uint
    return L


_routed = threading.local()


def lib() -> ctypes.CDLL:
    """The library the calls of this module go to: libsatk.so, loaded on
    first use (raises if it has not been built), or the one `routed_to`
    selects for the current thread."""
    global _lib
    r = getattr(_routed, "lib", None)
    if r is not None:
        return r
    with _lock:
        if _lib is None:
            _lib = load(LIB_PATH)
    return _lib


@contextlib.contextmanager
def routed_to(L: ctypes.CDLL):
    """Within the block, this thread's calls go to the library L (another
    build of the same sources, e.g. the bounds-checking debug build)."""
    prev = getattr(_routed, "lib", None)
    _routed.lib = L
    try:
        yield L
    finally:
        _routed.lib = prev


# Stands in for the data pointer of a zero-size tensor (torch gives 0) in a
# call whose batch is empty: the entry points check it is non-null and
# aligned, then return before any launch, so it is never dereferenced.
_EMPTY_BATCH_PTR = 256


def _ptr(t, empty_batch: bool = False):
    if t is None:
        return None
    if empty_batch and t.data_ptr() == 0:
        return ctypes.c_void_p(_EMPTY_BATCH_PTR)
    return ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(rc: int, name: str):
    if rc != 0:
        msg = lib().satk_status_string(rc).decode()
        raise SatkError(f"{name} returned {rc}: {msg}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise SatkError("every tensor must live on a CUDA device")


def _rowmajor_2d(t, name):
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise SatkError(f"{name} must be 2-D with unit column stride, got "
                        f"{tuple(t.shape)} {t.stride()}")


def topk_rows(logits: torch.Tensor, k: int, row_ends: torch.Tensor | None = None,
              out: torch.Tensor | None = None, *, sorted: bool = False) -> torch.Tensor:
    """Exact top-k column ids of each row of ``logits`` ([rows, cols] float32
    or bfloat16, any row stride).  ``out`` (int32 [rows, >= k], any row
    stride) receives the ids in columns [0, k); columns past k are never
    written.  ``sorted`` orders them by descending score, ties by ascending
    column (satk_topk_rows_sorted).  Returns ``out`` (allocated [rows, k]
    when not given)."""
    _need_cuda(logits, row_ends, out)
    _rowmajor_2d(logits, "logits")
    if logits.dtype == torch.float32:
        dt = SATK_F32
    elif logits.dtype == torch.bfloat16:
        dt = SATK_BF16
    else:
        raise SatkError(f"logits must be float32 or bfloat16, got {logits.dtype}")
    rows, cols = logits.shape
    if out is None:
        out = torch.empty((rows, k), dtype=torch.int32, device=logits.device)
    _rowmajor_2d(out, "out")
    if out.dtype != torch.int32 or out.shape[0] != rows or out.shape[1] < k:
        raise SatkError(f"out must be int32 [{rows}, >= {k}]")
    if row_ends is not None and (row_ends.dtype != torch.int32 or not row_ends.is_contiguous()
                                 or row_ends.numel() < rows):
        raise SatkError("row_ends must be contiguous int32 [rows]")
    ld = logits.stride(0) if rows > 1 else max(cols, 1)
    ld_out = out.stride(0) if rows > 1 else out.shape[1]
    f = lib().satk_topk_rows_sorted if sorted else lib().satk_topk_rows
    e = rows == 0
    rc = f(_ptr(logits, e), dt, rows, cols, ld, _ptr(row_ends, e), k, _ptr(out, e), ld_out,
           _stream(logits.device))
    _check(rc, "satk_topk_rows_sorted" if sorted else "satk_topk_rows")
    return out


def packed_row_words(n: int) -> int:
    return n + n // 32


def rescue_slots(k: int, n: int) -> int:
    return (k - 1) // n


def rescue_recv_words(T: int, n: int, k: int) -> int:
    return int(lib().satk_rescue_recv_words(T, n, k))


def dcp_pack(logits: torch.Tensor, local_idx: torch.Tensor,
             row_ends: torch.Tensor | None = None,
             out: torch.Tensor | None = None) -> torch.Tensor:
    """Pack a local top-n (``local_idx`` int32 [rows, n], -1 padded) of the
    bf16 ``logits`` [rows, S] into B' rows ``out`` (int32 [rows, n + n/32],
    contiguous)."""
    _need_cuda(logits, local_idx, row_ends, out)
    _rowmajor_2d(logits, "logits")
    _rowmajor_2d(local_idx, "local_idx")
    if logits.dtype != torch.bfloat16 or local_idx.dtype != torch.int32:
        raise SatkError("dcp_pack takes bfloat16 logits and int32 local_idx")
    rows, S = logits.shape
    n = local_idx.shape[1]
    if out is None:
        out = torch.empty((rows, packed_row_words(n)), dtype=torch.int32, device=logits.device)
    if out.dtype != torch.int32 or not out.is_contiguous() or \
            out.numel() != rows * packed_row_words(n):
        raise SatkError(f"out must be contiguous int32 [{rows}, {packed_row_words(n)}]")
    ld = logits.stride(0) if rows > 1 else max(S, 1)
    ld_idx = local_idx.stride(0) if rows > 1 else n
    e = rows == 0
    rc = lib().satk_dcp_pack(_ptr(logits, e), rows, S, ld, _ptr(local_idx, e), ld_idx, n,
                             _ptr(row_ends, e), _ptr(out, e), _stream(logits.device))
    _check(rc, "satk_dcp_pack")
    return out


def dcp_topk_pack(logits: torch.Tensor, n: int, row_ends: torch.Tensor | None = None,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """The local top-n of each bf16 row of ``logits`` [rows, S] written
    straight as B' rows ``out`` (int32 [rows, n + n/32], contiguous): what
    dcp_pack makes of topk_rows(logits, n)."""
    _need_cuda(logits, row_ends, out)
    _rowmajor_2d(logits, "logits")
    if logits.dtype != torch.bfloat16:
        raise SatkError("dcp_topk_pack takes bfloat16 logits")
    rows, S = logits.shape
    if out is None:
        out = torch.empty((rows, packed_row_words(n)), dtype=torch.int32, device=logits.device)
    if out.dtype != torch.int32 or not out.is_contiguous() or \
            out.numel() != rows * packed_row_words(n):
        raise SatkError(f"out must be contiguous int32 [{rows}, {packed_row_words(n)}]")
    if row_ends is not None and (row_ends.dtype != torch.int32 or not row_ends.is_contiguous()):
        raise SatkError("row_ends must be contiguous int32")
    ld = logits.stride(0) if rows > 1 else max(S, 1)
    e = rows == 0
    rc = lib().satk_dcp_topk_pack(_ptr(logits, e), rows, S, ld, _ptr(row_ends, e), n,
                                  _ptr(out, e), _stream(logits.device))
    _check(rc, "satk_dcp_topk_pack")
    return out


def dcp_merge_select(cand: torch.Tensor, k: int, *, packed: bool,
                     ids_out: torch.Tensor | None = None,
                     sat_word: torch.Tensor | None = None,
                     status: torch.Tensor | None = None) -> torch.Tensor:
    """Top-k merge over a rank-major candidate buffer read in place.

    packed=False: ``cand`` is [W, T, n, 2] int32 (float32 score bits, global
    id).  packed=True: ``cand`` is int32 [W, T, n + n/32] B' rows; then
    ``sat_word`` (int32 [T]) may receive the saturation words."""
    _need_cuda(cand, ids_out, sat_word, status)
    if cand.dtype != torch.int32 or not cand.is_contiguous():
        raise SatkError("cand must be contiguous int32")
    if packed:
        if cand.dim() != 3:
            raise SatkError("packed cand must be [W, T, n + n/32]")
        W, T, words = cand.shape
        n = words * 32 // 33
        if packed_row_words(n) != words:
            raise SatkError(f"packed rows of {words} words are not n + n/32")
        fmt = SATK_PACKED_BF16
    else:
        if cand.dim() != 4 or cand.shape[3] != 2:
            raise SatkError("pairs cand must be [W, T, n, 2]")
        W, T, n, _ = cand.shape
        fmt = SATK_PAIRS_F32
    if ids_out is None:
        ids_out = torch.empty((T, k), dtype=torch.int32, device=cand.device)
    _rowmajor_2d(ids_out, "ids_out")
    if ids_out.dtype != torch.int32 or ids_out.shape[0] != T or ids_out.shape[1] < k:
        raise SatkError(f"ids_out must be int32 [{T}, >= {k}]")
    for name, t in (("sat_word", sat_word), ("status", status)):
        if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
            raise SatkError(f"{name} must be contiguous int32")
    if sat_word is not None and sat_word.numel() < T:
        raise SatkError("sat_word must hold T words")
    ld_out = ids_out.stride(0) if T > 1 else ids_out.shape[1]
    e = T == 0
    rc = lib().satk_dcp_merge_select(_ptr(cand, e), fmt, W, T, n, k, _ptr(ids_out, e), ld_out,
                                     _ptr(sat_word, e), _ptr(status), _stream(cand.device))
    _check(rc, "satk_dcp_merge_select")
    return ids_out


def dcp_rescue_select(packed: torch.Tensor, logits: torch.Tensor, sat_word: torch.Tensor,
                      ids_out: torch.Tensor, k: int, *, recv: torch.Tensor | None = None,
                      row_ends: torch.Tensor | None = None,
                      status: torch.Tensor | None = None) -> torch.Tensor:
    """Second round of the packed merge: pushes of the saturated ranks into
    ``recv`` and the re-select of the saturated rows of ``ids_out`` (in
    place).  ``logits`` is bf16 [W, T, S] (unit column stride, rows at a
    common stride); ``row_ends`` int32 [W, T].  Returns ``recv``."""
    _need_cuda(packed, logits, sat_word, ids_out, recv, row_ends, status)
    if packed.dtype != torch.int32 or packed.dim() != 3 or not packed.is_contiguous():
        raise SatkError("packed must be contiguous int32 [W, T, n + n/32]")
    W, T, words = packed.shape
    n = words * 32 // 33
    if logits.dtype != torch.bfloat16 or logits.dim() != 3 or tuple(logits.shape[:2]) != (W, T):
        raise SatkError(f"logits must be bfloat16 [{W}, {T}, S]")
    S = logits.shape[2]
    if S > 1 and logits.stride(2) != 1:
        raise SatkError("logits rows need unit column stride")
    ld = logits.stride(1) if T > 1 else (logits.stride(0) if W > 1 else max(S, 1))
    if W > 1 and T > 1 and logits.stride(0) != ld * T:
        raise SatkError("logits rows must sit at one common stride (rank-major)")
    words_needed = rescue_recv_words(T, n, k)
    if recv is None:
        recv = torch.zeros(max(words_needed, 1), dtype=torch.int32, device=packed.device)
    if recv.dtype != torch.int32 or not recv.is_contiguous() or recv.numel() < words_needed:
        raise SatkError(f"recv must be contiguous int32 with >= {words_needed} words")
    _rowmajor_2d(ids_out, "ids_out")
    ld_out = ids_out.stride(0) if T > 1 else ids_out.shape[1]
    e = T == 0
    rc = lib().satk_dcp_rescue_select(_ptr(packed, e), W, T, n, k, _ptr(logits, e), S, ld,
                                      _ptr(row_ends, e), _ptr(sat_word, e), _ptr(recv, e),
                                      _ptr(ids_out, e), ld_out, _ptr(status),
                                      _stream(packed.device))
    _check(rc, "satk_dcp_rescue_select")
    return recv


def dcp_emit_rows(ids: torch.Tensor, W: int, dcp_rank: int, req_id: torch.Tensor,
                  block_table: torch.Tensor, block_size: int, stride_rows: int, *,
                  k: int | None = None, max_blocks: int | None = None,
                  rows_out: torch.Tensor | None = None,
                  valid_out: torch.Tensor | None = None,
                  status: torch.Tensor | None = None):
    """This rank's physical KV rows of the selected global ids ``ids``
    ([T, >= k] int32, as a merge writes them): ``block_table`` is int32
    [R, width] (unit column stride; ``max_blocks`` defaults to its width),
    ``req_id`` int32 [T].  Returns (rows_out [T, >= k] int32, valid_out [T]
    int32)."""
    _need_cuda(ids, req_id, block_table, rows_out, valid_out, status)
    _rowmajor_2d(ids, "ids")
    _rowmajor_2d(block_table, "block_table")
    if ids.dtype != torch.int32 or req_id.dtype != torch.int32 or block_table.dtype != torch.int32:
        raise SatkError("ids, req_id and block_table must be int32")
    T = ids.shape[0]
    k = ids.shape[1] if k is None else k
    if not req_id.is_contiguous() or req_id.numel() < T:
        raise SatkError("req_id must be contiguous int32 with T entries")
    R, width = block_table.shape
    max_blocks = width if max_blocks is None else max_blocks
    if rows_out is None:
        rows_out = torch.empty((T, k), dtype=torch.int32, device=ids.device)
    if valid_out is None:
        valid_out = torch.empty(T, dtype=torch.int32, device=ids.device)
    _rowmajor_2d(rows_out, "rows_out")
    if rows_out.dtype != torch.int32 or rows_out.shape[0] != T or rows_out.shape[1] < k:
        raise SatkError(f"rows_out must be int32 [{T}, >= {k}]")
    if valid_out.dtype != torch.int32 or not valid_out.is_contiguous() or valid_out.numel() < T:
        raise SatkError("valid_out must be contiguous int32 with T entries")
    ld_ids = ids.stride(0) if T > 1 else ids.shape[1]
    ld_rows = rows_out.stride(0) if T > 1 else rows_out.shape[1]
    ld_table = block_table.stride(0) if R > 1 else max(width, 1)
    e = T == 0
    rc = lib().satk_dcp_emit_rows(_ptr(ids, e), T, k, ld_ids, W, dcp_rank, _ptr(req_id, e),
                                  _ptr(block_table, e), R, ld_table, max_blocks, block_size,
                                  stride_rows, _ptr(rows_out, e), ld_rows, _ptr(valid_out, e),
                                  _ptr(status), _stream(ids.device))
    _check(rc, "satk_dcp_emit_rows")
    return rows_out, valid_out
