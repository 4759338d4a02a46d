"""CPU oracle for the exact per-row top-K path -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import this package.  The product library never
does, and this package imports nothing from it: the two share no code.

The arithmetic lives in ``satk_oracle.c`` (plain C, full sort per row,
pthreads over rows); this module compiles it with gcc on first use and
wraps it with ctypes over numpy arrays.  Every function mirrors one call of
the C ABI and states which page section it follows (see the C file header).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "satk_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsatk_oracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile the oracle shared library in place (gcc, no CUDA)."""
    stale = (
        force
        or not os.path.exists(_LIB_PATH)
        or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    )
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = [
            "gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread",
            "-o", tmp, _SRC, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, i32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
            lib.oracle_default_threads.restype = ctypes.c_int
            lib.oracle_topk_rows.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp,
                                             i32, vp, i64, ctypes.c_int]
            lib.oracle_dcp_pack.argtypes = [vp, i64, i64, i64, vp, i64, i32, vp,
                                            vp, ctypes.c_int]
            lib.oracle_merge_pairs.argtypes = [vp, i32, i64, i32, i32, vp, i64,
                                               ctypes.c_int]
            lib.oracle_merge_packed.argtypes = [vp, i32, i64, i32, i32, vp, i64,
                                                vp, vp, ctypes.c_int]
            lib.oracle_rescue.argtypes = [vp, i32, i64, i32, i32, vp, i64, i64,
                                          vp, vp, vp, vp, i64, vp, ctypes.c_int]
            lib.oracle_topk_rows_sorted.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp,
                                                    i32, vp, i64, ctypes.c_int]
            lib.oracle_emit_rows.argtypes = [vp, i64, i32, i64, i32, i32, vp, vp, i64,
                                             i64, i32, i32, i64, vp, i64, vp, vp]
            for f in ("oracle_topk_rows", "oracle_dcp_pack", "oracle_merge_pairs",
                      "oracle_merge_packed", "oracle_rescue", "oracle_emit_rows",
                      "oracle_topk_rows_sorted"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: oracle rejected its arguments (rc={rc})")


def topk_rows(x, k, row_ends=None, out=None, ld_out=None, nthreads=0, sorted=False):
    """Exact per-row top-K of ``x`` ([rows, cols] float32, or uint16 holding
    bf16 bits).  Returns (or fills) an int32 [rows, ld_out] array; only
    columns [0, k) of each row are written.  ``sorted``: the same ids in
    descending score order, ties by ascending column."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        dt = F32
    elif x.dtype == np.uint16:
        dt = BF16
    else:
        raise TypeError(f"x must be float32 or uint16 (bf16 bits), got {x.dtype}")
    rows, cols = x.shape
    ld_out = k if ld_out is None else ld_out
    if out is None:
        out = np.full((rows, ld_out), -7, dtype=np.int32)
    assert out.dtype == np.int32 and out.flags.c_contiguous
    re = _c(row_ends, np.int32)
    f = _load().oracle_topk_rows_sorted if sorted else _load().oracle_topk_rows
    rc = f(_ptr(x), dt, rows, cols, cols, _ptr(re), k, _ptr(out), out.shape[1], nthreads)
    _check(rc, "topk_rows")
    return out


def dcp_pack(logits_bits, local_idx, row_ends=None, nthreads=0):
    """Pack a local top-N into B' rows: [rows, n + n/32] int32."""
    lg = _c(logits_bits, np.uint16)
    li = _c(local_idx, np.int32)
    rows, S = lg.shape
    n = li.shape[1]
    out = np.zeros((rows, n + n // 32), dtype=np.int32)
    re = _c(row_ends, np.int32)
    rc = _load().oracle_dcp_pack(_ptr(lg), rows, S, S, _ptr(li), n, n, _ptr(re),
                                 _ptr(out), nthreads)
    _check(rc, "dcp_pack")
    return out


def merge_pairs(cand, k, nthreads=0):
    """Top-K of the rank-major pairs buffer ``cand`` ([W, T, n, 2] of 4-byte
    elements: float32 score bits, int32 gid), flat-order output [T, k]."""
    c = np.ascontiguousarray(cand)
    assert c.itemsize == 4 and c.ndim == 4 and c.shape[3] == 2
    W, T, n, _ = c.shape
    ids = np.full((T, k), -7, dtype=np.int32)
    rc = _load().oracle_merge_pairs(_ptr(c), W, T, n, k, _ptr(ids), k, nthreads)
    _check(rc, "merge_pairs")
    return ids


def merge_packed(packed, k, nthreads=0):
    """Round-1 select over gathered B' rows ([W, T, n + n/32] int32).
    Returns (ids [T, k], sat_word [T], status)."""
    p = _c(packed, np.int32)
    W, T, words = p.shape
    n = words * 32 // 33
    assert n + n // 32 == words
    ids = np.full((T, k), -7, dtype=np.int32)
    sat = np.zeros(T, dtype=np.int32)
    status = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_merge_packed(_ptr(p), W, T, n, k, _ptr(ids), k, _ptr(sat),
                                     _ptr(status), nthreads)
    _check(rc, "merge_packed")
    return ids, sat, int(status[0])


def rescue_slots(k, n):
    return (k - 1) // n


def rescue(packed, k, logits_bits, sat_word, ids, row_ends=None, recv=None,
           nthreads=0):
    """Second round: pushes of the saturated ranks into ``recv`` ([T, slots,
    k + k/32] int32) and the re-select, overwriting the saturated rows of
    ``ids`` in place.  ``logits_bits`` is [W, T, S] uint16 (bf16 bits).
    Returns (ids, recv, status)."""
    p = _c(packed, np.int32)
    W, T, words = p.shape
    n = words * 32 // 33
    lg = _c(logits_bits, np.uint16)
    assert lg.shape[0] == W and lg.shape[1] == T
    S = lg.shape[2]
    slots = rescue_slots(k, n)
    if recv is None:
        recv = np.zeros((T, max(slots, 1), k + k // 32), dtype=np.int32)
    assert recv.dtype == np.int32 and recv.flags.c_contiguous
    assert ids.dtype == np.int32 and ids.flags.c_contiguous
    sw = _c(sat_word, np.int32)
    re = _c(row_ends, np.int32)
    status = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_rescue(_ptr(p), W, T, n, k, _ptr(lg), S, S, _ptr(re),
                               _ptr(sw), _ptr(recv), _ptr(ids), ids.shape[1],
                               _ptr(status), nthreads)
    _check(rc, "rescue")
    return ids, recv, int(status[0])


def emit_rows(ids, W, rank, req_id, block_table, block_size, stride_rows,
              max_blocks=None, ld_rows=None):
    """This rank's physical KV rows of the selected ids ([T, k] int32): the
    owned ids (gid % W == rank) whose block gid // W // block_size is below
    ``max_blocks`` (default: the table's width), mapped through
    ``block_table`` ([R, width] int32) and ``req_id`` ([T] int32).  Returns
    (rows_out [T, ld_rows] int32 with columns [k, ld_rows) left at -7,
    valid_out [T] int32, status)."""
    i = _c(ids, np.int32)
    T, k = i.shape
    rq = _c(req_id, np.int32)
    bt = _c(block_table, np.int32)
    R, width = bt.shape
    max_blocks = width if max_blocks is None else max_blocks
    ld_rows = k if ld_rows is None else ld_rows
    rows = np.full((T, ld_rows), -7, dtype=np.int32)
    valid = np.full(T, -7, dtype=np.int32)
    status = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_emit_rows(_ptr(i), T, k, k, W, rank, _ptr(rq), _ptr(bt), R, width,
                                  max_blocks, block_size, stride_rows, _ptr(rows), ld_rows,
                                  _ptr(valid), _ptr(status))
    _check(rc, "emit_rows")
    return rows, valid, int(status[0])
