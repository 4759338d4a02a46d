"""Exact per-row top-K for a DSA sparse-attention indexer on GB300.

The compute lives in libsatk.so (hand-written sm_103a CUDA kernels behind the
C ABI of include/satk.h); this package only builds it and marshals torch
tensors into it.

    from sparse_attention_indexer_radix_gb300 import topk_rows, dcp_pack, \\
        dcp_topk_pack, dcp_merge_select, dcp_rescue_select, dcp_emit_rows
"""
from .binding import (MERGE_MAX_CANDIDATES, STATUS_BAD_REQUEST, STATUS_DUPLICATE_KEYS,
                      STATUS_SLOTS_EXCEEDED, TOPK_MAX_K, SatkError, dcp_emit_rows,
                      dcp_merge_select, dcp_pack, dcp_rescue_select, dcp_topk_pack,
                      packed_row_words,
                      rescue_recv_words, rescue_slots, topk_rows)

__all__ = ["topk_rows", "dcp_pack", "dcp_topk_pack", "dcp_merge_select", "dcp_rescue_select", "dcp_emit_rows",
           "packed_row_words", "rescue_slots", "rescue_recv_words", "SatkError",
           "STATUS_SLOTS_EXCEEDED", "STATUS_DUPLICATE_KEYS", "STATUS_BAD_REQUEST", "TOPK_MAX_K",
           "MERGE_MAX_CANDIDATES"]
