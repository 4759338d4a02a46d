/*
 * satk.h -- C ABI of libsatk.so: exact per-row top-K for a DSA sparse
 * attention indexer, on one GB300 (sm_103a).
 *
 * Pages cited by title and section:
 *  [P1] vLLM PR #65178 "DCP top-k merge reads the rank-major all-gather
 *       buffer in place": Overview (rank-major [W, R, K, 2] (score,
 *       global_id) buffer read in place), Details (topk in {512,1024,2048}).
 *  [P2] vLLM API page vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels:
 *       module docstring (B' word, exactness, saturation, rescue),
 *       DCPTopkPackKernel, DCPTopkSelectKernel, DCPTopkRescueKernel,
 *       DCPTopkRescueWorkspace, dcp_topk_pack_indices, dcp_topk_select,
 *       _check_exact.
 *  [P3] vLLM PR #57206 "Use DeepSelect for eligible sparse-indexer prefill
 *       chunks": Purpose (causal per-row end bounds, preallocated output),
 *       Test Plan (strided output, untouched padding, -1 tails).
 *
 * Conventions shared by every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  No entry
 *    point allocates, frees or synchronises; each enqueues its kernels on
 *    `stream` (NULL = the legacy default stream) and returns at once.
 *    Inputs must stay unmodified, and outputs untouched by others, until
 *    the stream reaches the call.
 *  - Sizes are element counts; strides (`ld_*`) are in elements.
 *  - Host-side argument checks run before any launch.  A rejected call
 *    launches nothing and returns a negative SATK_E* code; there is no
 *    fallback of any kind.  SATK_ECUDA reports a launch failure.
 *  - Scores rank descending with NaN dropped, +-inf ordinary and -0.0 just
 *    below +0.0; ties break toward the lower id.
 *  - `status` (where taken) is a nullable device int32; the kernels OR
 *    SATK_STATUS_* bits into it and never clear it.
 */
#ifndef SATK_H_
#define SATK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without the CUDA headers: the same opaque struct pointer. */
struct CUstream_st;
typedef struct CUstream_st *satk_stream_t;

enum satk_dtype { SATK_F32 = 0, SATK_BF16 = 1 };
enum satk_format { SATK_PAIRS_F32 = 0, SATK_PACKED_BF16 = 1 };

enum satk_rc {
  SATK_OK = 0,
  SATK_EINVAL = -1,       /* a pointer, size, stride or alignment is invalid */
  SATK_EUNSUPPORTED = -2, /* valid, but outside the instantiated range       */
  SATK_ECUDA = -3         /* the launch itself failed                         */
};

/* device status bits */
#define SATK_STATUS_SLOTS_EXCEEDED 1 /* more saturated ranks than rescue slots:
                                        the row keeps its round-1 ids [P2
                                        DCPTopkSelectKernel] */
#define SATK_STATUS_DUPLICATE_KEYS 2 /* a repeated (score, id) candidate sat
                                        on the cut: fewer than K ids kept   */
#define SATK_STATUS_BAD_REQUEST 4    /* satk_dcp_emit_rows: a req_id outside
                                        the block table; that row emits
                                        nothing                             */

/* Largest K of satk_topk_rows and of the rescue push. */
#define SATK_TOPK_MAX_K 4096
/* Largest W * n of the merges, and of W * n + ((k-1)/n) * k in the rescue. */
#define SATK_MERGE_MAX_CANDIDATES 32768
/* Local ids of the packed format are below 2**17 [P2 module docstring]. */
#define SATK_LOCAL_INDEX_LIMIT (1 << 17)

/*
 * satk_topk_rows -- exact top-k of each row of a logits matrix [P3 Purpose].
 *
 * logits : [rows, ld_logits] of `dtype` (SATK_F32 float, SATK_BF16 raw
 *          bfloat16); row i's candidates are columns [0, end_i), end_i =
 *          clamp(row_ends[i], 0, cols), or cols when row_ends is NULL.
 *          Columns >= end_i are never read.
 * k      : 1..SATK_TOPK_MAX_K.
 * out    : int32 [rows, ld_out], ld_out >= k.  Row i receives the column
 *          ids of its k best scores: first those strictly above the k-th
 *          score, ascending, then those equal to it (the lowest columns of
 *          the tie), ascending; a row with fewer than k non-NaN candidates
 *          lists them all in ascending order, then -1.  Columns [k, ld_out)
 *          are never written.
 * Errors : SATK_EINVAL for NULL logits/out, rows < 0, cols < 0,
 *          ld_logits < cols, k outside 1..SATK_TOPK_MAX_K, ld_out < k,
 *          cols >= 2**31, or an unknown dtype.
 */
int satk_topk_rows(const void *logits, int dtype, int64_t rows, int64_t cols,
                   int64_t ld_logits, const int32_t *row_ends, int32_t k,
                   int32_t *out, int64_t ld_out, satk_stream_t stream);

/*
 * satk_topk_rows_sorted -- satk_topk_rows with the chosen ids in score
 * order: descending score, ties by ascending column (a score-sorted output
 * option; the pages' selectors never sort, they emit in an order fixed by
 * their thread layout [P2 DCPTopkSelectKernel]).  The chosen set, the -1
 * tail, the untouched columns
 * [k, ld_out), the arguments and the errors are those of satk_topk_rows.
 * Slower: every row takes one CTA and a shared-memory sort of the k ids.
 */
int satk_topk_rows_sorted(const void *logits, int dtype, int64_t rows,
                          int64_t cols, int64_t ld_logits,
                          const int32_t *row_ends, int32_t k, int32_t *out,
                          int64_t ld_out, satk_stream_t stream);

/*
 * satk_dcp_pack -- pack a local top-n into B' rows [P2 DCPTopkPackKernel,
 * dcp_topk_pack_indices].
 *
 * logits_bf16 : [rows, ld_logits] raw bfloat16 scores, S valid columns.
 * local_idx   : int32 [rows, ld_idx], slots [0, n) of each row; -1 pads.
 * n           : a positive multiple of 32.
 * row_ends    : nullable int32 [rows].
 * packed      : int32 [rows, n + n/32], contiguous.  Slot j holds
 *               (ord16(score) << 16) | (0xFFFF - (local & 0xFFFF)), or 0
 *               when local is outside [0, min(row_end, S, 2**17)) or its
 *               score is NaN; word n + j/32 holds bit (local >> 16) & 1 at
 *               bit j % 32.  ord16 flips a negative bf16 pattern and sets
 *               the sign bit of a non-negative one [P2 _ord16].
 * Errors      : SATK_EINVAL for NULL pointers, rows < 0, S < 0,
 *               ld_logits < S, n not a positive multiple of 32, ld_idx < n.
 */
int satk_dcp_pack(const uint16_t *logits_bf16, int64_t rows, int64_t S,
                  int64_t ld_logits, const int32_t *local_idx, int64_t ld_idx,
                  int32_t n, const int32_t *row_ends, int32_t *packed,
                  satk_stream_t stream);

/*
 * satk_dcp_topk_pack -- each bf16 row's local top-n written straight as a B'
 * row: the result of satk_dcp_pack applied to the ids satk_topk_rows(logits,
 * n) returns, in one pass over the logits and without the ids or the
 * gathered re-read of the scores [P2 DCPTopkPackKernel, dcp_topk_pack_indices;
 * P3 Purpose for the row top-K].
 *
 * logits_bf16 : [rows, ld_logits] raw bfloat16, S valid columns; row i's
 *               candidates are columns [0, min(row_ends[i], S)) (NULL row_ends:
 *               S).  Columns >= end are never read.
 * n           : a positive multiple of 32, at most SATK_TOPK_MAX_K.
 * packed      : int32 [rows, n + n/32], contiguous.  Slot j holds the B' word
 *               of the j-th id of the row's top-n layout (satk_topk_rows: the
 *               ids above the n-th score ascending, then its ties), or 0 past
 *               the last valid column or for a column >= 2**17; word n + j/32
 *               holds that column's bit 16 at bit j % 32.
 * Errors      : SATK_EINVAL for NULL pointers, rows < 0, S < 0, ld_logits < S,
 *               n not a positive multiple of 32 or above SATK_TOPK_MAX_K,
 *               S >= 2**31.
 */
int satk_dcp_topk_pack(const uint16_t *logits_bf16, int64_t rows, int64_t S,
                       int64_t ld_logits, const int32_t *row_ends, int32_t n,
                       int32_t *packed, satk_stream_t stream);

/*
 * satk_dcp_merge_select -- top-k over a rank-major candidate buffer read in
 * place [P1 Overview; P2 DCPTopkSelectKernel].
 *
 * cand   : SATK_PAIRS_F32: [W, T, n, 2] 4-byte elements (float score,
 *          int32 global id); an entry with id < 0 or a NaN score is empty.
 *          SATK_PACKED_BF16: int32 [W, T, n + n/32] B' rows; global id
 *          local * W + r for rank r, 0 words empty.
 *          Both contiguous; the pairs buffer 16-byte aligned.
 * W, n   : ranks and candidates per rank; W * n <=
 *          SATK_MERGE_MAX_CANDIDATES; packed needs W <= 16 and n % 32 == 0;
 *          pairs needs n % 32 == 0.
 * k      : 1..W*n is useful; any k >= 1 is accepted.  The chosen set is
 *          the k best under (score desc, global id asc); fewer than k
 *          non-empty candidates keep them all.
 * ids_out: int32 [T, ld_out], ld_out >= k: the chosen global ids in
 *          ascending flat candidate order (rank-major, then slot), then -1.
 * sat_word: packed only (nullable): int32 [T], (mask << 16) | tau16 with
 *          tau16 the ord16 of the k-th chosen candidate (0 when fewer than
 *          k were chosen) and bit r of mask set iff all n slots of rank r
 *          hold words with ord16 > tau16; a mask with more than (k-1)/n
 *          bits is cleared and SATK_STATUS_SLOTS_EXCEEDED raised
 *          [P2 DCPTopkSelectKernel docstring].
 * Errors : SATK_EINVAL for NULL cand/ids_out, W < 1, T < 0, n < 1, k < 1,
 *          ld_out < k, an unknown format, a shape rule above, a pairs
 *          buffer not 16-byte aligned, or a non-NULL sat_word with the
 *          pairs format; SATK_EUNSUPPORTED when W * n exceeds
 *          SATK_MERGE_MAX_CANDIDATES.
 */
int satk_dcp_merge_select(const void *cand, int format, int32_t W, int64_t T,
                          int32_t n, int32_t k, int32_t *ids_out,
                          int64_t ld_out, int32_t *sat_word, int32_t *status,
                          satk_stream_t stream);

/*
 * satk_dcp_rescue_select -- second round of the packed merge for the rows
 * whose sat_word mask is non-zero [P2 module docstring, DCPTopkRescueKernel,
 * push_local_topk].
 *
 * packed      : int32 [W, T, n + n/32], the round-1 input.
 * logits_bf16 : [W, T, ld_logits] raw bfloat16 (rank-major rows of S
 *               valid columns); row_ends nullable int32 [W, T].
 * sat_word    : int32 [T] as written by satk_dcp_merge_select.
 * recv        : int32 scratch of satk_rescue_recv_words(T, n, k) words,
 *               [T, (k-1)/n, k + k/32].  For a row with mask != 0, slot s
 *               receives the s-th saturated rank's local top-min(k, valid)
 *               in B' layout (the same column order as satk_topk_rows), 0
 *               after; other slots and rows are not written.
 * ids_out     : int32 [T, ld_out]; rows with mask != 0 are overwritten with
 *               the top-k of the other ranks' round-1 candidates at or above
 *               tau16 plus the pushed lists (slot s owned by the s-th set
 *               bit of mask), in ascending flat order (round-1 region
 *               rank-major, then slot-major); other rows are untouched.
 * A row whose mask has more than (k-1)/n bits, or a bit at or above W, is
 * left unchanged and raises SATK_STATUS_SLOTS_EXCEEDED.
 * Errors      : SATK_EINVAL for NULL packed/logits/sat_word/recv/ids_out,
 *               W outside 1..16, T < 0, n or k not positive multiples of 32,
 *               n >= k, k > SATK_TOPK_MAX_K, ld_out < k, S < 0,
 *               ld_logits < S; SATK_EUNSUPPORTED when
 *               W * n + ((k-1)/n) * k exceeds SATK_MERGE_MAX_CANDIDATES.
 */
int satk_dcp_rescue_select(const int32_t *packed, int32_t W, int64_t T,
                           int32_t n, int32_t k, const uint16_t *logits_bf16,
                           int64_t S, int64_t ld_logits,
                           const int32_t *row_ends, const int32_t *sat_word,
                           int32_t *recv, int32_t *ids_out, int64_t ld_out,
                           int32_t *status, satk_stream_t stream);

/* Words of the rescue scratch: T * ((k-1)/n) * (k + k/32)
 * [P2 DCPTopkRescueWorkspace].  0 for invalid arguments. */
size_t satk_rescue_recv_words(int64_t T, int32_t n, int32_t k);

/* Scratch words available to satk_dcp_rescue_select_noalloc (8 MiB). */
#define SATK_RESCUE_NOALLOC_MAX_WORDS (2 * 1024 * 1024)

/*
 * satk_dcp_rescue_select_noalloc -- satk_dcp_rescue_select without the
 * `recv` argument, for callers that cannot allocate device memory (code
 * that only receives pointers to its inputs and outputs, or runs where
 * cudaMalloc may not be called).  The pages have no counterpart: it is a
 * convenience of this library.
 *
 * The pushed lists go to a fixed array inside the library's own device
 * memory, SATK_RESCUE_NOALLOC_MAX_WORDS int32 words on every GPU that loads
 * the library, kept until the process exits.  Nothing is allocated and no
 * allocating routine is called.  All other arguments, results, status bits
 * and errors are those of satk_dcp_rescue_select; in addition a call whose
 * satk_rescue_recv_words(T, n, k) exceeds SATK_RESCUE_NOALLOC_MAX_WORDS is
 * rejected with SATK_EUNSUPPORTED before anything is launched.
 *
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current) and keeps it for the
 *   rest of the process; make that first call before any stream capture.
 *   A failed look-up returns SATK_ECUDA.  Resetting the device after that
 *   (cudaDeviceReset, or anything else that destroys its primary context)
 *   is not supported: the array moves when the library's module is loaded
 *   again, and the kept address would be stale.
 * - Every call on a device uses the same array and leaves its contents
 *   behind.  Nothing in it needs to start at zero: each slot a call reads
 *   is written by that same call first.  Calls that can run at the same
 *   time on the GPU (different streams without ordering) race on it.
 */
int satk_dcp_rescue_select_noalloc(const int32_t *packed, int32_t W, int64_t T,
                                   int32_t n, int32_t k,
                                   const uint16_t *logits_bf16, int64_t S,
                                   int64_t ld_logits, const int32_t *row_ends,
                                   const int32_t *sat_word, int32_t *ids_out,
                                   int64_t ld_out, int32_t *status,
                                   satk_stream_t stream);

/*
 * satk_dcp_emit_rows -- this rank's physical KV rows of the selected tokens
 * [P2 DCPTopkSelectKernel docstring (emit_rows), dcp_topk_merge_rows].
 *
 * ids         : int32 [T, ld_ids], columns [0, k): the selected global ids
 *               of each row (as written by satk_dcp_merge_select or
 *               satk_dcp_rescue_select; -1 entries are skipped).
 * W, dcp_rank : ranks, and this rank (0 <= dcp_rank < W).  A global id g
 *               belongs to rank g % W; its local index is l = g / W.
 * req_id      : int32 [T], the request of each row: its row of block_table.
 * block_table : int32 [table_rows, ld_block_table], physical block ids of
 *               each request; max_blocks (<= ld_block_table) is the table's
 *               width: a token in block b = l / block_size >= max_blocks is
 *               dropped.
 * stride_rows : physical rows per block id.  The row of token l is
 *               block_table[req_id[t], b] * stride_rows + l % block_size,
 *               stored as the low 32 bits (the page computes it in 32-bit
 *               integers).
 * rows_out    : int32 [T, ld_rows_out], ld_rows_out >= k: the rows of this
 *               rank's tokens in the order of their ids, then -1 up to k.
 *               Columns [k, ld_rows_out) are never written.
 * valid_out   : int32 [T], the number of rows emitted.
 * A req_id outside [0, table_rows) emits nothing for its row and raises
 * SATK_STATUS_BAD_REQUEST.
 * Errors      : SATK_EINVAL for NULL ids/req_id/block_table/rows_out/
 *               valid_out, T < 0, k < 1, ld_ids < k, W < 1, dcp_rank outside
 *               [0, W), table_rows < 0, max_blocks < 0,
 *               ld_block_table < max_blocks, block_size < 1,
 *               ld_rows_out < k, T >= 2**31.
 */
int satk_dcp_emit_rows(const int32_t *ids, int64_t T, int32_t k, int64_t ld_ids,
                       int32_t W, int32_t dcp_rank, const int32_t *req_id,
                       const int32_t *block_table, int64_t table_rows,
                       int64_t ld_block_table, int32_t max_blocks,
                       int32_t block_size, int64_t stride_rows,
                       int32_t *rows_out, int64_t ld_rows_out,
                       int32_t *valid_out, int32_t *status,
                       satk_stream_t stream);

/*
 * satk_debug_flags -- the bounds-check bits of the debug build.  A library
 * built with -DSATK_DEBUG (libsatk_debug.so) checks, inside its kernels,
 * every shared-memory list index, output position, histogram bin and
 * scratch index that the code relies on an invariant for; a failed check
 * skips the access and ORs a bit into a device word (1 list index, 2 output
 * position, 4 histogram bin, 8 scratch or plane-word index) instead of
 * trapping.  This call waits for the device, returns the word and, when
 * `clear` is non-zero, zeroes it; 0xffffffff if the device could not be
 * read.  The normal build checks nothing and returns 0.  Not part of the
 * pages' interface: a test aid of this library.
 */
uint32_t satk_debug_flags(int clear);

/* A static, human-readable string for an SATK_* return code. */
const char *satk_status_string(int rc);

/* Short names, the same functions. */
int topk_rows(const void *logits, int dtype, int64_t rows, int64_t cols,
              int64_t ld_logits, const int32_t *row_ends, int32_t k,
              int32_t *out, int64_t ld_out, satk_stream_t stream);
int topk_rows_sorted(const void *logits, int dtype, int64_t rows,
                     int64_t cols, int64_t ld_logits, const int32_t *row_ends,
                     int32_t k, int32_t *out, int64_t ld_out,
                     satk_stream_t stream);
int dcp_pack(const uint16_t *logits_bf16, int64_t rows, int64_t S,
             int64_t ld_logits, const int32_t *local_idx, int64_t ld_idx,
             int32_t n, const int32_t *row_ends, int32_t *packed,
             satk_stream_t stream);
int dcp_topk_pack(const uint16_t *logits_bf16, int64_t rows, int64_t S,
                  int64_t ld_logits, const int32_t *row_ends, int32_t n,
                  int32_t *packed, satk_stream_t stream);
int dcp_merge_select(const void *cand, int format, int32_t W, int64_t T,
                     int32_t n, int32_t k, int32_t *ids_out, int64_t ld_out,
                     int32_t *sat_word, int32_t *status, satk_stream_t stream);
int dcp_rescue_select(const int32_t *packed, int32_t W, int64_t T, int32_t n,
                      int32_t k, const uint16_t *logits_bf16, int64_t S,
                      int64_t ld_logits, const int32_t *row_ends,
                      const int32_t *sat_word, int32_t *recv,
                      int32_t *ids_out, int64_t ld_out, int32_t *status,
                      satk_stream_t stream);
int dcp_emit_rows(const int32_t *ids, int64_t T, int32_t k, int64_t ld_ids,
                  int32_t W, int32_t dcp_rank, const int32_t *req_id,
                  const int32_t *block_table, int64_t table_rows,
                  int64_t ld_block_table, int32_t max_blocks,
                  int32_t block_size, int64_t stride_rows, int32_t *rows_out,
                  int64_t ld_rows_out, int32_t *valid_out, int32_t *status,
                  satk_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SATK_H_ */
