/*
 * satk_oracle.c -- plain, slow CPU oracle for the exact per-row top-K path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file: only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm use it.  It shares no code,
 * header, table or helper with the CUDA library under
 * sparse_attention_indexer_radix_gb300/csrc; the two meet only through the
 * seeded input generators.
 *
 * Sources (cited by page title and section):
 *  [P1] vLLM PR #65178 "DCP top-k merge reads the rank-major all-gather
 *       buffer in place" -- Overview (the [W, R, K, 2] rank-major layout and
 *       the (score, global_id) pairs), Validation (fp64 reference over all
 *       candidates).
 *  [P2] vLLM API page "vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels"
 *       -- module docstring (interleave-1 ownership, the B' word, exactness,
 *       saturation and rescue), DCPTopkPackKernel, DCPTopkSelectKernel,
 *       DCPTopkRescueKernel, push_local_topk (inside DCPTopkSelectKernel),
 *       _decode_key, _ord16, _make_radix_select, assert_packed_merge_contract.
 *  [P3] vLLM PR #57206 "Use DeepSelect for eligible sparse-indexer prefill
 *       chunks" -- Purpose (causal per-row end bounds, preallocated output),
 *       Test Plan (short rows, -1 tails, untouched padding).
 *
 * Every function below is either the plain definition (a full sort of the
 * row, then a rule to lay the chosen set out) or, for the packed decode
 * merge and its rescue, the steps of [P2] in the page's order.  No blocking,
 * radix passes or fusion.
 *
 * Orders used (readings, stated once here):
 *  - scores rank descending; NaN is dropped; +inf is the top and -inf the
 *    bottom of the ordinary values; -0.0 ranks just below +0.0 ([P2] ranks by
 *    the ordered bf16 bits, which separate the two zeros);
 *  - ties in score break toward the lower id (column for row top-K, global
 *    id for the merges) [P2 DCPTopkSelectKernel docstring];
 *  - row top-K output layout: the chosen ids scoring strictly above the K-th
 *    score in ascending column order, then the chosen ids equal to it in
 *    ascending column order (the order of [P2] push_local_topk's emit pass);
 *    a row with fewer than K valid columns lists them all in ascending
 *    column order; then -1 up to K; columns [K, ld_out) are never written;
 *  - merge output layout: the chosen candidates in ascending flat candidate
 *    order (rank-major, then slot), then -1;
 *  - owned physical rows: in the order of the ids they come from (the owned
 *    subsequence of a merge output row), then -1 up to k.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_F32 0
#define OR_BF16 1
#define OR_LOCAL_LIMIT (1 << 17) /* [P2] module docstring: local ids < 2**17 */

/* ------------------------------------------------------------------------ */
/* worker pool: rows [0, rows) split into contiguous ranges                 */
/* ------------------------------------------------------------------------ */

typedef void (*row_fn)(void *ctx, int64_t row);

typedef struct {
  row_fn fn;
  void *ctx;
  int64_t begin, end;
} span_t;

static void *run_span(void *p) {
  span_t *s = (span_t *)p;
  for (int64_t r = s->begin; r < s->end; ++r) s->fn(s->ctx, r);
  return NULL;
}

int oracle_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n < 1 ? 1 : (int)n;
}

static void for_rows(int64_t rows, int nthreads, row_fn fn, void *ctx) {
  if (nthreads <= 0) nthreads = oracle_default_threads();
  if (nthreads > rows) nthreads = (int)(rows > 0 ? rows : 1);
  if (nthreads <= 1) {
    for (int64_t r = 0; r < rows; ++r) fn(ctx, r);
    return;
  }
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  span_t *sp = (span_t *)malloc(sizeof(span_t) * (size_t)nthreads);
  int64_t per = rows / nthreads, extra = rows % nthreads, at = 0;
  for (int i = 0; i < nthreads; ++i) {
    int64_t len = per + (i < extra ? 1 : 0);
    sp[i].fn = fn;
    sp[i].ctx = ctx;
    sp[i].begin = at;
    sp[i].end = at + len;
    at += len;
    pthread_create(&tid[i], NULL, run_span, &sp[i]);
  }
  for (int i = 0; i < nthreads; ++i) pthread_join(tid[i], NULL);
  free(tid);
  free(sp);
}

/* ------------------------------------------------------------------------ */
/* score order on real values                                                */
/* ------------------------------------------------------------------------ */

static float bf16_value(uint16_t h) {
  /* bf16 is the upper half of an IEEE binary32. */
  uint32_t b = (uint32_t)h << 16;
  float f;
  memcpy(&f, &b, sizeof f);
  return f;
}

/* >0 when a ranks above b, <0 below, 0 same rank.  a, b not NaN. */
static int score_cmp(float a, float b) {
  if (a > b) return 1;
  if (a < b) return -1;
  /* equal as reals: only the two zeros differ, +0 above -0 */
  int sa = signbit(a) ? 1 : 0, sb = signbit(b) ? 1 : 0;
  return sb - sa;
}

typedef struct {
  float score;
  int64_t id;   /* tie-break key (column or global id) */
  int64_t aux;  /* carried along (flat candidate index) */
} item_t;

/* score descending, id ascending */
static int item_cmp(const void *pa, const void *pb) {
  const item_t *a = (const item_t *)pa, *b = (const item_t *)pb;
  int c = score_cmp(a->score, b->score);
  if (c != 0) return -c;
  if (a->id < b->id) return -1;
  if (a->id > b->id) return 1;
  return 0;
}

static int i64_cmp(const void *pa, const void *pb) {
  int64_t a = *(const int64_t *)pa, b = *(const int64_t *)pb;
  return a < b ? -1 : (a > b ? 1 : 0);
}

/* ------------------------------------------------------------------------ */
/* row top-K  [P3 Purpose, Test Plan; P2 push_local_topk emit order]         */
/* ------------------------------------------------------------------------ */

/*
 * Chosen set and layout of one row, shared by the prefill top-K and the
 * rescue push.  vals[0, end) are the row's scores, is_nan marks dropped
 * ones.  Writes n_out column ids into cols_out (capacity k) and returns it.
 */
static int64_t row_topk_layout(const float *vals, const unsigned char *is_nan,
                               int64_t end, int32_t k, int64_t *cols_out,
                               item_t *scratch, int sorted) {
  int64_t n = 0;
  for (int64_t c = 0; c < end; ++c) {
    if (is_nan[c]) continue;
    scratch[n].score = vals[c];
    scratch[n].id = c;
    scratch[n].aux = c;
    ++n;
  }
  /* the plain definition: full sort, score desc, column asc */
  qsort(scratch, (size_t)n, sizeof(item_t), item_cmp);
  if (sorted) { /* score-sorted layout: the first min(n, k) of the sort */
    const int64_t m = n < k ? n : k;
    for (int64_t i = 0; i < m; ++i) cols_out[i] = scratch[i].id;
    return m;
  }
  if (n < k) {
    for (int64_t i = 0; i < n; ++i) cols_out[i] = scratch[i].id;
    qsort(cols_out, (size_t)n, sizeof(int64_t), i64_cmp);
    return n;
  }
  float kth = scratch[k - 1].score;
  int64_t n_gt = 0;
  while (n_gt < k && score_cmp(scratch[n_gt].score, kth) > 0) ++n_gt;
  for (int64_t i = 0; i < k; ++i) cols_out[i] = scratch[i].id;
  /* strictly above the K-th score, by column */
  qsort(cols_out, (size_t)n_gt, sizeof(int64_t), i64_cmp);
  /* equal to it: the sort already holds the lowest columns, by column */
  qsort(cols_out + n_gt, (size_t)(k - n_gt), sizeof(int64_t), i64_cmp);
  return k;
}

typedef struct {
  const void *x;
  int dtype;
  int64_t cols, ld;
  const int32_t *row_ends;
  int32_t k;
  int32_t *out;
  int64_t ld_out;
  int sorted;
} topk_ctx_t;

static void topk_row(void *p, int64_t row) {
  topk_ctx_t *c = (topk_ctx_t *)p;
  int64_t end = c->cols;
  if (c->row_ends) {
    int64_t e = c->row_ends[row];
    end = e < 0 ? 0 : (e > c->cols ? c->cols : e);
  }
  float *vals = (float *)malloc(sizeof(float) * (size_t)(end + 1));
  unsigned char *nan_flag = (unsigned char *)malloc((size_t)(end + 1));
  item_t *scratch = (item_t *)malloc(sizeof(item_t) * (size_t)(end + 1));
  int64_t *sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)(c->k + 1));
  for (int64_t col = 0; col < end; ++col) {
    float v;
    if (c->dtype == OR_F32)
      v = ((const float *)c->x)[row * c->ld + col];
    else
      v = bf16_value(((const uint16_t *)c->x)[row * c->ld + col]);
    vals[col] = v;
    nan_flag[col] = isnan(v) ? 1 : 0;
  }
  int64_t n = row_topk_layout(vals, nan_flag, end, c->k, sel, scratch, c->sorted);
  int32_t *o = c->out + row * c->ld_out;
  for (int64_t i = 0; i < n; ++i) o[i] = (int32_t)sel[i];
  for (int64_t i = n; i < c->k; ++i) o[i] = -1;
  free(vals);
  free(nan_flag);
  free(scratch);
  free(sel);
}

int oracle_topk_rows(const void *x, int dtype, int64_t rows, int64_t cols,
                     int64_t ld, const int32_t *row_ends, int32_t k,
                     int32_t *out, int64_t ld_out, int nthreads) {
  if (!x || !out || rows < 0 || cols < 0 || ld < cols || k < 1 ||
      ld_out < k || (dtype != OR_F32 && dtype != OR_BF16))
    return -1;
  topk_ctx_t c = {x, dtype, cols, ld, row_ends, k, out, ld_out, 0};
  for_rows(rows, nthreads, topk_row, &c);
  return 0;
}

/* The same chosen set in score order: descending score, ties by ascending
 * column (the plain full sort's first min(n_valid, K) entries), then -1. */
int oracle_topk_rows_sorted(const void *x, int dtype, int64_t rows,
                            int64_t cols, int64_t ld, const int32_t *row_ends,
                            int32_t k, int32_t *out, int64_t ld_out,
                            int nthreads) {
  if (!x || !out || rows < 0 || cols < 0 || ld < cols || k < 1 ||
      ld_out < k || (dtype != OR_F32 && dtype != OR_BF16))
    return -1;
  topk_ctx_t c = {x, dtype, cols, ld, row_ends, k, out, ld_out, 1};
  for_rows(rows, nthreads, topk_row, &c);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* ord16 and the B' word  [P2 _ord16, DCPTopkPackKernel, module docstring]   */
/* ------------------------------------------------------------------------ */

/* Order-preserving 16-bit key of a bf16 bit pattern: a negative pattern is
 * bit-inverted, a non-negative one gets its sign bit set. */
static uint32_t ord16_of(uint16_t h) {
  if (h & 0x8000u) return (uint32_t)(~h) & 0xFFFFu;
  return (uint32_t)h | 0x8000u;
}

static int bf16_is_nan(uint16_t h) { return (h & 0x7FFFu) > 0x7F80u; }

typedef struct {
  const uint16_t *logits;
  int64_t S, ld;
  const int32_t *local_idx;
  int64_t ld_idx;
  int32_t n;
  const int32_t *row_ends;
  int32_t *packed;
} pack_ctx_t;

static void pack_row(void *p, int64_t row) {
  pack_ctx_t *c = (pack_ctx_t *)p;
  int64_t words = c->n + c->n / 32;
  int32_t *dst = c->packed + row * words;
  /* the usable bound: min(row_end, S, 2**17) */
  int64_t end = c->S < OR_LOCAL_LIMIT ? c->S : OR_LOCAL_LIMIT;
  if (c->row_ends && (int64_t)c->row_ends[row] < end) end = c->row_ends[row];
  for (int32_t w = 0; w < c->n / 32; ++w) dst[c->n + w] = 0;
  for (int32_t j = 0; j < c->n; ++j) {
    int64_t local = c->local_idx[row * c->ld_idx + j];
    uint32_t word = 0;
    if (local >= 0 && local < end) {
      uint16_t h = c->logits[row * c->ld + local];
      if (!bf16_is_nan(h)) {
        word = (ord16_of(h) << 16) | (0xFFFFu - ((uint32_t)local & 0xFFFFu));
        if (((uint32_t)local >> 16) & 1u)
          dst[c->n + j / 32] = (int32_t)((uint32_t)dst[c->n + j / 32] |
                                         (1u << (j % 32)));
      }
    }
    dst[j] = (int32_t)word;
  }
}

int oracle_dcp_pack(const uint16_t *logits, int64_t rows, int64_t S,
                    int64_t ld, const int32_t *local_idx, int64_t ld_idx,
                    int32_t n, const int32_t *row_ends, int32_t *packed,
                    int nthreads) {
  if (!logits || !local_idx || !packed || rows < 0 || S < 0 || ld < S ||
      n < 32 || n % 32 != 0 || ld_idx < n)
    return -1;
  pack_ctx_t c = {logits, S, ld, local_idx, ld_idx, n, row_ends, packed};
  for_rows(rows, nthreads, pack_row, &c);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* merge select: top-K over (score desc, gid asc), flat-order output         */
/* [P1 Overview; P2 DCPTopkSelectKernel, _make_radix_select]                 */
/* ------------------------------------------------------------------------ */

/*
 * items[0, m) sorted by item_cmp.  Returns how many of the leading items are
 * chosen: all when m < k; the first k when the k-th is strictly above the
 * (k+1)-th; otherwise (the same (score, id) repeats across the cut, which a
 * valid producer never sends) only the items strictly above the k-th, as the
 * select of [P2] leaves such repeats out.  *dup is set in that last case.
 */
static int64_t chosen_prefix(const item_t *items, int64_t m, int32_t k,
                             int *dup) {
  *dup = 0;
  if (m <= k) return m;
  if (item_cmp(&items[k - 1], &items[k]) != 0) return k;
  *dup = 1;
  int64_t i = k - 1;
  while (i > 0 && item_cmp(&items[i - 1], &items[k - 1]) == 0) --i;
  return i;
}

static int aux_cmp(const void *pa, const void *pb) {
  int64_t a = ((const item_t *)pa)->aux, b = ((const item_t *)pb)->aux;
  return a < b ? -1 : (a > b ? 1 : 0);
}

/* Writes the chosen items' ids into out (ascending aux = flat order), -1
 * after, and returns the chosen count.  Reorders items. */
static int64_t emit_flat(item_t *items, int64_t m, int32_t k, int32_t *out,
                         int *dup) {
  int64_t c = chosen_prefix(items, m, k, dup);
  qsort(items, (size_t)c, sizeof(item_t), aux_cmp);
  for (int64_t i = 0; i < c; ++i) out[i] = (int32_t)items[i].id;
  for (int64_t i = c; i < k; ++i) out[i] = -1;
  return c;
}

typedef struct {
  const float *score_gid; /* [W, T, n, 2] of 4-byte elements */
  int32_t W;
  int64_t T;
  int32_t n, k;
  int32_t *ids;
  int64_t ld_out;
} pairs_ctx_t;

static void pairs_row(void *p, int64_t t) {
  pairs_ctx_t *c = (pairs_ctx_t *)p;
  int64_t total = (int64_t)c->W * c->n, m = 0;
  item_t *items = (item_t *)malloc(sizeof(item_t) * (size_t)(total + 1));
  for (int32_t r = 0; r < c->W; ++r)
    for (int32_t j = 0; j < c->n; ++j) {
      const float *e = c->score_gid + (((int64_t)r * c->T + t) * c->n + j) * 2;
      int32_t gid;
      memcpy(&gid, &e[1], sizeof gid);
      if (gid < 0 || isnan(e[0])) continue; /* empty entry (reading) */
      items[m].score = e[0];
      items[m].id = gid;
      items[m].aux = (int64_t)r * c->n + j;
      ++m;
    }
  qsort(items, (size_t)m, sizeof(item_t), item_cmp);
  int dup;
  emit_flat(items, m, c->k, c->ids + t * c->ld_out, &dup);
  free(items);
}

int oracle_merge_pairs(const void *cand, int32_t W, int64_t T, int32_t n,
                       int32_t k, int32_t *ids, int64_t ld_out, int nthreads) {
  if (!cand || !ids || W < 1 || T < 0 || n < 1 || k < 1 || ld_out < k)
    return -1;
  pairs_ctx_t c = {(const float *)cand, W, T, n, k, ids, ld_out};
  for_rows(T, nthreads, pairs_row, &c);
  return 0;
}

/* packed candidates: the B' word decoded per [P2 _decode_key] */
typedef struct {
  uint32_t ord;   /* ord16 of the score */
  int64_t gid;    /* local * W + owner */
  int64_t flat;
} pcand_t;

static int pcand_to_item(const pcand_t *pc, item_t *it) {
  /* rank by ord16 (the page's score order), then gid ascending: carry the
   * ord16 as a float-valued score so item_cmp applies. ord16 < 2**16 is
   * exact in a float. */
  it->score = (float)pc->ord;
  it->id = pc->gid;
  it->aux = pc->flat;
  return 0;
}

static int decode_word(uint32_t word, uint32_t plane, int32_t j, int32_t owner,
                       int32_t W, pcand_t *out, int64_t flat) {
  /* [P2 _decode_key]: only the word 0 is padding.  Any other word is a
   * candidate, a score field of 0 included: it ranks below every other
   * score (the pack never sends one: 0 is the ord16 of a NaN pattern) */
  if (word == 0) return 0;
  uint32_t local = (0xFFFFu - (word & 0xFFFFu)) |
                   (((plane >> (j % 32)) & 1u) << 16);
  out->ord = word >> 16;
  out->gid = (int64_t)local * W + owner;
  out->flat = flat;
  return 1;
}

typedef struct {
  const int32_t *packed; /* [W, T, n + n/32] */
  int32_t W;
  int64_t T;
  int32_t n, k;
  int32_t *ids;
  int64_t ld_out;
  int32_t *sat_word;
  int32_t *row_status;
} packed_ctx_t;

static void packed_row(void *p, int64_t t) {
  packed_ctx_t *c = (packed_ctx_t *)p;
  int64_t words = c->n + c->n / 32, total = (int64_t)c->W * c->n, m = 0;
  item_t *items = (item_t *)malloc(sizeof(item_t) * (size_t)(total + 1));
  for (int32_t r = 0; r < c->W; ++r) {
    const int32_t *row = c->packed + ((int64_t)r * c->T + t) * words;
    for (int32_t j = 0; j < c->n; ++j) {
      pcand_t pc;
      if (decode_word((uint32_t)row[j], (uint32_t)row[c->n + j / 32], j, r,
                      c->W, &pc, (int64_t)r * c->n + j))
        pcand_to_item(&pc, &items[m++]);
    }
  }
  qsort(items, (size_t)m, sizeof(item_t), item_cmp);
  int dup;
  /* tau16: ord16 of the K-th chosen key, 0 when fewer than K chosen */
  uint32_t tau = 0;
  if (chosen_prefix(items, m, c->k, &dup) == c->k)
    tau = (uint32_t)items[c->k - 1].score;
  emit_flat(items, m, c->k, c->ids + t * c->ld_out, &dup);
  int32_t st = dup ? 2 : 0;
  if (c->sat_word) {
    /* rank r saturated iff all its n slots hold a word with ord16 > tau */
    uint32_t mask = 0;
    for (int32_t r = 0; r < c->W; ++r) {
      const int32_t *row = c->packed + ((int64_t)r * c->T + t) * words;
      int full = 1;
      for (int32_t j = 0; j < c->n; ++j) {
        uint32_t w = (uint32_t)row[j];
        if (w == 0 || (w >> 16) <= tau) {
          full = 0;
          break;
        }
      }
      if (full) mask |= 1u << r;
    }
    int32_t slots = (c->k - 1) / c->n;
    if (__builtin_popcount(mask) > slots) {
      mask = 0; /* more saturated ranks than rescue slots: keep round 1 */
      st |= 1;
    }
    c->sat_word[t] = (int32_t)((mask << 16) | tau);
  }
  if (c->row_status) c->row_status[t] = st;
  free(items);
}

int oracle_merge_packed(const int32_t *packed, int32_t W, int64_t T, int32_t n,
                        int32_t k, int32_t *ids, int64_t ld_out,
                        int32_t *sat_word, int32_t *status, int nthreads) {
  if (!packed || !ids || W < 1 || W > 16 || T < 0 || n < 32 || n % 32 ||
      k < 1 || ld_out < k)
    return -1;
  int32_t *row_status = (int32_t *)calloc((size_t)(T + 1), sizeof(int32_t));
  packed_ctx_t c = {packed, W, T, n, k, ids, ld_out, sat_word, row_status};
  for_rows(T, nthreads, packed_row, &c);
  if (status) {
    int32_t s = 0;
    for (int64_t t = 0; t < T; ++t) s |= row_status[t];
    *status |= s;
  }
  free(row_status);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* rescue: push of the saturated ranks, then the second-round select        */
/* [P2 module docstring; DCPTopkSelectKernel push_local_topk;               */
/*  DCPTopkRescueKernel]                                                     */
/* ------------------------------------------------------------------------ */

typedef struct {
  const int32_t *packed;
  int32_t W;
  int64_t T;
  int32_t n, k;
  const uint16_t *logits; /* [W, T, S] rows at stride ld */
  int64_t S, ld;
  const int32_t *row_ends; /* [W, T] or NULL */
  const int32_t *sat_word;
  int32_t *recv; /* [T, slots, k + k/32] */
  int32_t *ids;
  int64_t ld_out;
  int32_t *row_status;
} rescue_ctx_t;

static void rescue_row(void *p, int64_t t) {
  rescue_ctx_t *c = (rescue_ctx_t *)p;
  uint32_t sw = (uint32_t)c->sat_word[t];
  uint32_t mask = sw >> 16, tau = sw & 0xFFFFu;
  if (mask == 0) return; /* round 1 was exact */
  int32_t slots = (c->k - 1) / c->n;
  if (__builtin_popcount(mask) > slots || (mask >> c->W) != 0) {
    c->row_status[t] |= 1; /* outside the contract: leave the row */
    return;
  }
  int64_t rw = c->k + c->k / 32, words = c->n + c->n / 32;
  int32_t owner[16];
  int32_t num_sat = 0;
  /* 1. each saturated rank's local top-min(K, valid), B' layout, slot s */
  for (int32_t r = 0; r < c->W; ++r) {
    if (!((mask >> r) & 1u)) continue;
    int32_t s = num_sat++;
    owner[s] = r;
    const uint16_t *lrow = c->logits + ((int64_t)r * c->T + t) * c->ld;
    int64_t end = c->S < OR_LOCAL_LIMIT ? c->S : OR_LOCAL_LIMIT;
    if (c->row_ends) {
      int64_t e = c->row_ends[(int64_t)r * c->T + t];
      if (e < end) end = e;
    }
    if (end < 0) end = 0;
    float *vals = (float *)malloc(sizeof(float) * (size_t)(end + 1));
    unsigned char *nf = (unsigned char *)malloc((size_t)(end + 1));
    item_t *scratch = (item_t *)malloc(sizeof(item_t) * (size_t)(end + 1));
    int64_t *sel = (int64_t *)malloc(sizeof(int64_t) * (size_t)(c->k + 1));
    for (int64_t col = 0; col < end; ++col) {
      vals[col] = bf16_value(lrow[col]);
      nf[col] = bf16_is_nan(lrow[col]) ? 1 : 0;
    }
    int64_t cnt = row_topk_layout(vals, nf, end, c->k, sel, scratch, 0);
    int32_t *slot = c->recv + (t * slots + s) * rw;
    for (int64_t i = 0; i < rw; ++i) slot[i] = 0;
    for (int64_t i = 0; i < cnt; ++i) {
      uint32_t l = (uint32_t)sel[i];
      slot[i] = (int32_t)((ord16_of(lrow[l]) << 16) | (0xFFFFu - (l & 0xFFFFu)));
      if ((l >> 16) & 1u)
        slot[c->k + i / 32] =
            (int32_t)((uint32_t)slot[c->k + i / 32] | (1u << (i % 32)));
    }
    free(vals);
    free(nf);
    free(scratch);
    free(sel);
  }
  /* 2. candidates: round-1 words of the other ranks at or above tau, then
   *    the pushed lists (slot s owned by the s-th set bit of the mask) */
  int64_t r1 = (int64_t)c->W * c->n, total = r1 + (int64_t)slots * c->k, m = 0;
  item_t *items = (item_t *)malloc(sizeof(item_t) * (size_t)(total + 1));
  for (int32_t r = 0; r < c->W; ++r) {
    if ((mask >> r) & 1u) continue;
    const int32_t *row = c->packed + ((int64_t)r * c->T + t) * words;
    for (int32_t j = 0; j < c->n; ++j) {
      pcand_t pc;
      if (decode_word((uint32_t)row[j], (uint32_t)row[c->n + j / 32], j, r,
                      c->W, &pc, (int64_t)r * c->n + j) &&
          pc.ord >= tau)
        pcand_to_item(&pc, &items[m++]);
    }
  }
  for (int32_t s = 0; s < num_sat; ++s) {
    const int32_t *slot = c->recv + (t * slots + s) * rw;
    for (int32_t j = 0; j < c->k; ++j) {
      pcand_t pc;
      if (decode_word((uint32_t)slot[j], (uint32_t)slot[c->k + j / 32], j,
                      owner[s], c->W, &pc, r1 + (int64_t)s * c->k + j))
        pcand_to_item(&pc, &items[m++]);
    }
  }
  /* 3. the same select as round 1; overwrite the row's ids */
  qsort(items, (size_t)m, sizeof(item_t), item_cmp);
  int dup;
  emit_flat(items, m, c->k, c->ids + t * c->ld_out, &dup);
  if (dup) c->row_status[t] |= 2;
  free(items);
}

int oracle_rescue(const int32_t *packed, int32_t W, int64_t T, int32_t n,
                  int32_t k, const uint16_t *logits, int64_t S, int64_t ld,
                  const int32_t *row_ends, const int32_t *sat_word,
                  int32_t *recv, int32_t *ids, int64_t ld_out,
                  int32_t *status, int nthreads) {
  if (!packed || !logits || !sat_word || !recv || !ids || W < 1 || W > 16 ||
      T < 0 || n < 32 || n % 32 || k < 32 || k % 32 || n >= k ||
      ld_out < k || ld < S)
    return -1;
  int32_t *row_status = (int32_t *)calloc((size_t)(T + 1), sizeof(int32_t));
  rescue_ctx_t c = {packed, W,        T,    n,   k,      logits,
                    S,      ld,       row_ends, sat_word, recv, ids,
                    ld_out, row_status};
  for_rows(T, nthreads, rescue_row, &c);
  if (status) {
    int32_t s = 0;
    for (int64_t t = 0; t < T; ++t) s |= row_status[t];
    *status |= s;
  }
  free(row_status);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* owned physical KV rows of the selected tokens                             */
/* [P2 DCPTopkSelectKernel docstring (emit_rows); dcp_topk_merge_rows        */
/*  docstring (rows_out, valid_out)]                                         */
/* ------------------------------------------------------------------------ */

/*
 * Row t: walk ids[t, 0:k) in order.  An id g >= 0 with g % W == rank is a
 * token of this rank, local index l = g / W, in block b = l / B.  A block
 * b >= max_blocks (past the block table's width) is dropped; otherwise the
 * physical row block_table[req_id[t], b] * stride_rows + l % B, taken modulo
 * 2**32 as a signed 32-bit value (the page computes it in 32-bit integers),
 * is appended to rows_out[t].  Then -1 up to k (columns [k, ld_rows) are
 * never written) and valid_out[t] = the count.  A req_id outside
 * [0, table_rows) appends nothing and sets status bit 4 (reading: the page
 * does not check it).
 */
int oracle_emit_rows(const int32_t *ids, int64_t T, int32_t k, int64_t ld_ids,
                     int32_t W, int32_t rank, const int32_t *req_id,
                     const int32_t *block_table, int64_t table_rows,
                     int64_t ld_table, int32_t max_blocks, int32_t block_size,
                     int64_t stride_rows, int32_t *rows_out, int64_t ld_rows,
                     int32_t *valid_out, int32_t *status) {
  if (!ids || !req_id || !block_table || !rows_out || !valid_out || T < 0 ||
      k < 1 || ld_ids < k || W < 1 || rank < 0 || rank >= W ||
      table_rows < 0 || max_blocks < 0 || ld_table < max_blocks ||
      block_size < 1 || ld_rows < k)
    return -1;
  int32_t st = 0;
  for (int64_t t = 0; t < T; ++t) {
    const int32_t *id = ids + t * ld_ids;
    int32_t *out = rows_out + t * ld_rows;
    const int32_t req = req_id[t];
    int32_t n = 0;
    if (req < 0 || (int64_t)req >= table_rows) {
      st |= 4;
    } else {
      const int32_t *table = block_table + (int64_t)req * ld_table;
      for (int32_t j = 0; j < k; ++j) {
        const int32_t g = id[j];
        if (g < 0 || g % W != rank) continue;
        const int32_t local = g / W;
        const int32_t b = local / block_size;
        if (b >= max_blocks) continue;
        const int64_t phys = (int64_t)table[b] * stride_rows + local % block_size;
        const uint32_t low = (uint32_t)((uint64_t)phys & 0xFFFFFFFFu);
        int32_t v;
        memcpy(&v, &low, sizeof v);
        out[n++] = v;
      }
    }
    for (int32_t j = n; j < k; ++j) out[j] = -1;
    valid_out[t] = n;
  }
  if (status) *status |= st;
  return 0;
}
