// topk_rows_impl.cuh -- the kernels and launch code of satk_topk_rows and
// satk_topk_rows_sorted, templated on the element type and the row
// alignment.  Each (type, alignment) pair is instantiated in a translation
// unit of its own (topk_rows_f32_a32.cu, ...), which keeps the build parallel;
// topk_rows.cu holds the C entry points.
//
// Every path reads each valid column from HBM once: a sampled threshold, a
// filtered collection into a shared-memory list, an exact select on the
// list.  The launch picks the path by shape:
//  - rows of a few thousand columns: one warp per row (satk_warp.cuh);
//  - few long rows: a cluster of 2-8 CTAs per row (satk_cluster.cuh);
//  - otherwise one CTA of 128 or 256 threads per row (satk_rows.cuh).
// The score-sorted variant sorts the chosen ids: on the warp of a short row
// (a bucket sort of the chosen set in registers and shared memory), else
// after the CTA path (a block bitonic sort).
#pragma once

#include <climits>
#include <cmath>

#include "satk_cluster.cuh"
#include "satk_host.hpp"
#include "satk_rows.cuh"
#include "satk_warp.cuh"

namespace satk {
namespace {

// 256 threads per row; rows whose sampled list fits the smaller list with
// room to spare (short_cta_rows_fit) take 128 (more rows resident per SM,
// shorter barriers: short rows are bound by the per-row select, not by the
// stream).
constexpr int kBlock = 256;
constexpr int kShortBlock = 128;
// the widest rows measured faster on 128 threads: fp32 and bf16
template <typename T>
constexpr int short_cols_max() {
  return sizeof(T) == 2 ? 45056 : 24576;
}

__device__ __forceinline__ int row_end_of(const int32_t *row_ends, int64_t row, int cols) {
  if (row_ends == nullptr) return cols;
  const int e = row_ends[row];
  return e < 0 ? 0 : (e > cols ? cols : e);
}

// Where a row's chosen candidates go: put(pos, key, column) for output
// position pos of the row's top-K layout, fill(pos) past the last one;
// start(t, nt) runs once per row, on threads t of nt, before any put.  The
// warp path calls put_entry(pos, list index, key, column).
//  IdOut     -- the column ids, then -1 (satk_topk_rows).
//  PackedOut -- the B' row of satk_dcp_topk_pack: word pos = the key's
//               ord16 (bf16 keys are ord16 << 16) | (0xFFFF - column[15:0]),
//               bit pos % 32 of word K + pos / 32 = column[16]; a column at
//               or above 2**17 packs as 0, and so does every position past
//               the last candidate (vLLM API page
//               vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels,
//               DCPTopkPackKernel).  The plane words are zeroed in start and
//               set with atomic ORs.
struct IdOut {
  int32_t *o;
  int K;
  __device__ __forceinline__ void start(int, int) const {}
  __device__ __forceinline__ void put(int pos, uint32_t, int col) const {
    if (satk_check(pos >= 0 && pos < K, kDbgOut)) o[pos] = col;
  }
  __device__ __forceinline__ void put_entry(int pos, int, uint32_t key, int col) const {
    put(pos, key, col);
  }
  __device__ __forceinline__ void fill(int pos) const {
    if (satk_check(pos >= 0 && pos < K, kDbgOut)) o[pos] = -1;
  }
};
struct PackedOut {
  int32_t *o;
  int K;
  __device__ __forceinline__ void start(int t, int nt) const {
    for (int i = t; i < K / 32; i += nt) o[K + i] = 0;
  }
  __device__ __forceinline__ void put(int pos, uint32_t key, int col) const {
    if (!satk_check(pos >= 0 && pos < K, kDbgOut)) return;
    uint32_t w = 0u;
    if (col < SATK_LOCAL_INDEX_LIMIT) {
      w = (key & 0xffff0000u) | (0xffffu - (static_cast<uint32_t>(col) & 0xffffu));
      if (col >> 16) atomicOr(o + K + pos / 32, 1 << (pos & 31));
    }
    o[pos] = static_cast<int32_t>(w);
  }
  __device__ __forceinline__ void put_entry(int pos, int, uint32_t key, int col) const {
    put(pos, key, col);
  }
  __device__ __forceinline__ void fill(int pos) const {
    if (satk_check(pos >= 0 && pos < K, kDbgOut)) o[pos] = 0;
  }
};

template <typename T, int BLOCK, int SUB, int ALIGN, class Out = IdOut>
__global__ void __launch_bounds__(BLOCK, 1024 / BLOCK) topk_rows_kernel(const T *__restrict__ x, int64_t ld,
                                                          int cols,
                                                          const int32_t *__restrict__ row_ends,
                                                          int K, int32_t *__restrict__ out,
                                                          int64_t ld_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<ListSmem<BLOCK, SUB> *>(smem_raw);
  const int64_t row = blockIdx.x;
  const int end = row_end_of(row_ends, row, cols);
  const Out dst{out + row * ld_out, K};
  dst.start(threadIdx.x, BLOCK);
  zero_hist(sm.sel);
  __syncthreads();
  topk_row<T, BLOCK, SUB, ALIGN>(
      x + row * ld, end, K,
      [&](int pos, int i) {
        if ((unsigned)pos < (unsigned)K) dst.put(pos, sm.key[i], static_cast<int>(sm.val[i]));
      },
      [&](int pos) { dst.fill(pos); }, sm);
}

template <typename T, int BLOCK, int SUB, int ALIGN, class Out = IdOut>
int launch(const T *x, int64_t rows, int cols, int64_t ld, const int32_t *row_ends, int K,
           int32_t *out, int64_t ld_out, cudaStream_t st) {
  auto kern = topk_rows_kernel<T, BLOCK, SUB, ALIGN, Out>;
  const size_t smem = sizeof(ListSmem<BLOCK, SUB>);
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  kern<<<dim3(static_cast<unsigned>(rows)), BLOCK, smem, st>>>(x, ld, cols, row_ends, K, out,
                                                               ld_out);
  return launch_status();
}

// Byte offset of the sorted kernel's composite buffer after the list.
template <int SUB>
__host__ __device__ constexpr size_t sorted_buf_offset() {
  return (sizeof(ListSmem<kBlock, SUB>) + 15) / 16 * 16;
}

// Short rows: one warp per row (satk_warp.cuh), kWarpRowsPerCta rows per
// CTA, seven CTAs per SM (their workspaces fill the shared memory).
template <typename T, int ALIGN, class Out = IdOut>
__global__ void __launch_bounds__(32 * kWarpRowsPerCta, 7)
    topk_rows_warp_kernel(const T *__restrict__ x, int64_t rows, int64_t ld, int cols,
                          const int32_t *__restrict__ row_ends, int K,
                          int32_t *__restrict__ out, int64_t ld_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int warp = warp_id();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpRowsPerCta + warp;
  if (row >= rows) return;  // warp-uniform; the warps never synchronise
  WarpRowSmem &ws = reinterpret_cast<WarpRowSmem *>(smem_raw)[warp];
  for (int i = lane_id(); i < 256; i += 32) ws.hist[i] = 0u;
  const Out dst{out + row * ld_out, K};
  dst.start(lane_id(), 32);
  __syncwarp();
  warp_topk_row<T, ALIGN>(x + row * ld, row_end_of(row_ends, row, cols), K, dst, ws);
}

template <typename T, int ALIGN, class Out = IdOut>
int launch_warp(const T *x, int64_t rows, int cols, int64_t ld, const int32_t *row_ends, int K,
                int32_t *out, int64_t ld_out, cudaStream_t st) {
  auto kern = topk_rows_warp_kernel<T, ALIGN, Out>;
  const size_t smem = sizeof(WarpRowSmem) * kWarpRowsPerCta;
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  const int64_t grid = (rows + kWarpRowsPerCta - 1) / kWarpRowsPerCta;
  kern<<<dim3(static_cast<unsigned>(grid)), 32 * kWarpRowsPerCta, smem, st>>>(
      x, rows, ld, cols, row_ends, K, out, ld_out);
  return launch_status();
}

// Whether a row of `cols` columns keeps its sampled candidate list within
// one warp's kWarpList entries: the expected list K r / mu (r and mu as in
// the sample step) plus four standard deviations (about list / sqrt(r)) of
// the r-th sample order statistic.  Rows that still overflow take the exact
// path, so this only decides speed.
inline bool warp_rows_fit(int cols, int K) {
  if (K > 512 || cols > 65536) return false;
  if (cols <= kWarpList) return true;
  const double mu = static_cast<double>(K) * kWarpSample / cols;
  const double r = std::ceil(mu + 4.0 * std::sqrt(mu) + 4.0);
  const double list = K * r / mu;
  return list + 4.0 * list / std::sqrt(r) <= kWarpList;
}

// Few long rows: a cluster of C CTAs per row (satk_cluster.cuh); the grid
// is rows x C, CTA blockIdx.x % C of the cluster taking slice
// blockIdx.x % C of row blockIdx.x / C.
template <typename T, int BLOCK, int SUB, int ALIGN, int C, class Out = IdOut>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(BLOCK, 1024 / BLOCK)
    topk_rows_cluster_kernel(const T *__restrict__ x, int64_t ld, int cols,
                             const int32_t *__restrict__ row_ends, int K,
                             int32_t *__restrict__ out, int64_t ld_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto &cs = *reinterpret_cast<ClusterSmem<BLOCK, SUB> *>(smem_raw);
  cg::cluster_group cl = cg::this_cluster();
  const int64_t row = blockIdx.x / C;
  const Out dst{out + row * ld_out, K};
  if (cl.block_rank() == 0) dst.start(threadIdx.x, BLOCK);  // before the first cluster barrier
  zero_hist(cs.ls.sel);
  __syncthreads();
  cluster_topk_row<T, BLOCK, SUB, ALIGN, C>(
      cl, x + row * ld, row_end_of(row_ends, row, cols), K,
      [&](int pos, uint32_t key, int col) { dst.put(pos, key, col); },
      [&](int pos) { dst.fill(pos); }, cs);
}

template <typename T, int BLOCK, int SUB, int ALIGN, int C, class Out = IdOut>
int launch_cluster(const T *x, int64_t rows, int cols, int64_t ld, const int32_t *row_ends,
                   int K, int32_t *out, int64_t ld_out, cudaStream_t st) {
  auto kern = topk_rows_cluster_kernel<T, BLOCK, SUB, ALIGN, C, Out>;
  const size_t smem = sizeof(ClusterSmem<BLOCK, SUB>);
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  kern<<<dim3(static_cast<unsigned>(rows * C)), BLOCK, smem, st>>>(x, ld, cols, row_ends, K,
                                                                   out, ld_out);
  return launch_status();
}

// Cluster size for `rows` rows when one CTA per row would not fill one wave
// of resident CTAs (0: no cluster): the smallest of 2, 4, 8 whose clusters
// fill a wave, else 8.  A cluster adds barriers to every step of a row,
// which pays only while SMs would otherwise sit idle, and the fewer CTAs
// share a row the fewer remote reads each barrier round costs (measured on
// the current kernels: 1310 fp32 rows of 400 KB, 2.15 waves, 142.6 us on
// two-CTA clusters against 118.3 us one CTA per row; 256 bf16 rows of 256 KB
// with K = 2048, 0.56 waves, 52.5 us on two-CTA clusters against 114 us on
// eight; four rows of 524288 columns take eight).
template <typename T, int BLOCK, int SUB, int ALIGN>
int cluster_size(int64_t rows, int cols) {
  if (rows > INT32_MAX / 8 || cols < 8 * 2 * ListSmem<BLOCK, SUB>::CAP) return 0;
  // the occupancy query counts the shared memory only once the kernel may
  // take it (above 48 KB)
  auto kern = topk_rows_kernel<T, BLOCK, SUB, ALIGN>;
  if (!allow_smem(kern, sizeof(ListSmem<BLOCK, SUB>))) return 0;
  const int64_t resident =
      resident_ctas(reinterpret_cast<const void *>(kern), BLOCK, sizeof(ListSmem<BLOCK, SUB>));
  if (resident <= 0 || rows >= resident) return 0;
  int c = 8;
  for (int t = 2; t < 8; t *= 2)
    if (rows * t >= resident) {
      c = t;
      break;
    }
  return c;
}

template <typename T, int BLOCK, int SUB, int ALIGN, class Out = IdOut>
int launch_rows_cta(const T *x, int64_t rows, int cols, int64_t ld, const int32_t *row_ends,
                    int K, int32_t *out, int64_t ld_out, cudaStream_t st) {
  switch (cluster_size<T, BLOCK, SUB, ALIGN>(rows, cols)) {
    case 2:
      return launch_cluster<T, BLOCK, SUB, ALIGN, 2, Out>(x, rows, cols, ld, row_ends, K, out,
                                                          ld_out, st);
    case 4:
      return launch_cluster<T, BLOCK, SUB, ALIGN, 4, Out>(x, rows, cols, ld, row_ends, K, out,
                                                          ld_out, st);
    case 8:
      return launch_cluster<T, BLOCK, SUB, ALIGN, 8, Out>(x, rows, cols, ld, row_ends, K, out,
                                                          ld_out, st);
    default:
      return launch<T, BLOCK, SUB, ALIGN, Out>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
  }
}

// Whether rows of `cols` columns take the 128-thread CTA: its list (four
// warps x 512 entries) must hold the sampled list -- K r / mu entries with
// mu = K x samples / cols and r as in the sample step, samples = 128 x
// row_sample<T>() -- plus four standard deviations (about list / sqrt(r))
// within 80 % of its capacity, because a warp segment that overflows sends
// its row to the exact pass, which in a launch of several waves can outlast
// the whole launch.  Measured on 4096 causal fp32 rows at K = 512, 128
// against 256 threads: 18432 columns 97 -> 87 us, 20480 103 -> 93 us;
// at 35840 columns two rows overflowed and the launch took 223 us against
// 134 us.  bf16 rows (16 samples per thread) fit wider rows: 30720 columns
// 101 -> 91 us, 43008 115 -> 108 us.  Rows above short_cols_max<T>() stay
// on 256 threads whatever the estimate.
template <typename T>
inline bool short_cta_rows_fit(int cols, int K) {
  constexpr int CAP = ListSmem<kShortBlock, 512>::CAP;
  if (K > 512 || cols > short_cols_max<T>()) return false;
  if (cols <= CAP) return true;
  const double mu = static_cast<double>(K) * kShortBlock * row_sample<T>() / cols;
  const double r = std::ceil(mu + 4.0 * std::sqrt(mu) + 4.0);
  const double list = K * r / mu;
  return list + 4.0 * list / std::sqrt(r) <= 0.8 * CAP;
}

// The list holds (BLOCK/32) warps x SUB candidates.
template <typename T, int ALIGN, class Out = IdOut>
int launch_rows(const T *x, int64_t rows, int cols, int64_t ld, const int32_t *row_ends, int K,
                int32_t *out, int64_t ld_out, cudaStream_t st) {
  if (warp_rows_fit(cols, K))
    return launch_warp<T, ALIGN, Out>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
  if (short_cta_rows_fit<T>(cols, K)) {
    // above 16384 columns the 128-thread CTA pays through occupancy only: a
    // batch that does not fill one wave of 256-thread CTAs keeps the wider
    // CTA, whose extra threads shorten each row
    bool use_short = cols <= 16384;
    if (!use_short) {
      auto wide = topk_rows_kernel<T, kBlock, 512, ALIGN, Out>;
      const size_t smem = sizeof(ListSmem<kBlock, 512>);
      if (allow_smem(wide, smem)) {
        const int64_t wave = resident_ctas(reinterpret_cast<const void *>(wide), kBlock, smem);
        use_short = wave > 0 && rows >= wave;
      }
    }
    if (use_short)
      return launch<T, kShortBlock, 512, ALIGN, Out>(x, rows, cols, ld, row_ends, K, out,
                                                     ld_out, st);
  }
  if (K <= 1024)
    return launch_rows_cta<T, kBlock, 512, ALIGN, Out>(x, rows, cols, ld, row_ends, K, out,
                                                       ld_out, st);
  return launch_rows_cta<T, kBlock, 1024, ALIGN, Out>(x, rows, cols, ld, row_ends, K, out,
                                                      ld_out, st);
}

// ------------------------------------------------------- score-sorted --

// In-place bitonic sort of P (a power of two) 64-bit values in shared
// memory into descending order.  Every thread of the block takes part.
template <int BLOCK, int P>
__device__ void bitonic_sort_desc(uint64_t *buf) {
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < P / 2; i += BLOCK) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const uint64_t a = buf[lo], b = buf[hi];
        // blocks whose size bit is clear end descending, the others
        // ascending; at size == P every block ends descending
        const bool desc = (lo & size) == 0;
        if (desc ? a < b : a > b) {
          buf[lo] = b;
          buf[hi] = a;
        }
      }
      __syncthreads();
    }
  }
}

// ---- score-sorted on one warp (short rows)
//
// The warp path's ordered emit records, for every output position below
// K, the list index of the entry chosen there (a 16-bit map in the warp's
// histogram words, 0xFFFF where no candidate).  The warp then gathers the
// chosen entries as (key << 32 | ~column) composites into registers --
// entry e * 32 + l in lane l, P = 32 E of them -- after which the list area
// is free for the sort's scratch:
//  - bucket sort (the usual case): bucket b(key) = floor((key - kmin) *
//    512 / (span + 1)) is monotone in the key, so with buckets taken from
//    the highest down an entry's output position is the count of entries
//    in higher buckets plus its rank by composite (key desc, column asc)
//    among its own bucket's entries, counted by a walk over the bucket;
//  - a bitonic network over the registers when a bucket holds more than 32
//    entries (heavy ties).

struct SortMapOut {
  uint16_t *m;
  int K;
  __device__ __forceinline__ void start(int, int) const {}
  __device__ __forceinline__ void put_entry(int pos, int i, uint32_t, int) const {
    if (satk_check(pos >= 0 && pos < K, kDbgOut)) m[pos] = static_cast<uint16_t>(i);
  }
  __device__ __forceinline__ void fill(int pos) const {
    if (satk_check(pos >= 0 && pos < K, kDbgOut)) m[pos] = 0xffffu;
  }
};

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(kFull, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(kFull, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Compare-exchange of registers a (lower index) and b: with desc the
// larger ends in a.
__device__ __forceinline__ void cex(uint64_t &a, uint64_t &b, bool desc) {
  const bool sw = desc ? a < b : a > b;
  const uint64_t x = a;
  a = sw ? b : a;
  b = sw ? x : b;
}

// Bitonic sort, descending, of the 32 E values v (afterwards lane l holds
// entries l E + e).  Pair (i, i + stride) of a block whose size bit is
// clear ends with the larger value first; at size == P every block is such
// a block.  Sizes up to E sort each lane's registers (unrolled); beyond E
// only the loops over the registers are unrolled (a fully unrolled network
// outgrows the instruction cache), and the direction of a pair is the
// lane's.
template <int E>
__device__ __forceinline__ void warp_bitonic_desc(uint64_t (&v)[E]) {
  constexpr int P = 32 * E;
  const int lane = lane_id();
#pragma unroll
  for (int size = 2; size <= E; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((e & stride) == 0) cex(v[e], v[e + stride], ((lane * E + e) & size) == 0);
    }
  }
#pragma unroll 1
  for (int size = 2 * E; size <= P; size <<= 1) {
    const bool desc = ((lane * E) & size) == 0;
#pragma unroll 1
    for (int stride = size >> 1; stride >= E; stride >>= 1) {  // partner lane ^ (stride / E)
      const int m = stride / E;
      const bool keep_max = desc == ((lane & m) == 0);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint64_t o = shfl_xor_u64(v[e], m);
        v[e] = keep_max ? (o > v[e] ? o : v[e]) : (o < v[e] ? o : v[e]);
      }
    }
#pragma unroll
    for (int stride = E / 2; stride > 0; stride >>= 1) {  // partner register e + stride
#pragma unroll
      for (int e = 0; e < E; ++e)
        if ((e & stride) == 0) cex(v[e], v[e + stride], desc);
    }
  }
}

// The bucket sort over NB = 512 buckets: composites c (0: no entry),
// scratch tmp (32 E values), ranked columns to cols[0, n) (the output row),
// hist (NB words) zero on entry.  Returns n, the count of entries, or -1 (nothing written)
// when a bucket holds more than 32 entries.
template <int E>
__device__ int warp_bucket_rank(const uint64_t (&c)[E], uint64_t *tmp, int32_t *cols,
                                uint32_t *hist) {
  constexpr int NB = 512;
  const int lane = lane_id();
  uint32_t kmn = 0xffffffffu, kmx = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const uint32_t k = static_cast<uint32_t>(c[e] >> 32);
    if (c[e] != 0u) {
      kmn = min(kmn, k);
      kmx = max(kmx, k);
    }
  }
  kmn = __reduce_min_sync(kFull, kmn);
  kmx = __reduce_max_sync(kFull, kmx);
  if (kmx < kmn) return 0;  // no entry (warp-uniform)
  const float scale = static_cast<float>(NB) / (static_cast<float>(kmx - kmn) + 1.0f);
  int d[E];  // bucket, the highest keys in bucket 0
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const uint32_t rel = static_cast<uint32_t>(c[e] >> 32) - kmn;
    const int b = min(NB - 1, static_cast<int>(__float2uint_rz(static_cast<float>(rel) * scale)));
    d[e] = NB - 1 - b;
    if (c[e] != 0u) atomicAdd(hist + d[e], 1u);
  }
  __syncwarp();
  // exclusive prefix over the buckets: lane l owns buckets BPL l .. BPL l + BPL - 1
  constexpr int BPL = NB / 32;
  uint32_t h[BPL], run = 0u, big = 0u;
#pragma unroll
  for (int j = 0; j < BPL; ++j) {
    h[j] = hist[BPL * lane + j];
    run += h[j];
    big = max(big, h[j]);
  }
  big = __reduce_max_sync(kFull, big);
  const uint32_t n = __reduce_add_sync(kFull, run);
  uint32_t base = static_cast<uint32_t>(warp_incl_scan(static_cast<int>(run))) - run;
  __syncwarp();
  if (big > 32u) return -1;  // warp-uniform
#pragma unroll
  for (int j = 0; j < BPL; ++j) {
    hist[BPL * lane + j] = base;
    base += h[j];
  }
  __syncwarp();
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (c[e] != 0u) tmp[atomicAdd(hist + d[e], 1u)] = c[e];
  __syncwarp();  // hist[b] is now the end of bucket b
  // per entry: bucket start (bits 0-9), bucket length (10-15), rank (16-)
  uint32_t info[E];
  uint32_t maxlen = 0u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const uint32_t lo = d[e] == 0 ? 0u : hist[d[e] - 1];
    const uint32_t len = c[e] != 0u ? hist[d[e]] - lo : 0u;
    info[e] = lo | (len << 10);
    maxlen = max(maxlen, len);
  }
  maxlen = __reduce_max_sync(kFull, maxlen);
  // member j of every entry's bucket in one step: E independent loads
  for (uint32_t j = 0; j < maxlen; ++j) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const uint32_t lo = info[e] & 1023u, len = (info[e] >> 10) & 63u;
      if (j < len && tmp[lo + j] > c[e]) info[e] += 1u << 16;
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (c[e] != 0u)
      cols[(info[e] & 1023u) + (info[e] >> 16)] =
          static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(c[e]));
  __syncwarp();
  return static_cast<int>(n);
}

// Seven CTAs per SM, as the unsorted warp kernel: the index map lives in
// the warp's histogram (idle and zero while the emit runs); after the
// gather the list area holds the scatter scratch and the 512 bucket
// counters, and the ranked columns go straight to the output row.
template <typename T, int ALIGN, int E>
__global__ void __launch_bounds__(32 * kWarpRowsPerCta, 7)
    topk_rows_warp_sorted_kernel(const T *__restrict__ x, int64_t rows, int64_t ld, int cols,
                                 const int32_t *__restrict__ row_ends, int K,
                                 int32_t *__restrict__ out, int64_t ld_out) {
  static_assert(sizeof(uint64_t) * 32 * E <= 1024 * sizeof(uint32_t) &&
                    (1024 + 512) * sizeof(uint32_t) <= sizeof(WarpRowSmem::buf),
                "the scatter scratch and the 512 bucket counters fit the list area");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int warp = warp_id(), lane = lane_id();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpRowsPerCta + warp;
  if (row >= rows) return;  // warp-uniform; the warps never synchronise
  WarpRowSmem &ws = reinterpret_cast<WarpRowSmem *>(smem_raw)[warp];
  // the emit writes map[pos] for every pos < K (no fill needed before the
  // row: the histogram must be zero then)
  uint16_t *map = reinterpret_cast<uint16_t *>(ws.hist);
  for (int i = lane; i < 256; i += 32) ws.hist[i] = 0u;
  __syncwarp();
  warp_topk_row<T, ALIGN>(x + row * ld, row_end_of(row_ends, row, cols), K, SortMapOut{map, K},
                          ws);
  __syncwarp();
  uint64_t c[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int p = e * 32 + lane;
    const uint32_t i = p < K ? map[p] : 0xffffu;
    c[e] = i == 0xffffu ? 0u
                        : (static_cast<uint64_t>(ws.key()[i]) << 32) |
                              (0xffffffffu - static_cast<uint32_t>(ws.col()[i]));
  }
  __syncwarp();  // the list and the map are read: the list area is the sort's scratch now
  uint64_t *tmp = reinterpret_cast<uint64_t *>(ws.buf);
  uint32_t *cnt512 = ws.buf + 1024;  // the list area's last 2 KB: the bucket counters
  for (int i = lane; i < 512; i += 32) cnt512[i] = 0u;
  __syncwarp();
  int32_t *o = out + row * ld_out;
  const int nb = warp_bucket_rank<E>(c, tmp, o, cnt512);
  if (nb >= 0) {  // warp-uniform
    for (int q = nb + lane; q < K; q += 32) o[q] = -1;
    return;
  }
  warp_bitonic_desc<E>(c);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int q = lane * E + e;
    if (q < K)
      o[q] = c[e] == 0u ? -1 : static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(c[e]));
  }
}

template <typename T, int ALIGN, int E>
int launch_warp_sorted(const T *x, int64_t rows, int cols, int64_t ld, const int32_t *row_ends,
                       int K, int32_t *out, int64_t ld_out, cudaStream_t st) {
  auto kern = topk_rows_warp_sorted_kernel<T, ALIGN, E>;
  const size_t smem = sizeof(WarpRowSmem) * kWarpRowsPerCta;
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  const int64_t grid = (rows + kWarpRowsPerCta - 1) / kWarpRowsPerCta;
  kern<<<dim3(static_cast<unsigned>(grid)), 32 * kWarpRowsPerCta, smem, st>>>(
      x, rows, ld, cols, row_ends, K, out, ld_out);
  return launch_status();
}

// The chosen set of topk_rows_kernel in score order: the row path emits
// (key << 32 | ~column) composites into shared memory, a bitonic sort puts
// them in descending order (key desc, then column asc), and the columns are
// written out; positions without a candidate hold 0 and become -1.
template <typename T, int SUB, int ALIGN, int P>
__global__ void __launch_bounds__(kBlock, 4) topk_rows_sorted_kernel(
    const T *__restrict__ x, int64_t ld, int cols, const int32_t *__restrict__ row_ends, int K,
    int32_t *__restrict__ out, int64_t ld_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<ListSmem<kBlock, SUB> *>(smem_raw);
  uint64_t *buf = reinterpret_cast<uint64_t *>(smem_raw + sorted_buf_offset<SUB>());
  const int64_t row = blockIdx.x;
  zero_hist(sm.sel);
  for (int i = threadIdx.x; i < P; i += kBlock) buf[i] = 0u;
  __syncthreads();
  topk_row<T, kBlock, SUB, ALIGN>(
      x + row * ld, row_end_of(row_ends, row, cols), K,
      [&](int pos, int i) {
        if ((unsigned)pos < (unsigned)K)
          buf[pos] = (static_cast<uint64_t>(sm.key[i]) << 32) | (0xffffffffu - sm.val[i]);
      },
      [](int) {}, sm);
  __syncthreads();
  bitonic_sort_desc<kBlock, P>(buf);
  int32_t *o = out + row * ld_out;
  for (int q = threadIdx.x; q < K; q += kBlock) {
    const uint64_t c = buf[q];
    o[q] = c == 0u ? -1 : static_cast<int32_t>(0xffffffffu - static_cast<uint32_t>(c));
  }
}

template <typename T, int SUB, int ALIGN, int P>
int launch_sorted(const T *x, int64_t rows, int cols, int64_t ld, const int32_t *row_ends, int K,
                  int32_t *out, int64_t ld_out, cudaStream_t st) {
  auto kern = topk_rows_sorted_kernel<T, SUB, ALIGN, P>;
  const size_t smem = sorted_buf_offset<SUB>() + sizeof(uint64_t) * P;
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  kern<<<dim3(static_cast<unsigned>(rows)), kBlock, smem, st>>>(x, ld, cols, row_ends, K, out,
                                                                ld_out);
  return launch_status();
}

template <typename T, int ALIGN>
int launch_rows_sorted(const T *x, int64_t rows, int cols, int64_t ld, const int32_t *row_ends,
                       int K, int32_t *out, int64_t ld_out, cudaStream_t st) {
  if (warp_rows_fit(cols, K)) {  // K <= 512: one warp per row, sort widths 128 and 512
    if (K <= 128)
      return launch_warp_sorted<T, ALIGN, 4>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
    return launch_warp_sorted<T, ALIGN, 16>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
  }
  if (K <= 512)
    return launch_sorted<T, 512, ALIGN, 512>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
  if (K <= 1024)
    return launch_sorted<T, 512, ALIGN, 1024>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
  if (K <= 2048)
    return launch_sorted<T, 1024, ALIGN, 2048>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
  return launch_sorted<T, 1024, ALIGN, 4096>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
}

}  // namespace

// One (type, alignment) pair of the row kernels: the entry points of
// topk_rows.cu call these, defined in the per-pair translation units.
int topk_rows_launch_f32_a32(const float *x, int64_t rows, int cols, int64_t ld,
                             const int32_t *row_ends, int K, int32_t *out, int64_t ld_out,
                             bool sorted, cudaStream_t st);
int topk_rows_launch_f32_a16(const float *x, int64_t rows, int cols, int64_t ld,
                             const int32_t *row_ends, int K, int32_t *out, int64_t ld_out,
                             bool sorted, cudaStream_t st);
int topk_rows_launch_f32_a0(const float *x, int64_t rows, int cols, int64_t ld,
                            const int32_t *row_ends, int K, int32_t *out, int64_t ld_out,
                            bool sorted, cudaStream_t st);
int topk_rows_launch_bf16_a16(const uint16_t *x, int64_t rows, int cols, int64_t ld,
                              const int32_t *row_ends, int K, int32_t *out, int64_t ld_out,
                              bool sorted, cudaStream_t st);
int topk_rows_launch_bf16_a0(const uint16_t *x, int64_t rows, int cols, int64_t ld,
                             const int32_t *row_ends, int K, int32_t *out, int64_t ld_out,
                             bool sorted, cudaStream_t st);
// The local top-K of bf16 rows written as B' rows (PackedOut) of K + K/32
// words: satk_dcp_topk_pack.
int topk_pack_launch_bf16_a16(const uint16_t *x, int64_t rows, int cols, int64_t ld,
                              const int32_t *row_ends, int K, int32_t *packed, cudaStream_t st);
int topk_pack_launch_bf16_a0(const uint16_t *x, int64_t rows, int cols, int64_t ld,
                             const int32_t *row_ends, int K, int32_t *packed, cudaStream_t st);

}  // namespace satk
