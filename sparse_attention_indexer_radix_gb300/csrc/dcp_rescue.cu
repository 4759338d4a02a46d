// dcp_rescue.cu -- satk_dcp_rescue_select: the second round of the packed
// merge (vLLM API page vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge
// .kernels: module docstring, push_local_topk inside DCPTopkSelectKernel,
// DCPTopkRescueKernel).
//
// On the page each saturated rank pushes its local top-K into every rank's
// receive slot with peer stores and a release flag, and a persistent kernel
// spins on the flags before re-selecting.  Here all W ranks' rows are in
// one device buffer, so the push is an ordinary kernel writing `recv` and
// stream order replaces the flags: nothing waits on anything.
//
// rescue_push_kernel  : one CTA per (row, slot) (a cluster of CTAs for long
//                       rank rows); slot s of a row with a
//                       non-zero mask takes the s-th set bit's rank, runs the
//                       row top-K on that rank's bf16 logits (the streaming
//                       path of satk_rows.cuh) and writes the list in the B'
//                       layout to recv[t, s].
// rescue_select_kernel: one CTA per row; a zero mask costs one load.  The
//                       candidates are the round-1 words of the ranks outside
//                       the mask, then the pushed lists, those scoring at or
//                       above tau16 filtered into the shared-memory list; the
//                       list merge select picks K (the register select of
//                       satk_merge.cuh when the list would overflow).
#include <climits>

#include "satk_cluster.cuh"
#include "satk_host.hpp"
#include "satk_merge.cuh"
#include "satk_rows.cuh"

namespace satk {
namespace {

constexpr int kPushBlock = 256;
// Rank rows of at least kPushClusterCols columns are pushed by clusters of
// kPushCluster CTAs (measured on the decode workload: rescue 56 -> 49 us
// with four, 54 us with eight); the grid holds every (row, slot) pair.
constexpr int kPushCluster = 4;
constexpr int64_t kPushClusterCols = 32768;
constexpr int64_t kPushClusterMaxPairs = (int64_t{1} << 31) / (2 * kPushCluster);

__device__ __forceinline__ int nth_set_bit(uint32_t mask, int s) {
  for (int q = 0; q < s; ++q) mask &= mask - 1u;
  return __ffs(mask) - 1;
}

template <int SUB, int ALIGN>
__global__ void __launch_bounds__(kPushBlock) rescue_push_kernel(
    const uint16_t *__restrict__ logits, int64_t S, int64_t ld, int W, int64_t T, int K,
    int slots, const int32_t *__restrict__ row_ends, const int32_t *__restrict__ sat_word,
    int32_t *__restrict__ recv, int32_t *__restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  using SM = ListSmem<kPushBlock, SUB>;
  auto &sm = *reinterpret_cast<SM *>(smem_raw);
  uint32_t *bp = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SM));
  const int64_t t = blockIdx.x / slots;
  const int s = blockIdx.x % slots;
  const uint32_t mask = static_cast<uint32_t>(sat_word[t]) >> 16;
  if (mask == 0u) return;
  const int nsat = __popc(mask);
  if (nsat > slots || (mask >> W) != 0u) {
    if (s == 0 && threadIdx.x == 0 && status != nullptr)
      atomicOr(status, SATK_STATUS_SLOTS_EXCEEDED);
    return;
  }
  if (s >= nsat) return;
  const int r = nth_set_bit(mask, s);
  int64_t end = S < SATK_LOCAL_INDEX_LIMIT ? S : SATK_LOCAL_INDEX_LIMIT;
  if (row_ends != nullptr && (int64_t)row_ends[(int64_t)r * T + t] < end)
    end = row_ends[(int64_t)r * T + t];
  if (end < 0) end = 0;
  const int words = K + K / 32;
  for (int i = threadIdx.x; i < words; i += kPushBlock) bp[i] = 0u;
  zero_hist(sm.sel);
  __syncthreads();
  // the rank's local top-K in the B' layout: ord16 << 16 | ~local[15:0],
  // local[16] in the bit plane
  topk_row<uint16_t, kPushBlock, SUB, ALIGN>(
      logits + ((int64_t)r * T + t) * ld, static_cast<int>(end), K,
      [&](int pos, int i) {
        if ((unsigned)pos >= (unsigned)K) return;
        const uint32_t col = sm.val[i];
        bp[pos] = sm.key[i] | (0xffffu - (col & 0xffffu));
        if ((col >> 16) & 1u) atomicOr(bp + K + pos / 32, 1u << (pos & 31));
      },
      [](int) {}, sm);
  __syncthreads();
  int32_t *dst = recv + ((int64_t)t * slots + s) * words;
  for (int i = threadIdx.x; i < words; i += kPushBlock) dst[i] = static_cast<int32_t>(bp[i]);
}

template <int SUB, int ALIGN>
int launch_push(const uint16_t *logits, int64_t S, int64_t ld, int W, int64_t T, int K, int slots,
                const int32_t *row_ends, const int32_t *sat_word, int32_t *recv,
                int32_t *status, cudaStream_t st) {
  auto kern = rescue_push_kernel<SUB, ALIGN>;
  const size_t smem = sizeof(ListSmem<kPushBlock, SUB>) + sizeof(uint32_t) * (size_t)(K + K / 32);
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  kern<<<dim3(static_cast<unsigned>(T * slots)), kPushBlock, smem, st>>>(
      logits, S, ld, W, T, K, slots, row_ends, sat_word, recv, status);
  return launch_status();
}

// The push on a cluster of C CTAs per (row, slot) for long rank rows (only
// a few (row, rank) pairs push, so one CTA each leaves most SMs idle): the
// row path of satk_cluster.cuh, each CTA writing its own words of the B'
// list straight to recv, plane bits by atomics on words CTA 0 zeroes before
// the first cluster barrier.  A (row, slot) without a push leaves as a
// whole cluster (the decision reads only the row's sat_word).
template <int SUB, int ALIGN, int C>
__global__ void __cluster_dims__(C, 1, 1) __launch_bounds__(kPushBlock, 1024 / kPushBlock)
    rescue_push_cluster_kernel(const uint16_t *__restrict__ logits, int64_t S, int64_t ld, int W,
                               int64_t T, int K, int slots,
                               const int32_t *__restrict__ row_ends,
                               const int32_t *__restrict__ sat_word, int32_t *__restrict__ recv,
                               int32_t *__restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto &cs = *reinterpret_cast<ClusterSmem<kPushBlock, SUB> *>(smem_raw);
  cg::cluster_group cl = cg::this_cluster();
  const int64_t q = blockIdx.x / C;
  const int64_t t = q / slots;
  const int s = static_cast<int>(q % slots);
  const uint32_t mask = static_cast<uint32_t>(sat_word[t]) >> 16;
  if (mask == 0u) return;
  const int nsat = __popc(mask);
  if (nsat > slots || (mask >> W) != 0u) {
    if (s == 0 && cl.block_rank() == 0 && threadIdx.x == 0 && status != nullptr)
      atomicOr(status, SATK_STATUS_SLOTS_EXCEEDED);
    return;
  }
  if (s >= nsat) return;
  const int r = nth_set_bit(mask, s);
  int64_t end = S < SATK_LOCAL_INDEX_LIMIT ? S : SATK_LOCAL_INDEX_LIMIT;
  if (row_ends != nullptr && (int64_t)row_ends[(int64_t)r * T + t] < end)
    end = row_ends[(int64_t)r * T + t];
  if (end < 0) end = 0;
  uint32_t *dst = reinterpret_cast<uint32_t *>(recv) + ((int64_t)t * slots + s) * (K + K / 32);
  if (cl.block_rank() == 0)
    for (int i = threadIdx.x; i < K / 32; i += kPushBlock) dst[K + i] = 0u;
  zero_hist(cs.ls.sel);
  __syncthreads();
  cluster_topk_row<uint16_t, kPushBlock, SUB, ALIGN, C>(
      cl, logits + ((int64_t)r * T + t) * ld, static_cast<int>(end), K,
      [&](int pos, uint32_t key, int col) {
        if (!satk_check(pos >= 0 && pos < K, kDbgOut)) return;
        dst[pos] = key | (0xffffu - (static_cast<uint32_t>(col) & 0xffffu));
        if ((col >> 16) & 1) atomicOr(dst + K + pos / 32, 1u << (pos & 31));
      },
      [&](int pos) {
        if (satk_check(pos >= 0 && pos < K, kDbgOut)) dst[pos] = 0u;
      },
      cs);
}

template <int SUB, int ALIGN, int C>
int launch_push_cluster(const uint16_t *logits, int64_t S, int64_t ld, int W, int64_t T, int K,
                        int slots, const int32_t *row_ends, const int32_t *sat_word,
                        int32_t *recv, int32_t *status, cudaStream_t st) {
  auto kern = rescue_push_cluster_kernel<SUB, ALIGN, C>;
  const size_t smem = sizeof(ClusterSmem<kPushBlock, SUB>);
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  kern<<<dim3(static_cast<unsigned>(T * slots * C)), kPushBlock, smem, st>>>(
      logits, S, ld, W, T, K, slots, row_ends, sat_word, recv, status);
  return launch_status();
}

template <int BLOCK, int KPT>
struct RescueSmem {
  SelectSmem<BLOCK> sel;
  uint32_t gid[BLOCK * KPT];
};

// The register select over every candidate slot (KPT per thread): the
// exact path when the filtered list of rescue_select_kernel overflows.
template <int BLOCK, int KPT>
__device__ void rescue_select_regs(RescueSmem<BLOCK, KPT> &sm, const int32_t *__restrict__ packed,
                                   int W, int64_t T, int n, int K, int slots, uint32_t mask,
                                   uint32_t tau, const int32_t *__restrict__ recv,
                                   int32_t *__restrict__ out, int32_t *__restrict__ status) {
  const int64_t t = blockIdx.x;
  const int nsat = __popc(mask);
  const int lane = lane_id();
  const int r1 = W * n;
  const int total = r1 + slots * K;
  const int words_r1 = n + n / 32, words_k = K + K / 32;
  zero_hist(sm.sel);
  uint32_t keys[KPT];
#pragma unroll
  for (int g = 0; g < KPT; ++g) {
    const int fb = warp_id() * 32 * KPT + g * 32;
    uint32_t key = 0u, gid = 0u;
    if (fb < r1) {
      const int r = fb / n, j = fb - r * n + lane;
      if (((mask >> r) & 1u) == 0u) {
        const int32_t *row = packed + ((int64_t)r * T + t) * words_r1;
        const uint32_t w = static_cast<uint32_t>(__ldg(row + j));
        const uint32_t plane = static_cast<uint32_t>(__ldg(row + n + ((j - lane) >> 5)));
        key = bprime_key(w);
        if ((key >> 16) < tau) key = 0u;  // below the round-1 cut
        gid = bprime_local(w, plane, j) * (uint32_t)W + (uint32_t)r;
      }
    } else if (fb < total) {
      const int q = fb - r1;
      const int s = q / K, j = q - s * K + lane;
      if (s < nsat) {
        const int32_t *sl = recv + ((int64_t)t * slots + s) * words_k;
        const uint32_t w = static_cast<uint32_t>(sl[j]);
        const uint32_t plane = static_cast<uint32_t>(sl[K + ((j - lane) >> 5)]);
        key = bprime_key(w);
        gid = bprime_local(w, plane, j) * (uint32_t)W + (uint32_t)nth_set_bit(mask, s);
      }
    }
    keys[g] = key;
    if (satk_check(fb + lane < BLOCK * KPT, kDbgScratch)) sm.gid[fb + lane] = gid;
  }
  __syncthreads();
  const MergeOut m = merge_core<BLOCK, KPT, 16>(
      keys, [&](int i) { return sm.gid[flat_pos<KPT, 1>(i)]; },
      [&](int pos, int32_t v) {
        if ((unsigned)pos < (unsigned)K) out[pos] = v;
      },
      K, false, sm.sel);
  if (m.dup && status != nullptr && threadIdx.x == 0)
    atomicOr(status, SATK_STATUS_DUPLICATE_KEYS);
}

// One CTA per row; a zero mask costs one load.  The candidates at or above
// tau16 -- the round-1 words of the ranks outside the mask, then the pushed
// lists -- are filtered in flat order into the shared-memory list (each warp
// over a contiguous stretch, 32 candidates per step), and the list merge
// select picks K.  The round-1 choice (K candidates scoring >= tau16) is
// among them, so no candidate below tau16 can be chosen.  A warp segment
// that would overflow sends the row to the register select over every slot.
template <int BLOCK, int KPT, int SUB>
__global__ void __launch_bounds__(BLOCK) rescue_select_kernel(
    const int32_t *__restrict__ packed, int W, int64_t T, int n, int K, int slots,
    const int32_t *__restrict__ sat_word, const int32_t *__restrict__ recv,
    int32_t *__restrict__ ids, int64_t ld_out, int32_t *__restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<ListSmem<BLOCK, SUB> *>(smem_raw);
  constexpr int NW = BLOCK / 32;
  const int64_t t = blockIdx.x;
  const uint32_t sw = static_cast<uint32_t>(sat_word[t]);
  const uint32_t mask = sw >> 16, tau = sw & 0xffffu;
  if (mask == 0u) return;  // round 1 was exact
  const int nsat = __popc(mask);
  if (nsat > slots || (mask >> W) != 0u) return;  // reported by the push
  const int lane = lane_id(), warp = warp_id();
  const unsigned lt = (1u << lane) - 1u;
  const int r1 = W * n;
  const int words_r1 = n + n / 32, words_k = K + K / 32;
  const int nchunks = (r1 + nsat * K) / 32;  // n, K multiples of 32
  const int per = (nchunks + NW - 1) / NW;
  const int c0 = min(nchunks, warp * per), c1 = min(nchunks, c0 + per);
  zero_hist(sm.sel);
  if (threadIdx.x == 0) sm.flag = 0;
  __syncthreads();
  uint32_t *lk = sm.key + warp * SUB;
  uint32_t *lv = sm.val + warp * SUB;
  int cnt = 0;
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  // the words of up to kLoadBatch chunks are loaded before any is listed,
  // so their latencies overlap
  constexpr int kLoadBatch = 8;
  bool over = false;
  for (int cb = c0; cb < c1 && !over; cb += kLoadBatch) {
    uint32_t wv[kLoadBatch], pv[kLoadBatch], ov[kLoadBatch];
    int jv[kLoadBatch];
#pragma unroll
    for (int q = 0; q < kLoadBatch; ++q) {
      const int c = cb + q;
      wv[q] = 0u;
      pv[q] = 0u;
      ov[q] = 0u;
      jv[q] = 0;
      if (c < c1) {
        const int fb = c * 32;
        if (fb < r1) {
          const int r = fb / n, j = fb - r * n + lane;
          if (((mask >> r) & 1u) == 0u) {
            const int32_t *row = packed + ((int64_t)r * T + t) * words_r1;
            wv[q] = static_cast<uint32_t>(__ldg(row + j));
            pv[q] = static_cast<uint32_t>(__ldg(row + n + ((j - lane) >> 5)));
          }
          ov[q] = static_cast<uint32_t>(r);
          jv[q] = j;
        } else {
          const int qq = fb - r1;
          const int s = qq / K, j = qq - s * K + lane;
          const int32_t *sl = recv + ((int64_t)t * slots + s) * words_k;
          wv[q] = static_cast<uint32_t>(sl[j]);
          pv[q] = static_cast<uint32_t>(sl[K + ((j - lane) >> 5)]);
          ov[q] = static_cast<uint32_t>(nth_set_bit(mask, s));
          jv[q] = j;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kLoadBatch; ++q) {
      if (cb + q < c1 && !over) {  // warp-uniform
        uint32_t key = bprime_list_key(wv[q]);
        if (key <= tau) key = 0u;  // ord16 below the round-1 cut (or empty); keys are ord16 + 1
        const unsigned b = __ballot_sync(kFull, key != 0u);
        if (cnt + __popc(b) > SUB) {  // warp-uniform
          if (lane == 0) sm.flag = 1;
          over = true;
        } else {
          if (key != 0u) {
            const int pos = cnt + __popc(b & lt);
            if (satk_check(pos < SUB, kDbgList)) {
              lk[pos] = key;
              lv[pos] = bprime_local(wv[q], pv[q], jv[q]) * (uint32_t)W + ov[q];
            }
            kmn = min(kmn, key);
            kmx = max(kmx, key);
          }
          cnt += __popc(b);
        }
      }
    }
  }
  const WarpStats st{cnt, __reduce_min_sync(kFull, kmn), __reduce_max_sync(kFull, kmx)};
  __syncthreads();
  int32_t *out = ids + t * ld_out;
  if (sm.flag == 0) {  // block-uniform
    const bool dup = list_merge_emit<BLOCK, SUB>(
        sm, Seg{warp * SUB, cnt}, K,
        [&](int pos, int32_t v) {
          if ((unsigned)pos < (unsigned)K) out[pos] = v;
        },
        st).dup;
    if (dup && status != nullptr && threadIdx.x == 0)
      atomicOr(status, SATK_STATUS_DUPLICATE_KEYS);
    return;
  }
  __syncthreads();
  rescue_select_regs<BLOCK, KPT>(*reinterpret_cast<RescueSmem<BLOCK, KPT> *>(smem_raw), packed,
                                 W, T, n, K, slots, mask, tau, recv, out, status);
}

template <int BLOCK, int KPT>
int launch_rescue_select(const int32_t *packed, int W, int64_t T, int n, int K, int slots,
                         const int32_t *sat_word, const int32_t *recv, int32_t *ids,
                         int64_t ld_out, int32_t *status, cudaStream_t st) {
  constexpr int SUB = 512;  // list of (BLOCK / 32) x 512 entries
  auto kern = rescue_select_kernel<BLOCK, KPT, SUB>;
  const size_t smem = sizeof(RescueSmem<BLOCK, KPT>) > sizeof(ListSmem<BLOCK, SUB>)
                          ? sizeof(RescueSmem<BLOCK, KPT>)
                          : sizeof(ListSmem<BLOCK, SUB>);
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  kern<<<dim3(static_cast<unsigned>(T)), BLOCK, smem, st>>>(packed, W, T, n, K, slots, sat_word,
                                                            recv, ids, ld_out, status);
  return launch_status();
}

}  // namespace
}  // namespace satk

extern "C" size_t satk_rescue_recv_words(int64_t T, int32_t n, int32_t k) {
  if (T < 0 || n < 1 || k < 1) return 0;
  return static_cast<size_t>(T) * static_cast<size_t>((k - 1) / n) *
         static_cast<size_t>(k + k / 32);
}

extern "C" int satk_dcp_rescue_select(const int32_t *packed, int32_t W, int64_t T, int32_t n,
                                      int32_t k, const uint16_t *logits_bf16, int64_t S,
                                      int64_t ld_logits, const int32_t *row_ends,
                                      const int32_t *sat_word, int32_t *recv,
                                      int32_t *ids_out, int64_t ld_out, int32_t *status,
                                      satk_stream_t stream) {
  using namespace satk;
  if (packed == nullptr || logits_bf16 == nullptr || sat_word == nullptr || recv == nullptr ||
      ids_out == nullptr || W < 1 || W > 16 || T < 0 || n < 32 || n % 32 != 0 || k < 32 ||
      k % 32 != 0 || n >= k || k > SATK_TOPK_MAX_K || ld_out < k || S < 0 || ld_logits < S ||
      T > INT_MAX / 16)
    return SATK_EINVAL;
  const int slots = (k - 1) / n;
  if ((int64_t)W * n + (int64_t)slots * k > SATK_MERGE_MAX_CANDIDATES ||
      T * slots > INT_MAX)
    return SATK_EUNSUPPORTED;
  if (T == 0) return SATK_OK;
  const cudaStream_t st = as_stream(stream);

  // 1. pushes of the saturated ranks
  const bool vec = aligned16(logits_bf16) && (ld_logits * 2) % 16 == 0;
  int rc;
  if (S >= kPushClusterCols && vec && T * slots <= kPushClusterMaxPairs) {
    if (k <= 1024)
      rc = launch_push_cluster<512, 16, kPushCluster>(logits_bf16, S, ld_logits, W, T, k, slots,
                                                      row_ends, sat_word, recv, status, st);
    else
      rc = launch_push_cluster<1024, 16, kPushCluster>(logits_bf16, S, ld_logits, W, T, k, slots,
                                                       row_ends, sat_word, recv, status, st);
  } else if (k <= 1024)
    rc = vec ? launch_push<512, 16>(logits_bf16, S, ld_logits, W, T, k, slots, row_ends,
                                      sat_word, recv, status, st)
             : launch_push<512, 0>(logits_bf16, S, ld_logits, W, T, k, slots, row_ends,
                                       sat_word, recv, status, st);
  else
    rc = vec ? launch_push<1024, 16>(logits_bf16, S, ld_logits, W, T, k, slots, row_ends,
                                       sat_word, recv, status, st)
             : launch_push<1024, 0>(logits_bf16, S, ld_logits, W, T, k, slots, row_ends,
                                        sat_word, recv, status, st);
  if (rc != SATK_OK) return rc;

  // 2. the re-select over round-1 words and the pushed lists
  const int total = W * n + slots * k;
  if (total <= 512 * 8)
    return launch_rescue_select<512, 8>(packed, W, T, n, k, slots, sat_word, recv, ids_out,
                                        ld_out, status, st);
  if (total <= 512 * 32)
    return launch_rescue_select<512, 32>(packed, W, T, n, k, slots, sat_word, recv, ids_out,
                                         ld_out, status, st);
  return launch_rescue_select<1024, 32>(packed, W, T, n, k, slots, sat_word, recv, ids_out,
                                        ld_out, status, st);
}
