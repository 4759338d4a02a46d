// dcp_merge.cu -- satk_dcp_pack and satk_dcp_merge_select.
//
// Pack: vLLM API page vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels,
// DCPTopkPackKernel and dcp_topk_pack_indices.  Merge: the same page,
// DCPTopkSelectKernel (packed B' rows, saturation word), and vLLM PR #65178
// "DCP top-k merge reads the rank-major all-gather buffer in place",
// Overview (the (score, global id) pairs read from the rank-major
// [W, T, n, 2] buffer without a reorder copy).
//
// Both merge formats read the rank-major buffer in place: the flat
// candidate f of row t is slot f % n of rank f / n, so with n % 32 == 0
// every warp-wide group of 32 consecutive candidates lies inside one rank
// and its 32 slots are contiguous in memory.  One CTA per row.
#include <climits>

#include "satk_host.hpp"
#include "satk_merge.cuh"

namespace satk {
namespace {

// ------------------------------------------------------------------ pack --

__global__ void __launch_bounds__(512) dcp_pack_kernel(const uint16_t *__restrict__ logits,
                                                       int64_t S, int64_t ld,
                                                       const int32_t *__restrict__ local_idx,
                                                       int64_t ld_idx, int n,
                                                       const int32_t *__restrict__ row_ends,
                                                       int32_t *__restrict__ packed) {
  const int64_t row = blockIdx.x;
  int64_t end = S < SATK_LOCAL_INDEX_LIMIT ? S : SATK_LOCAL_INDEX_LIMIT;
  if (row_ends != nullptr && (int64_t)row_ends[row] < end) end = row_ends[row];
  const int64_t words = n + n / 32;
  const uint16_t *lr = logits + row * ld;
  int32_t *pr = packed + row * words;
  for (int j0 = 0; j0 < n; j0 += blockDim.x) {
    const int j = j0 + threadIdx.x;
    if (j < n) {  // n and blockDim are multiples of 32: whole warps
      const int32_t l = local_idx[row * ld_idx + j];
      uint32_t word = 0u;
      bool hi = false;
      if (l >= 0 && (int64_t)l < end) {
        const uint32_t k = key_bf16(__ldg(reinterpret_cast<const unsigned short *>(lr + l)));
        if (k != 0u) {  // not NaN
          word = k | (0xffffu - ((uint32_t)l & 0xffffu));
          hi = (((uint32_t)l >> 16) & 1u) != 0u;
        }
      }
      pr[j] = static_cast<int32_t>(word);
      const unsigned bits = __ballot_sync(kFull, hi);
      if (lane_id() == 0) pr[n + j / 32] = static_cast<int32_t>(bits);
    }
  }
}

// ----------------------------------------------------------------- merge --

template <int BLOCK, int KPT>
struct MergeSmem {
  SelectSmem<BLOCK> sel;
  int notsat[16];
  uint32_t gid[BLOCK * KPT];
};

// PACKED: cand = int32 [W, T, n + n/32] B' rows.
// !PACKED: cand = [W, T, n, 2] (float score bits, int32 gid) pairs.
template <int BLOCK, int KPT, bool PACKED>
__global__ void __launch_bounds__(BLOCK) merge_select_kernel(
    const int32_t *__restrict__ cand, int W, int64_t T, int n, int K,
    int32_t *__restrict__ ids, int64_t ld_out, int32_t *__restrict__ sat_word,
    int32_t *__restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<MergeSmem<BLOCK, KPT> *>(smem_raw);
  const int64_t t = blockIdx.x;
  const int lane = lane_id();
  const int total = W * n;
  zero_hist(sm.sel);
  if (threadIdx.x < 16) sm.notsat[threadIdx.x] = 0;

  // ---- load the row's candidates in place (rank-major)
  uint32_t keys[KPT];
  const int fb0 = warp_id() * 32 * KPT;
  {
    int r = fb0 / n, j0 = fb0 - r * n;
#pragma unroll
    for (int g = 0; g < KPT; ++g) {
      const int f = fb0 + g * 32 + lane;
      uint32_t key = 0u, gid = 0u;
      if (r < W) {
        const int j = j0 + lane;
        if constexpr (PACKED) {
          const int32_t *row = cand + ((int64_t)r * T + t) * (n + n / 32);
          const uint32_t w = static_cast<uint32_t>(__ldg(row + j));
          const uint32_t plane = static_cast<uint32_t>(__ldg(row + n + (j0 >> 5)));
          key = bprime_key(w);
          gid = bprime_local(w, plane, j) * (uint32_t)W + (uint32_t)r;
        } else {
          const int2 pr = __ldg(reinterpret_cast<const int2 *>(cand) + ((int64_t)r * T + t) * n + j);
          key = pr.y >= 0 ? key_f32(static_cast<uint32_t>(pr.x)) : 0u;
          gid = static_cast<uint32_t>(pr.y);
        }
      }
      keys[g] = key;
      sm.gid[f] = gid;
      j0 += 32;
      if (j0 >= n) {
        j0 -= n;
        ++r;
      }
    }
  }
  (void)total;
  __syncthreads();

  int32_t *out = ids + t * ld_out;
  auto gid_of = [&](int i) { return sm.gid[flat_pos<KPT, 1>(i)]; };
  constexpr int KB = PACKED ? 16 : 32;
  const MergeOut m = merge_core<BLOCK, KPT, KB>(
      keys, gid_of,
      [&](int pos, int32_t v) {
        if ((unsigned)pos < (unsigned)K) out[pos] = v;
      },
      K,
      PACKED && sat_word != nullptr, sm.sel);

  int bits = m.dup ? SATK_STATUS_DUPLICATE_KEYS : 0;
  if constexpr (PACKED) {
    if (sat_word != nullptr) {
      // tau16: ord16 of the K-th chosen candidate, 0 below K chosen
      const uint32_t tau = (m.nsel == K) ? (m.kmin >> 16) : 0u;
      // rank r is saturated iff all its n slots hold words scoring > tau16
      int r = fb0 / n;
#pragma unroll
      for (int g = 0; g < KPT; ++g) {
        if (r < W) {
          const bool above = keys[g] != 0u && (keys[g] >> 16) > tau;
          if (__ballot_sync(kFull, above) != kFull && lane == 0) sm.notsat[r] = 1;
        }
        // advance one group of 32
        if (((fb0 + (g + 1) * 32) % n) == 0) ++r;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        uint32_t mask = 0u;
        for (int q = 0; q < W; ++q)
          if (sm.notsat[q] == 0) mask |= 1u << q;
        const int slots = (K - 1) / n;
        if (__popc(mask) > slots) {
          mask = 0u;  // more saturated ranks than slots: keep round 1
          bits |= SATK_STATUS_SLOTS_EXCEEDED;
        }
        sat_word[t] = static_cast<int32_t>((mask << 16) | tau);
      }
    }
  }
  if (bits != 0 && status != nullptr && threadIdx.x == 0) atomicOr(status, bits);
}

template <int BLOCK, int KPT, bool PACKED>
int launch_merge(const int32_t *cand, int W, int64_t T, int n, int K, int32_t *ids,
                 int64_t ld_out, int32_t *sat_word, int32_t *status, cudaStream_t st) {
  auto kern = merge_select_kernel<BLOCK, KPT, PACKED>;
  const size_t smem = sizeof(MergeSmem<BLOCK, KPT>);
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  kern<<<dim3(static_cast<unsigned>(T)), BLOCK, smem, st>>>(cand, W, T, n, K, ids, ld_out,
                                                            sat_word, status);
  return launch_status();
}

template <bool PACKED>
int dispatch_merge(const int32_t *cand, int W, int64_t T, int n, int K, int32_t *ids,
                   int64_t ld_out, int32_t *sat_word, int32_t *status, cudaStream_t st) {
  const int total = W * n;
  if (total <= 512 * 2)
    return launch_merge<512, 2, PACKED>(cand, W, T, n, K, ids, ld_out, sat_word, status, st);
  if (total <= 512 * 8)
    return launch_merge<512, 8, PACKED>(cand, W, T, n, K, ids, ld_out, sat_word, status, st);
  if (total <= 512 * 32)
    return launch_merge<512, 32, PACKED>(cand, W, T, n, K, ids, ld_out, sat_word, status, st);
  return launch_merge<1024, 32, PACKED>(cand, W, T, n, K, ids, ld_out, sat_word, status, st);
}

}  // namespace
}  // namespace satk

extern "C" int satk_dcp_pack(const uint16_t *logits_bf16, int64_t rows, int64_t S,
                             int64_t ld_logits, const int32_t *local_idx, int64_t ld_idx,
                             int32_t n, const int32_t *row_ends, int32_t *packed,
                             satk_stream_t stream) {
  using namespace satk;
  if (logits_bf16 == nullptr || local_idx == nullptr || packed == nullptr || rows < 0 ||
      S < 0 || ld_logits < S || n < 32 || n % 32 != 0 || ld_idx < n || rows > INT_MAX)
    return SATK_EINVAL;
  if (rows == 0) return SATK_OK;
  const int block = n < 512 ? n : 512;
  dcp_pack_kernel<<<dim3(static_cast<unsigned>(rows)), block, 0, as_stream(stream)>>>(
      logits_bf16, S, ld_logits, local_idx, ld_idx, n, row_ends, packed);
  return launch_status();
}

extern "C" int satk_dcp_merge_select(const void *cand, int format, int32_t W, int64_t T,
                                     int32_t n, int32_t k, int32_t *ids_out, int64_t ld_out,
                                     int32_t *sat_word, int32_t *status,
                                     satk_stream_t stream) {
  using namespace satk;
  if (cand == nullptr || ids_out == nullptr || W < 1 || T < 0 || n < 1 || k < 1 ||
      ld_out < k || T > INT_MAX || n % 32 != 0)
    return SATK_EINVAL;
  if (format == SATK_PACKED_BF16) {
    if (W > 16) return SATK_EINVAL;
  } else if (format == SATK_PAIRS_F32) {
    if (sat_word != nullptr || (reinterpret_cast<uintptr_t>(cand) & 7u) != 0) return SATK_EINVAL;
  } else {
    return SATK_EINVAL;
  }
  if ((int64_t)W * n > SATK_MERGE_MAX_CANDIDATES) return SATK_EUNSUPPORTED;
  if (T == 0) return SATK_OK;
  const int32_t *c = static_cast<const int32_t *>(cand);
  const cudaStream_t st = as_stream(stream);
  if (format == SATK_PACKED_BF16)
    return dispatch_merge<true>(c, W, T, n, k, ids_out, ld_out, sat_word, status, st);
  return dispatch_merge<false>(c, W, T, n, k, ids_out, ld_out, nullptr, status, st);
}
