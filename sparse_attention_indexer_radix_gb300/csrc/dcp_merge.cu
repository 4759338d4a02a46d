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
#include "satk_rows.cuh"

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
      if (satk_check(f < BLOCK * KPT, kDbgScratch)) sm.gid[f] = gid;
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

// ----------------------------------------------------- pairs, in place --
//
// The (score, global id) pairs of row t: flat candidate f = r * n + j sits
// at pair ((r * T + t) * n + j) of the rank-major buffer.  As for a row of
// logits: a sampled threshold, one filtered pass that records flat indices
// in per-warp list segments (each warp over its own stretch of the flat
// range, walked in runs that stay inside one rank), then the select on the
// list -- by score, and by global id among candidates tied with the K-th
// score.  A pair with id < 0 or a NaN score is empty.

__device__ __forceinline__ uint32_t pair_key(int2 p) {
  return p.y >= 0 ? key_f32(static_cast<uint32_t>(p.x)) : 0u;
}

// One pair, streamed (read once: no L1 allocation).
__device__ __forceinline__ int2 ldg_stream(const int2 *p) {
  int2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.s32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// Brings the n pairs of each rank for row t into L2 (one bulk prefetch per
// rank: the rank's slots of a row are contiguous, n * 8 bytes, 256-byte
// aligned when the buffer is 16-byte aligned and n % 32 == 0).
__device__ __forceinline__ void prefetch_row_l2(const int2 *cand, int W, int64_t T, int n,
                                                int64_t t) {
  for (int r = 0; r < W; ++r) {
    const int2 *p = cand + (static_cast<int64_t>(r) * T + t) * n;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                 :
                 : "l"(p), "r"(static_cast<uint32_t>(n) * 8u)
                 : "memory");
  }
}

constexpr int kPairsSPT = 4;  // sampled pairs per thread

template <int BLOCK, int SUB>
struct PairsSmem {
  ListSmem<BLOCK, SUB> ls;
  int2 samp[kPairsSPT * BLOCK];  // the row's sample, [q][thread]
};

// Asynchronous copies (no registers held) of this thread's kPairsSPT
// sampled pairs of row t into samp: the runs of 32 consecutive candidates
// spread evenly over the flat range, lane l taking candidate l of a run.
template <int BLOCK>
__device__ __forceinline__ void pairs_sample_async(int2 *samp, const int2 *cand, int total,
                                                   int64_t T, int n, int64_t t) {
  constexpr int NRUNS = BLOCK * kPairsSPT / 32;
#pragma unroll
  for (int q = 0; q < kPairsSPT; ++q) {
    const int run = warp_id() * kPairsSPT + q;
    const int f = (static_cast<int>((static_cast<int64_t>(run) * total) / NRUNS) & ~31) + lane_id();
    const int r = f / n;
    const int2 *src = cand + ((static_cast<int64_t>(r) * T + t) * n + (f - r * n));
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(samp + q * BLOCK + threadIdx.x));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// One row t of the pairs merge; `next` (or -1) is the row this CTA takes
// after it: once this row's pairs are read, the next row's pairs are
// prefetched into L2 and its sample is copied into shared memory, so that
// HBM keeps streaming while this row's list select runs.
template <int BLOCK, int SUB>
__device__ __forceinline__ void pairs_merge_row(PairsSmem<BLOCK, SUB> &ps,
                                                const int2 *__restrict__ cand, int W, int64_t T,
                                                int n, int K, int32_t *__restrict__ ids,
                                                int64_t ld_out, int32_t *__restrict__ status,
                                                const int64_t t, const int64_t next) {
  using SM = ListSmem<BLOCK, SUB>;
  SM &sm = ps.ls;
  constexpr int NW = BLOCK / 32;
  constexpr int CAP = SM::CAP;
  constexpr int SPT = kPairsSPT;
  constexpr int U = 8;  // steps loaded before any is taken
  const int lane = lane_id(), warp = warp_id();
  const int total = W * n;
  auto at = [&](int f) {  // pair of flat candidate f
    const int r = f / n;
    return cand + ((static_cast<int64_t>(r) * T + t) * n + (f - r * n));
  };
  zero_hist(sm.sel);
  if (threadIdx.x == 0) sm.flag = 0;
  __syncthreads();

  // ---- threshold
  const bool all = total <= CAP;
  float t0f = __uint_as_float(0xff800000u);
  if (!all) {
    constexpr int S = BLOCK * SPT;
    float v[SPT];  // sampled scores, NaN for an empty pair
    // this thread's own copies (issued by pairs_sample_async before the row)
    asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
    for (int q = 0; q < SPT; ++q) {
      const int2 pr = ps.samp[q * BLOCK + threadIdx.x];
      v[q] = pr.y >= 0 ? __int_as_float(pr.x) : __uint_as_float(0x7fc00000u);
    }
    const int r = sample_rank(K, S, total);
    bool ok;
    t0f = block_value_threshold<BLOCK, SPT>(v, r, sm.sel, ok);
    if (!ok) {  // block-uniform: an unusable value range, rank by ordered keys
#pragma unroll
      for (int q = 0; q < SPT; ++q)
        sm.key[warp * SUB + q * 32 + lane] = key_f32(__float_as_uint(v[q]));
      __syncwarp();
      const Sel sl = list_select<BLOCK>([&](int i) { return sm.key[i]; },
                                        Seg{warp * SUB, 32 * SPT}, r, sm.sel, 3);
      t0f = threshold_float<32>(sl.take_all ? 1u : sl.T);
    }
    __syncthreads();
  }

  // ---- filtered pass: keys and global ids of the kept pairs, flat order.
  // Lane l takes pair 32 s + l of each step (one 8-byte load per pair, a
  // warp's load is 256 contiguous bytes); a ballot per step gives every
  // kept pair its list position in flat order.  Each warp walks a stretch
  // of whole 32-pair steps; a step never crosses a rank (n % 32 == 0).
  const int nsteps = total / 32;
  const int per = (nsteps + NW - 1) / NW;
  const int s0 = min(nsteps, warp * per), s1 = min(nsteps, s0 + per);
  // shared addresses of this warp's key segment; a value sits CAP words
  // after its key
  const uint32_t lk = static_cast<uint32_t>(__cvta_generic_to_shared(sm.key + warp * SUB));
  static_assert(offsetof(SM, val) - offsetof(SM, key) == CAP * sizeof(uint32_t),
                "values follow the keys");
  const unsigned lt = (1u << lane) - 1u;
  int cnt = 0;
  bool room = true;  // warp-uniform: no step has passed SUB entries
  auto take = [&](const int2 v) {  // one step: 32 pairs, one per lane
    const bool keep = __int_as_float(v.x) >= t0f && v.y >= 0;
    const unsigned b = __ballot_sync(kFull, keep);
    const int nc = cnt + __popc(b);
    room = room && nc <= SUB;  // past SUB: counted only, the row takes the exact path
    const uint32_t a = lk + 4u * static_cast<uint32_t>(cnt + __popc(b & lt));
    // branch-free: the key and id stores are predicated on keep && room
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %0, 0;\n\t"
        "@p st.shared.b32 [%1], %2;\n\t"
        "@p st.shared.b32 [%1+%4], %3;\n\t}"
        :
        : "r"(static_cast<int>(keep && room)), "r"(a),
          "r"(key_f32_num(static_cast<uint32_t>(v.x))), "r"(v.y), "n"(CAP * 4)
        : "memory");
    cnt = nc;
  };
  for (int sr = s0; sr < s1;) {  // runs inside one rank (warp-uniform)
    const int f = sr * 32;
    const int r = f / n;
    const int send = min(s1, (r + 1) * (n / 32));
    const int2 *p = cand + ((static_cast<int64_t>(r) * T + t) * n + (f - r * n)) + lane;
    int sb = sr;
    for (; sb + U <= send; sb += U, p += 32 * U) {
      int2 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = ldg_stream(p + 32 * u);
#pragma unroll
      for (int u = 0; u < U; ++u) take(v[u]);
    }
    for (; sb < send; ++sb, p += 32) take(ldg_stream(p));
    sr = send;
  }
  if (next >= 0) {
    if (!all) pairs_sample_async<BLOCK>(ps.samp, cand, total, T, n, next);
    if (threadIdx.x == 0) prefetch_row_l2(cand, W, T, n, next);
  }
  if (cnt > SUB && lane == 0) sm.flag = 1;
  Seg sg{warp * SUB, min(cnt, SUB)};
  int listed;  // wtot[3]: its next writer (the list emit) is behind barriers
  block_warp_prefix<BLOCK>(sg.cnt, sm.sel.wtot[3], &listed);
  const bool ok = sm.flag == 0 && (all || listed >= K);
  if (!ok) {  // block-uniform: record every non-empty pair (two list passes
              // cannot hold more than CAP, so take the exact digit path)
    __syncthreads();
    // exact: histogram of the top digit over all pairs, then collect keys
    // at or above the threshold digit, narrowing while it would overflow
    uint32_t prefix = 0u;
    int pbits = 0, need = K, above = 0;
    bool take_all = false;
    while (true) {
      const int width = pbits == 0 ? 11 : min(11, 32 - pbits);
      const int shift = 32 - pbits - width;
      for (int f = threadIdx.x; f < total; f += BLOCK) {
        const uint32_t k = pair_key(__ldg(at(f)));
        if (k != 0u && (pbits == 0 || (k >> (32 - pbits)) == prefix))
          atomicAdd(sm.sel.hist + ((k >> shift) & ((1u << width) - 1u)), 1u);
      }
      __syncthreads();
      const PassOut p = find_threshold<BLOCK, 2048>(sm.sel, need);
      if (p.d < 0) {
        take_all = pbits == 0;
        break;
      }
      above += p.above;
      need -= p.above;
      prefix = (prefix << width) | static_cast<uint32_t>(p.d);
      pbits += width;
      if (above + p.cnt <= CAP || pbits == 32) break;
    }
    const uint32_t thr = take_all ? 1u : (prefix << (32 - pbits));
    // At full resolution a tie wider than the list: the order among equal
    // scores is the global id, so find the `need`-th smallest id among the
    // tied pairs (digits of ~id from the top, 11/11/10 bits) and keep the
    // tied pairs with an id at or below it.
    const bool limited = !take_all && pbits == 32;
    uint32_t gmax = 0u;  // with limited: the largest id kept among the ties
    if (limited) {
      uint32_t gp = 0u;
      int gbits = 0, gneed = need;
      while (gbits < 32) {
        const int width = min(11, 32 - gbits);
        const int shift = 32 - gbits - width;
        for (int f = threadIdx.x; f < total; f += BLOCK) {
          const int2 pr = __ldg(at(f));
          if (pair_key(pr) == thr) {
            const uint32_t u = 0xffffffffu - static_cast<uint32_t>(pr.y);
            if (gbits == 0 || (u >> (32 - gbits)) == gp)
              atomicAdd(sm.sel.hist + ((u >> shift) & ((1u << width) - 1u)), 1u);
          }
        }
        __syncthreads();
        const PassOut p = find_threshold<BLOCK, 2048>(sm.sel, gneed);
        if (p.d < 0) break;  // not reached: at least `need` pairs tie at thr
        gneed -= p.above;
        gp = (gp << width) | static_cast<uint32_t>(p.d);
        gbits += width;
      }
      gmax = 0xffffffffu - gp;
    }
    // collection (flat order) of the chosen pairs' keys and ids
    int run = 0, par = 0;
    for (int f0 = 0; f0 < total; f0 += BLOCK) {
      const int f = f0 + threadIdx.x;
      const int2 pr = f < total ? __ldg(at(f)) : make_int2(0, -1);
      const uint32_t k = pair_key(pr);
      const bool keep = limited ? (k > thr || (k == thr && static_cast<uint32_t>(pr.y) <= gmax))
                                : (k != 0u && k >= thr);
      const unsigned bk = __ballot_sync(kFull, keep);
      int tot2;
      const int wb = block_warp_prefix<BLOCK>(__popc(bk), sm.sel.wtot[par], &tot2);
      par ^= 1;
      const int pos = run + wb + __popc(bk & ((1u << lane) - 1u));
      if (keep && satk_check(pos < CAP, kDbgList)) {
        sm.key[pos] = k;
        sm.val[pos] = static_cast<uint32_t>(pr.y);
      }
      run += tot2;
    }
    __syncthreads();
    const int nlist = min(CAP, run);
    const int chunk = (nlist + NW - 1) / NW;
    const int b0 = min(nlist, warp * chunk);
    sg = Seg{b0, min(nlist, b0 + chunk) - b0};
  }
  __syncwarp();

  // ---- select: by score, then by global id among ties with the K-th
  int32_t *out = ids + t * ld_out;
  const bool dup = list_merge_emit<BLOCK, SUB>(
      sm, sg, K, [&](int pos, int32_t v) { out[pos] = v; }).dup;
  if (dup && status != nullptr && threadIdx.x == 0) atomicOr(status, SATK_STATUS_DUPLICATE_KEYS);
}

// Persistent: CTA b takes rows b, b + gridDim.x, ... (the grid is the
// resident CTA count, so each CTA's next row is known and prefetched).
template <int BLOCK, int SUB>
__global__ void __launch_bounds__(BLOCK, 1024 / BLOCK) pairs_merge_kernel(
    const int2 *__restrict__ cand, int W, int64_t T, int n, int K, int32_t *__restrict__ ids,
    int64_t ld_out, int32_t *__restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto &ps = *reinterpret_cast<PairsSmem<BLOCK, SUB> *>(smem_raw);
  if (W * n > ListSmem<BLOCK, SUB>::CAP)  // the first row's sample
    pairs_sample_async<BLOCK>(ps.samp, cand, W * n, T, n, blockIdx.x);
  for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
    const int64_t next = t + gridDim.x < T ? t + gridDim.x : -1;
    pairs_merge_row<BLOCK, SUB>(ps, cand, W, T, n, K, ids, ld_out, status, t, next);
    __syncthreads();  // this row's list and histogram reads before the next row's writes
  }
}

template <int SUB>
int launch_pairs(const int32_t *cand, int W, int64_t T, int n, int K, int32_t *ids,
                 int64_t ld_out, int32_t *status, cudaStream_t st) {
  constexpr int BLOCK = 256;
  auto kern = pairs_merge_kernel<BLOCK, SUB>;
  const size_t smem = sizeof(PairsSmem<BLOCK, SUB>);
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  const int64_t resident = resident_ctas(reinterpret_cast<const void *>(kern), BLOCK, smem);
  if (resident < 1) return SATK_ECUDA;
  const int64_t grid = T < resident ? T : resident;
  kern<<<dim3(static_cast<unsigned>(grid)), BLOCK, smem, st>>>(
      reinterpret_cast<const int2 *>(cand), W, T, n, K, ids, ld_out, status);
  return launch_status();
}

// ---------------------------------------------------- packed, list engine --
//
// The packed round-1 merge when every candidate fits the list (W * n <=
// 16 * kPackedSub): each warp copies its stretch of the flat range (32
// candidates per step, in flat order) into its list segment, skipping
// empty words -- no threshold is needed -- and the list merge select picks
// K.  tau16 is the ord16 of the smallest chosen key (0 below K chosen);
// rank r is saturated iff all its n words are listed with ord16 > tau16,
// counted per rank from the list.
constexpr int kPackedBlock = 512;
constexpr int kPackedSub = 512;

__global__ void __launch_bounds__(kPackedBlock) packed_merge_list_kernel(
    const int32_t *__restrict__ cand, int W, int64_t T, int n, int K,
    int32_t *__restrict__ ids, int64_t ld_out, int32_t *__restrict__ sat_word,
    int32_t *__restrict__ status) {
  constexpr int BLOCK = kPackedBlock, SUB = kPackedSub, NW = BLOCK / 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<ListSmem<BLOCK, SUB> *>(smem_raw);
  __shared__ int above[16];  // per rank: words listed with ord16 > tau16
  const int64_t t = blockIdx.x;
  const int lane = lane_id(), warp = warp_id();
  const unsigned lt = (1u << lane) - 1u;
  const int words = n + n / 32;
  const int nchunks = W * n / 32;  // n % 32 == 0
  const int per = (nchunks + NW - 1) / NW;
  const int c0 = min(nchunks, warp * per), c1 = min(nchunks, c0 + per);
  zero_hist(sm.sel);
  if (threadIdx.x < 16) above[threadIdx.x] = 0;
  __syncthreads();
  uint32_t *lk = sm.key + warp * SUB;
  uint32_t *lv = sm.val + warp * SUB;
  int cnt = 0;
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  // per * 32 <= SUB: no overflow.  The words of up to kLoadBatch chunks
  // are loaded before any is listed, so their latencies overlap.
  constexpr int kLoadBatch = 8;
  for (int cb = c0; cb < c1; cb += kLoadBatch) {
    uint32_t wv[kLoadBatch], pv[kLoadBatch];
    int rv[kLoadBatch], jv[kLoadBatch];
#pragma unroll
    for (int q = 0; q < kLoadBatch; ++q) {
      const int c = cb + q;
      wv[q] = 0u;
      pv[q] = 0u;
      rv[q] = 0;
      jv[q] = 0;
      if (c < c1) {
        const int fb = c * 32;
        const int r = fb / n, j = fb - r * n + lane;
        const int32_t *row = cand + ((int64_t)r * T + t) * words;
        wv[q] = static_cast<uint32_t>(__ldg(row + j));
        pv[q] = static_cast<uint32_t>(__ldg(row + n + ((j - lane) >> 5)));
        rv[q] = r;
        jv[q] = j;
      }
    }
#pragma unroll
    for (int q = 0; q < kLoadBatch; ++q) {
      if (cb + q < c1) {  // warp-uniform
        const uint32_t key = bprime_list_key(wv[q]);
        const unsigned b = __ballot_sync(kFull, key != 0u);
        if (key != 0u) {
          const int pos = cnt + __popc(b & lt);
          if (satk_check(pos < SUB, kDbgList)) {
            lk[pos] = key;
            lv[pos] = bprime_local(wv[q], pv[q], jv[q]) * (uint32_t)W + (uint32_t)rv[q];
          }
          kmn = min(kmn, key);
          kmx = max(kmx, key);
        }
        cnt += __popc(b);
      }
    }
  }
  const WarpStats st{cnt, __reduce_min_sync(kFull, kmn), __reduce_max_sync(kFull, kmx)};
  __syncthreads();
  int32_t *out = ids + t * ld_out;
  const Seg sg{warp * SUB, cnt};
  const ListMergeOut m = list_merge_emit<BLOCK, SUB, true>(
      sm, sg, K,
      [&](int pos, int32_t v) {
        if ((unsigned)pos < (unsigned)K) out[pos] = v;
      },
      st);
  int bits = m.dup ? SATK_STATUS_DUPLICATE_KEYS : 0;
  if (sat_word != nullptr) {
    const uint32_t tau = (m.nsel == K) ? (m.kmin - 1u) : 0u;  // list keys are ord16 + 1
    for (int j = 0; j < sg.rounds(); ++j) {
      const int i = j * 32 + lane;
      if (i < sg.cnt && sm.key[sg.base + i] > tau + 1u)
        atomicAdd(&above[sm.val[sg.base + i] % static_cast<uint32_t>(W)], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint32_t mask = 0u;
      for (int q = 0; q < W; ++q)
        if (above[q] == n) mask |= 1u << q;
      const int slots = (K - 1) / n;
      if (__popc(mask) > slots) {
        mask = 0u;  // more saturated ranks than slots: keep round 1
        bits |= SATK_STATUS_SLOTS_EXCEEDED;
      }
      sat_word[t] = static_cast<int32_t>((mask << 16) | tau);
    }
  }
  if (bits != 0 && status != nullptr && threadIdx.x == 0) atomicOr(status, bits);
}

int launch_packed_list(const int32_t *cand, int W, int64_t T, int n, int K, int32_t *ids,
                       int64_t ld_out, int32_t *sat_word, int32_t *status, cudaStream_t st) {
  auto kern = packed_merge_list_kernel;
  const size_t smem = sizeof(ListSmem<kPackedBlock, kPackedSub>);
  if (!allow_smem(kern, smem)) return SATK_ECUDA;
  kern<<<dim3(static_cast<unsigned>(T)), kPackedBlock, smem, st>>>(cand, W, T, n, K, ids, ld_out,
                                                                   sat_word, status);
  return launch_status();
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
  if (PACKED && total <= (kPackedBlock / 32) * kPackedSub)
    return launch_packed_list(cand, W, T, n, K, ids, ld_out, sat_word, status, st);
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
    if (sat_word != nullptr || (reinterpret_cast<uintptr_t>(cand) & 15u) != 0) return SATK_EINVAL;
  } else {
    return SATK_EINVAL;
  }
  if ((int64_t)W * n > SATK_MERGE_MAX_CANDIDATES) return SATK_EUNSUPPORTED;
  if (T == 0) return SATK_OK;
  const int32_t *c = static_cast<const int32_t *>(cand);
  const cudaStream_t st = as_stream(stream);
  if (format == SATK_PACKED_BF16)
    return dispatch_merge<true>(c, W, T, n, k, ids_out, ld_out, sat_word, status, st);
  // pairs: the list holds 8 warps x SUB candidates (4096 up to K = 2048)
  if (k <= 2048) return launch_pairs<512>(c, W, T, n, k, ids_out, ld_out, status, st);
  return launch_pairs<1024>(c, W, T, n, k, ids_out, ld_out, status, st);
}
