// satk_rows.cuh -- exact top-K of one row, two ways.
//
// Semantics follow [Perf][DSA] Use DeepSelect for eligible sparse-indexer
// prefill chunks (vLLM PR #57206), Purpose and Test Plan: row i's
// candidates are its columns [0, end_i), the output is a preallocated
// (possibly strided) int32 row padded with -1.  The id layout is the one of
// push_local_topk's emit pass on the vLLM API page
// vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels: ids strictly above
// the K-th score in ascending column order, then the ids tied with it
// (lowest columns first) up to K.
//
// topk_reg_row   : the whole valid row is held in registers (one 16-byte
//                  load per VEC columns), radix select + ordered emit in
//                  place.  One HBM read, no re-reads.
// topk_stream_row: rows longer than the registers hold.  Pass 1 streams the
//                  row from HBM once and builds the top-digit histogram; the
//                  collection pass re-reads it (from L2 while the row is
//                  resident) and compacts, in column order, every candidate
//                  at or above the threshold digit into a shared-memory list
//                  of at most CAP entries; the register engine then runs on
//                  the list.  If the threshold digit holds too many
//                  candidates for the list, further digit passes narrow it
//                  first; at full key resolution only the first `need`
//                  entries of the tied key are kept, so the list never
//                  exceeds K.
#pragma once

#include <type_traits>

#include "satk_device.cuh"

namespace satk {

// ---------------------------------------------------------------- in regs --

template <typename T, int BLOCK, int KPT, bool VECLOAD, bool AGG, class Put, class Fill>
__device__ __forceinline__ void topk_reg_row(const T *__restrict__ xr, int end, int K, Put put,
                                             Fill fill, SelectSmem<BLOCK> &sm) {
  constexpr int VEC = VECLOAD ? KeyOf<T>::kVec : 1;
  constexpr int KB = KeyOf<T>::kBits;
  static_assert(KPT % VEC == 0, "KPT must hold whole vectors");
  uint32_t keys[KPT];
  if constexpr (VECLOAD) {
    uint4 raw[KPT / VEC];
#pragma unroll
    for (int g = 0; g < KPT / VEC; ++g) {
      const int c0 = flat_pos<KPT, VEC>(g * VEC);
      if (c0 + VEC <= end) raw[g] = ldg_stream(xr + c0);
    }
#pragma unroll
    for (int g = 0; g < KPT / VEC; ++g) {
      const int c0 = flat_pos<KPT, VEC>(g * VEC);
      if (c0 + VEC <= end) {
        KeyOf<T>::vec(raw[g], &keys[g * VEC]);
      } else {
#pragma unroll
        for (int s = 0; s < VEC; ++s)
          keys[g * VEC + s] = (c0 + s < end) ? KeyOf<T>::scalar(xr + c0 + s) : 0u;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < KPT; ++i) {
      const int c = flat_pos<KPT, 1>(i);
      keys[i] = c < end ? KeyOf<T>::scalar(xr + c) : 0u;
    }
  }
  auto gk = [&](int i) { return keys[i]; };
  const Sel sel = radix_select<BLOCK, KPT, KB, AGG>(gk, K, sm);
  emit_topk_layout<BLOCK, KPT, VEC>(
      gk, [&](int pos, int i) { put(pos, keys[i], flat_pos<KPT, VEC>(i)); }, fill, K, sel, sm);
}

// ------------------------------------------------------------- streaming --

template <int BLOCK, int CAP>
struct StreamSmem {
  SelectSmem<BLOCK> sel;
  uint32_t lkey[CAP];
  int32_t lcol[CAP];
};

// Visits the row [0, end) tile by tile with a warp-contiguous mapping: in a
// tile of BLOCK*U vectors, warp w owns vectors [w*32*U, (w+1)*32*U) and
// lane l reads vector w*32*U + u*32 + l at step u (coalesced per step).
// body(kk, colbase) gets the lane's U*VEC keys (0 past the end) and the
// column of kk[u*VEC] for each u via colbase[u]; every thread of the block
// calls body the same number of times (block-uniform trip count), so body
// may use warp collectives and barriers.  A last call with U=1 and VEC=1
// semantics handles the < VEC ragged columns (warp 0 lanes only).
template <typename T, int BLOCK, int U, bool VECLOAD, class Body, class TailBody>
__device__ __forceinline__ void for_row_tiles(const T *__restrict__ xr, int end, Body body,
                                              TailBody tail) {
  constexpr int VEC = VECLOAD ? KeyOf<T>::kVec : 1;
  const int lane = lane_id(), warp = warp_id();
  const int nvec = end / VEC;  // whole vectors
  for (int tile = 0; tile < nvec; tile += BLOCK * U) {
    uint32_t kk[U * VEC];
    int col[U];
    if constexpr (VECLOAD) {
      uint4 raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vi = tile + warp * (32 * U) + u * 32 + lane;
        col[u] = vi * VEC;
        if (vi < nvec) raw[u] = ldg_stream(xr + (size_t)vi * VEC);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vi = tile + warp * (32 * U) + u * 32 + lane;
        if (vi < nvec) {
          KeyOf<T>::vec(raw[u], &kk[u * VEC]);
        } else {
#pragma unroll
          for (int s = 0; s < VEC; ++s) kk[u * VEC + s] = 0u;
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = tile + warp * (32 * U) + u * 32 + lane;
        col[u] = c;
        kk[u] = c < end ? KeyOf<T>::scalar(xr + c) : 0u;
      }
    }
    body(kk, col);
  }
  if constexpr (VECLOAD) {
    const int t0 = nvec * VEC;
    if (t0 < end) {  // block-uniform
      const int c = t0 + lane;
      const bool mine = warp == 0 && c < end;
      const uint32_t k = mine ? KeyOf<T>::scalar(xr + c) : 0u;
      tail(k, c);
    }
  }
}

template <typename T, int BLOCK, int LKPT, bool VECLOAD, bool AGG, class Put, class Fill>
__device__ void topk_stream_row(const T *__restrict__ xr, int end, int K, Put put, Fill fill,
                                StreamSmem<BLOCK, BLOCK * LKPT> &sm) {
  constexpr int VEC = VECLOAD ? KeyOf<T>::kVec : 1;
  constexpr int U = VECLOAD ? 4 : 8;
  constexpr int KB = KeyOf<T>::kBits;
  constexpr int CAP = BLOCK * LKPT;
  constexpr int NK = U * VEC;
  static_assert(BLOCK * U * VEC < 65536, "tile counts must fit 16 bits");
  SelectSmem<BLOCK> &ss = sm.sel;
  const int lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;

  // ---- pass 1: top-digit histogram (HBM read)
  for_row_tiles<T, BLOCK, U, VECLOAD>(
      xr, end,
      [&](const uint32_t *kk, const int *) {
#pragma unroll
        for (int j = 0; j < NK; ++j) hist_add<AGG>(ss.hist, kk[j] >> 21, kk[j] != 0u);
      },
      [&](uint32_t k, int) { hist_add<AGG>(ss.hist, k >> 21, k != 0u); });
  __syncthreads();
  PassOut p = find_threshold<BLOCK, 2048>(ss, K);

  uint32_t thr;
  bool limited = false;
  int need = K;
  if (p.d < 0) {
    thr = 1u;  // fewer than K valid: every valid column
  } else {
    uint32_t prefix = (uint32_t)p.d;
    int pbits = 11;
    int above = p.above;
    int cnt = p.cnt;
    need = K - above;
    // ---- narrow the threshold digit until its candidates fit the list
    while (above + cnt > CAP && pbits < KB) {
      const int width = (KB - pbits >= 11) ? 11 : (KB - pbits);
      const int shift = 32 - pbits - width;
      const uint32_t dmask = (1u << width) - 1u;
      const int pb = pbits;
      const uint32_t pf = prefix;
      auto visit = [&](uint32_t k) {
        hist_add<AGG>(ss.hist, (k >> shift) & dmask, k != 0u && (k >> (32 - pb)) == pf);
      };
      for_row_tiles<T, BLOCK, U, VECLOAD>(
          xr, end,
          [&](const uint32_t *kk, const int *) {
#pragma unroll
            for (int j = 0; j < NK; ++j) visit(kk[j]);
          },
          [&](uint32_t k, int) { visit(k); });
      __syncthreads();
      if (width == 11)
        p = find_threshold<BLOCK, 2048>(ss, need);
      else if (width == 10)
        p = find_threshold<BLOCK, 1024>(ss, need);
      else
        p = find_threshold<BLOCK, 32>(ss, need);  // bf16 keys: 5 low bits
      above += p.above;
      need -= p.above;
      cnt = p.cnt;
      prefix = (prefix << width) | (uint32_t)p.d;
      pbits += width;
    }
    thr = prefix << (32 - pbits);
    limited = above + cnt > CAP;  // full resolution, tie too wide: keep `need`
  }

  // ---- collection: ordered compaction of the candidates into the list
  int runA = 0, runB = 0;  // block-uniform running counts
  int tile_par = 0;
  auto collect = [&](const uint32_t *kk, const int *col, auto nk_tag, auto vec_tag) {
    constexpr int NKT = decltype(nk_tag)::value;
    constexpr int VT = decltype(vec_tag)::value;
    int ca = 0, cb = 0;
#pragma unroll
    for (int j = 0; j < NKT; ++j) {
      const uint32_t k = kk[j];
      const bool a = limited ? (k > thr) : (k >= thr);
      const bool b = limited && k == thr;
      ca += __popc(__ballot_sync(kFull, a));
      cb += __popc(__ballot_sync(kFull, b));
    }
    int tot;
    const unsigned base =
        (unsigned)block_warp_prefix<BLOCK>((ca << 16) | cb, ss.wtot[tile_par], &tot);
    tile_par ^= 1;
    int ra = runA + (int)(base >> 16), rb = runB + (int)(base & 0xffffu);
#pragma unroll
    for (int u = 0; u < NKT / VT; ++u) {
      unsigned ba[VT], bb[VT];
      int pa = 0, pbb = 0;
#pragma unroll
      for (int s = 0; s < VT; ++s) {
        const uint32_t k = kk[u * VT + s];
        ba[s] = __ballot_sync(kFull, limited ? (k > thr) : (k >= thr));
        bb[s] = __ballot_sync(kFull, limited && k == thr);
        pa += __popc(ba[s] & lt);
        pbb += __popc(bb[s] & lt);
      }
#pragma unroll
      for (int s = 0; s < VT; ++s) {
        const uint32_t k = kk[u * VT + s];
        const bool a = (ba[s] >> lane) & 1u;
        const bool b = (bb[s] >> lane) & 1u;
        int pos = -1;
        if (a) pos = ra + pa + (limited ? min(rb + pbb, need) : 0);
        if (b && rb + pbb < need) pos = ra + pa + rb + pbb;
        if (pos >= 0 && pos < CAP) {
          sm.lkey[pos] = k;
          sm.lcol[pos] = col[u] + s;
        }
        pa += a;
        pbb += b;
      }
#pragma unroll
      for (int s = 0; s < VT; ++s) {
        ra += __popc(ba[s]);
        rb += __popc(bb[s]);
      }
    }
    runA += (int)((unsigned)tot >> 16);
    runB += (int)((unsigned)tot & 0xffffu);
  };
  using IntC1 = std::integral_constant<int, 1>;
  using IntCNK = std::integral_constant<int, NK>;
  using IntCV = std::integral_constant<int, VEC>;
  for_row_tiles<T, BLOCK, U, VECLOAD>(
      xr, end, [&](const uint32_t *kk, const int *col) { collect(kk, col, IntCNK{}, IntCV{}); },
      [&](uint32_t k, int c) {
        uint32_t kk1[1] = {k};
        int c1[1] = {c};
        collect(kk1, c1, IntC1{}, IntC1{});
      });
  __syncthreads();
  const int nlist = min(CAP, runA + (limited ? min(runB, need) : 0));

  // ---- the register engine on the list (column order = list order)
  uint32_t keys[LKPT];
#pragma unroll
  for (int i = 0; i < LKPT; ++i) {
    const int f = flat_pos<LKPT, 1>(i);
    keys[i] = f < nlist ? sm.lkey[f] : 0u;
  }
  auto gk = [&](int i) { return keys[i]; };
  const Sel sel = radix_select<BLOCK, LKPT, KB, AGG>(gk, K, ss);
  emit_topk_layout<BLOCK, LKPT, 1>(
      gk, [&](int pos, int i) { put(pos, keys[i], sm.lcol[flat_pos<LKPT, 1>(i)]); }, fill, K,
      sel, ss);
}

}  // namespace satk
