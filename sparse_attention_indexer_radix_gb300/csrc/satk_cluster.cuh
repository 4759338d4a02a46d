// satk_cluster.cuh -- the row path split over a thread-block cluster, for
// workloads of few long rows.
//
// With fewer rows than about twice the CTAs the GPU holds, one CTA per row
// leaves SMs idle in the last wave (and, with very few rows, in every wave).
// Here a cluster of C CTAs shares a row: CTA c streams the c-th contiguous
// slice of the row's columns into its own shared-memory list, and the
// selects run over the union of the C lists, each CTA adding the other
// CTAs' histograms and scalars through distributed shared memory (no
// multicast, no global scratch).  Every CTA computes the same thresholds, so
// each writes its own entries of the output directly:
//  1. T0 from the union of the C slices' samples (cluster select);
//  2. each CTA's filtered pass over its slice (satk_rows.cuh);
//  3. the exact select over the union of the lists (cluster select);
//  4. the ordered emit: CTA c's entries above the K-th key follow those of
//     CTAs < c, and the same for the tied entries, so the output is in
//     column order as on the other paths.
// A list overflow anywhere, or fewer than K candidates in all, sends the row
// to CTA 0 alone, which redoes it exactly over the whole row (the CTA
// path's exact pass); the other CTAs then only wait at the final barrier.
//
// Every cluster barrier is reached by all threads of all C CTAs the same
// number of times: each branch around one depends only on values that are
// identical across the cluster (the row end, cluster-wide sums and
// thresholds).
#pragma once

#include <cooperative_groups.h>

#include "satk_rows.cuh"

namespace satk {

namespace cg = cooperative_groups;

// Slots of the per-CTA values the cluster reads; each is written once per
// row, so no slot is rewritten while another CTA may still read it.
enum ClusterSlot : int {
  kPubSampleStats = 0,  // n, min, max of the sample keys
  kPubFlag = 3,         // list overflow
  kPubCount = 4,        // list entries
  kPubListStats = 5,    // n, min, max of the list keys
  kPubMinAbove = 8,     // smallest key >= T
  kPubCountA = 9,       // entries above the K-th key
  kPubCountB = 10,      // entries equal to it
  kPubSampleRange = 12, // smallest, largest sampled value (ordered ints)
  kPubSlots = 14
};

template <int BLOCK, int SUB>
struct ClusterSmem {
  ListSmem<BLOCK, SUB> ls;
  uint32_t pub[kPubSlots];
};

// The word at `local` in CTA c of the cluster.
__device__ __forceinline__ uint32_t cluster_word(cg::cluster_group &cl, uint32_t *local, int c) {
  return *cl.map_shared_rank(local, c);
}

// find_threshold over the sum of the C CTAs' histograms; does not zero them
// (their owners do, after a cluster barrier).  Ends with a block barrier.
template <int BLOCK, int NB, int C>
__device__ __forceinline__ PassOut cluster_find_threshold(cg::cluster_group &cl,
                                                          SelectSmem<BLOCK> &sm, int need) {
  static_assert(NB % 32 == 0, "bins come in groups of 32");
  constexpr int NW = BLOCK / 32;
  constexpr int NG = NB / 32;
  constexpr int GPW = (NG + NW - 1) / NW;
  const int lane = lane_id(), warp = warp_id();
  uint32_t cnt[GPW];
  int gs[GPW];
  int wsum = 0;
#pragma unroll
  for (int q = 0; q < GPW; ++q) {
    const int g = warp * GPW + q;
    cnt[q] = 0u;
    if (g < NG) {
      const int bin = NB - 1 - (g * 32 + lane);
#pragma unroll
      for (int c = 0; c < C; ++c) cnt[q] += cluster_word(cl, sm.hist + bin, c);
    }
    gs[q] = static_cast<int>(__reduce_add_sync(kFull, cnt[q]));
    wsum += gs[q];
  }
  int total;
  const int wbase = block_warp_prefix<BLOCK>(wsum, sm.wtot[0], &total);
  if (total >= need && wbase < need && wbase + wsum >= need) {  // warp-uniform
    int cum = wbase;
#pragma unroll
    for (int q = 0; q < GPW; ++q) {
      if (cum < need && cum + gs[q] >= need) {  // warp-uniform
        const int incl = warp_incl_scan(static_cast<int>(cnt[q]));
        const int before = cum + incl - static_cast<int>(cnt[q]);
        if (before < need && before + static_cast<int>(cnt[q]) >= need) {
          sm.scal[0] = NB - 1 - ((warp * GPW + q) * 32 + lane);
          sm.scal[1] = before;
          sm.scal[2] = static_cast<int>(cnt[q]);
        }
      }
      cum += gs[q];
    }
  }
  __syncthreads();
  PassOut p;
  p.total = total;
  if (total < need) {
    p.d = -1;
    p.above = 0;
    p.cnt = 0;
  } else {
    p.d = sm.scal[0];
    p.above = sm.scal[1];
    p.cnt = sm.scal[2];
  }
  return p;
}

// list_select (satk_list.cuh) over the union of the C CTAs' lists: the K
// largest of the non-zero keys gk(i) of every CTA's segments.  `slot` is
// the first of three pub slots for the count and key range; lz, the low
// key bits known to be zero (bf16 keys).  Identical result in every CTA of
// the cluster.
template <int BLOCK, int SUB, int C, class GetKey>
__device__ Sel cluster_list_select(cg::cluster_group &cl, GetKey gk, const Seg &sg, int K,
                                   ClusterSmem<BLOCK, SUB> &cs, int max_passes, int slot,
                                   WarpStats pre = stats_unknown(), int lz = 0) {
  SelectSmem<BLOCK> &sm = cs.ls.sel;
  const int lane = lane_id();
  uint32_t mn = 0xffffffffu, mx = 0u;
  int n = 0;
  if (pre.known()) {
    n = pre.n;
    mn = pre.mn;
    mx = pre.mx;
  } else {
    for (int j = 0; j < sg.rounds(); ++j) {
      const int i = j * 32 + lane;
      const uint32_t k = i < sg.cnt ? gk(sg.base + i) : 0u;
      if (k != 0u) {
        mn = min(mn, k);
        mx = max(mx, k);
        ++n;
      }
    }
    mn = __reduce_min_sync(kFull, mn);
    mx = __reduce_max_sync(kFull, mx);
    n = static_cast<int>(__reduce_add_sync(kFull, static_cast<unsigned>(n)));
  }
  if (lane == 0) {
    sm.red[warp_id()] = mn;
    sm.wtot[1][warp_id()] = static_cast<int>(mx);
    sm.wtot[2][warp_id()] = n;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t bn = 0u, bmn = 0xffffffffu, bmx = 0u;
#pragma unroll
    for (int w = 0; w < BLOCK / 32; ++w) {
      bmn = min(bmn, sm.red[w]);
      bmx = max(bmx, static_cast<uint32_t>(sm.wtot[1][w]));
      bn += static_cast<uint32_t>(sm.wtot[2][w]);
    }
    cs.pub[slot] = bn;
    cs.pub[slot + 1] = bmn;
    cs.pub[slot + 2] = bmx;
  }
  cl.sync();  // every CTA's count and range published
  int total = 0;
  mn = 0xffffffffu;
  mx = 0u;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    total += static_cast<int>(cluster_word(cl, &cs.pub[slot], c));
    mn = min(mn, cluster_word(cl, &cs.pub[slot + 1], c));
    mx = max(mx, cluster_word(cl, &cs.pub[slot + 2], c));
  }
  Sel r;
  r.tie = false;
  r.take_all = false;
  r.total = total;
  if (total < K) {
    r.take_all = true;
    r.T = 1u;
    r.need = 0;
    return r;
  }
  const uint32_t span = (mx - mn) >> lz;
  const int b = span == 0u ? 0 : 32 - __clz(span);
  int need = K;
  uint32_t prefix = 0u;
  int pbits = 0;
  // 8-bit digits: 256 bins, one per thread of the first 256, so each thread
  // reads C remote words per pass, all in flight at once (11-bit digits
  // made it 8 x C dependent remote reads per thread per pass)
  const int digit = kListDigitShort;
  while (pbits < b) {  // cluster-uniform: b, digit, need and the digits agree
    const int width = (b - pbits) < digit ? (b - pbits) : digit;
    const int shift = b - pbits - width;
    const uint32_t dmask = (1u << width) - 1u;
    for (int j = 0; j < sg.rounds(); ++j) {
      const int i = j * 32 + lane;
      const uint32_t k = i < sg.cnt ? gk(sg.base + i) : 0u;
      if (k != 0u) {
        const uint32_t rel = (k - mn) >> lz;
        if (pbits == 0 || (rel >> (shift + width)) == prefix)
          atomicAdd(sm.hist + ((rel >> shift) & dmask), 1u);
      }
    }
    cl.sync();  // every CTA's histogram complete
    const PassOut p = cluster_find_threshold<BLOCK, (1 << kListDigitShort), C>(cl, sm, need);
    cl.sync();  // every CTA done reading the histograms
    for (int i = threadIdx.x; i <= static_cast<int>(dmask); i += BLOCK) sm.hist[i] = 0u;
    __syncthreads();
    need -= p.above;
    prefix = (prefix << width) | static_cast<uint32_t>(p.d);
    pbits += width;
    if (p.cnt == need || --max_passes == 0) {
      r.T = mn + ((prefix << shift) << lz);
      r.need = need;
      return r;
    }
  }
  r.T = mn + (prefix << lz);
  r.need = need;
  r.tie = true;
  return r;
}

// Select over the union of the lists and the ordered emit: put(pos, key,
// col) for the entries above the K-th key in (CTA, list) order, then for
// the entries equal to it up to K; fill(pos) for [n, K) when only n < K
// candidates exist in all.  col0 is this CTA's first column (list values
// are slice-relative).
template <int BLOCK, int SUB, int C, class Put, class Fill>
__device__ void cluster_topk_emit(cg::cluster_group &cl, ClusterSmem<BLOCK, SUB> &cs,
                                  const Seg &sg, int K, int col0, Put put, Fill fill,
                                  WarpStats pre, int lz) {
  ListSmem<BLOCK, SUB> &sm = cs.ls;
  const int crank = static_cast<int>(cl.block_rank());
  const int lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  auto gk = [&](int i) { return sm.key[i]; };
  const Sel sel =
      cluster_list_select<BLOCK, SUB, C>(cl, gk, sg, K, cs, 8, kPubListStats, pre, lz);
  uint32_t v;
  if (sel.take_all) {
    v = 0u;  // every entry is above
  } else if (sel.tie) {
    v = sel.T;
  } else {  // exactly K keys >= T: v is the smallest of them
    uint32_t m = 0xffffffffu;
    for (int j = 0; j < sg.rounds(); ++j) {
      const int i = j * 32 + lane;
      const uint32_t k = i < sg.cnt ? sm.key[sg.base + i] : 0u;
      if (k >= sel.T) m = min(m, k);
    }
    m = block_min<BLOCK>(m, sm.sel);
    if (threadIdx.x == 0) cs.pub[kPubMinAbove] = m;
    cl.sync();
    v = 0xffffffffu;
#pragma unroll
    for (int c = 0; c < C; ++c) v = min(v, cluster_word(cl, &cs.pub[kPubMinAbove], c));
  }
  // counting walk (ballots kept in the zero histogram, as list_emit)
  uint32_t *bal = sm.sel.hist + warp_id() * 64;
  const int R = sg.rounds();
  int ca = 0, cb = 0;
  for (int j = 0; j < R; ++j) {
    const int i = j * 32 + lane;
    const uint32_t k = i < sg.cnt ? sm.key[sg.base + i] : 0u;
    const unsigned ba = __ballot_sync(kFull, k != 0u && k > v);
    const unsigned bb = __ballot_sync(kFull, k != 0u && k == v);
    if (lane == 0 && j < 32) {
      bal[2 * j] = ba;
      bal[2 * j + 1] = bb;
    }
    ca += __popc(ba);
    cb += __popc(bb);
  }
  int btot;
  const unsigned wbase =
      (unsigned)block_warp_prefix<BLOCK>((ca << 16) | cb, sm.sel.wtot[3], &btot);
  if (threadIdx.x == 0) {
    cs.pub[kPubCountA] = (unsigned)btot >> 16;
    cs.pub[kPubCountB] = (unsigned)btot & 0xffffu;
  }
  cl.sync();  // every CTA's counts published
  int offA = 0, offB = 0, totA = 0;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int a = static_cast<int>(cluster_word(cl, &cs.pub[kPubCountA], c));
    totA += a;
    if (c < crank) {
      offA += a;
      offB += static_cast<int>(cluster_word(cl, &cs.pub[kPubCountB], c));
    }
  }
  int ra = offA + (int)(wbase >> 16), rb = totA + offB + (int)(wbase & 0xffffu);
  for (int j = 0; j < R; ++j) {
    const int i = j * 32 + lane;
    unsigned ba, bb;
    if (j < 32) {
      ba = bal[2 * j];
      bb = bal[2 * j + 1];
    } else {
      const uint32_t k = i < sg.cnt ? sm.key[sg.base + i] : 0u;
      ba = __ballot_sync(kFull, k != 0u && k > v);
      bb = __ballot_sync(kFull, k != 0u && k == v);
    }
    if ((ba >> lane) & 1u) {
      const int pos = ra + __popc(ba & lt);
      if ((unsigned)pos < (unsigned)K)
        put(pos, sm.key[sg.base + i], static_cast<int>(sm.val[sg.base + i]) + col0);
    }
    if ((bb >> lane) & 1u) {
      const int pos = rb + __popc(bb & lt);
      if ((unsigned)pos < (unsigned)K)
        put(pos, sm.key[sg.base + i], static_cast<int>(sm.val[sg.base + i]) + col0);
    }
    ra += __popc(ba);
    rb += __popc(bb);
  }
  __syncwarp();
  bal[lane] = 0u;
  bal[lane + 32] = 0u;
  __syncthreads();
  if (sel.take_all && crank == C - 1)
    for (int q = totA + static_cast<int>(threadIdx.x); q < K; q += BLOCK) fill(q);
}

// The whole row on a cluster of C CTAs (this CTA is rank cl.block_rank()):
// T0 of a row split over the cluster from the union of the C slices'
// samples (kRowSample runs of 32 columns per warp, spread over each slice,
// held in registers): the sampled values' range is exchanged once, every
// CTA builds a value-linear 256-bin histogram of its own samples, and the
// sum of the C histograms read through distributed shared memory gives the
// bin of the r-th largest value (a finer round inside a bin holding more
// than 32 samples); T0 is that bin's lower edge moved down by a few ulps,
// on T's grid.  Three cluster barriers (five with the finer round) where
// the ordered-key digits of the union take up to seven.  Every branch
// depends only on cluster-wide values, so all CTAs take the same number of
// barriers.  ok = false (cluster-uniform, after one barrier) when the
// range is not usable (an infinity, a single value): the caller ranks the
// samples by ordered keys.  -inf when fewer than r values are valid.  The
// histogram is zero on entry and on return.
template <typename T, int BLOCK, int SUB, int C>
__device__ float cluster_value_threshold(cg::cluster_group &cl, const T *__restrict__ xs,
                                         int send, int r, ClusterSmem<BLOCK, SUB> &cs,
                                         bool &ok) {
  constexpr int SPT = kRowSample;
  constexpr int NW = BLOCK / 32;
  constexpr int NRUNS = BLOCK * SPT / 32;
  SelectSmem<BLOCK> &sel = cs.ls.sel;
  const int lane = lane_id(), warp = warp_id();
  float v[SPT];
#pragma unroll
  for (int q = 0; q < SPT; ++q) {
    const int run = warp * SPT + q;
    const int start = static_cast<int>((static_cast<int64_t>(run) * send) / NRUNS) & ~31;
    v[q] = as_float<T>(load_raw(xs + start + lane));
  }
  float mn = __uint_as_float(0x7f800000u), mx = __uint_as_float(0xff800000u);
#pragma unroll
  for (int q = 0; q < SPT; ++q) {
    mn = fminf(mn, v[q]);  // NaN ignored
    mx = fmaxf(mx, v[q]);
  }
  const int wmn = __reduce_min_sync(kFull, float_order(mn));
  const int wmx = __reduce_max_sync(kFull, float_order(mx));
  if (lane == 0) {
    sel.wtot[1][warp] = wmn;
    sel.wtot[2][warp] = wmx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int bmn = sel.wtot[1][0], bmx = sel.wtot[2][0];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      bmn = min(bmn, sel.wtot[1][w]);
      bmx = max(bmx, sel.wtot[2][w]);
    }
    cs.pub[kPubSampleRange] = static_cast<uint32_t>(bmn);
    cs.pub[kPubSampleRange + 1] = static_cast<uint32_t>(bmx);
  }
  cl.sync();  // every CTA's range published
  int imn = static_cast<int>(cluster_word(cl, &cs.pub[kPubSampleRange], 0));
  int imx = static_cast<int>(cluster_word(cl, &cs.pub[kPubSampleRange + 1], 0));
#pragma unroll
  for (int c = 1; c < C; ++c) {
    imn = min(imn, static_cast<int>(cluster_word(cl, &cs.pub[kPubSampleRange], c)));
    imx = max(imx, static_cast<int>(cluster_word(cl, &cs.pub[kPubSampleRange + 1], c)));
  }
  mn = float_of_order(imn);
  mx = float_of_order(imx);
  ok = true;
  const float ninf = __uint_as_float(0xff800000u);
  if (mx < mn) return ninf;  // no valid sample in the row (cluster-uniform)
  const float span = mx - mn;
  if (!(span > 0.f) || !(span < __uint_as_float(0x7f800000u))) {  // cluster-uniform
    ok = false;
    return 0.f;
  }
  const float sc = 256.f * __frcp_rn(span);
#pragma unroll
  for (int q = 0; q < SPT; ++q)
    if (v[q] == v[q]) atomicAdd(sel.hist + value_bin(v[q], mn, sc), 1u);
  __syncthreads();
  cl.sync();  // every CTA's histogram complete
  const PassOut p = cluster_find_threshold<BLOCK, 256, C>(cl, sel, r);
  cl.sync();  // every CTA done reading the histograms
  for (int i = threadIdx.x; i < 256; i += BLOCK) sel.hist[i] = 0u;
  __syncthreads();
  if (p.d < 0) return ninf;  // fewer than r valid samples (cluster-uniform)
  float t = mn + static_cast<float>(p.d) * __frcp_rn(sc);
  if (p.cnt > 32 && p.d < 255) {  // cluster-uniform: a crowded bin, a finer round inside it
    const float sc2 = sc * 256.f;
    const float lo2 = t;
#pragma unroll
    for (int q = 0; q < SPT; ++q)
      if (v[q] == v[q] && value_bin(v[q], mn, sc) == p.d)
        atomicAdd(sel.hist + value_bin(v[q], lo2, sc2), 1u);
    __syncthreads();
    cl.sync();  // every CTA's finer histogram complete
    const PassOut p2 = cluster_find_threshold<BLOCK, 256, C>(cl, sel, r - p.above);
    cl.sync();  // every CTA done reading them
    for (int i = threadIdx.x; i < 256; i += BLOCK) sel.hist[i] = 0u;
    __syncthreads();
    if (p2.d >= 0) t = lo2 + static_cast<float>(p2.d) * __frcp_rn(sc2);
  }
  return grid_floor<T>(t - fabsf(t) * 9.5367e-7f - 1e-37f);
}

// put(pos, key, column) for output position pos of the row's top-K layout
// (the layout of topk_row), fill(pos) for the positions past the last
// candidate.  The histogram must be zero on entry.
template <typename T, int BLOCK, int SUB, int ALIGN, int C, class Put, class Fill>
__device__ void cluster_topk_row(cg::cluster_group &cl, const T *__restrict__ xr, int end,
                                 int K, Put put, Fill fill, ClusterSmem<BLOCK, SUB> &cs) {
  constexpr int KB = KeyOf<T>::kBits;
  constexpr int CAP = ListSmem<BLOCK, SUB>::CAP;
  constexpr bool VECLOAD = ALIGN != 0;
  ListSmem<BLOCK, SUB> &sm = cs.ls;
  const int crank = static_cast<int>(cl.block_rank());
  // this CTA's slice: groups [g0, g1) of 8 columns; the last CTA also takes
  // the < 8 ragged columns
  const int ngroups = end / 8;
  const int gper = (ngroups + C - 1) / C;
  const int g0 = min(ngroups, crank * gper), g1 = min(ngroups, g0 + gper);
  const int col0 = g0 * 8;
  const int send = crank == C - 1 ? end - col0 : (g1 - g0) * 8;
  const T *xs = xr + col0;
  // every slice fits a list: each CTA takes all its valid columns
  const bool all = end <= C * (CAP - 8);
  prefetch_row_head<T, BLOCK, ALIGN>(xs, send);
  float t0f = __uint_as_float(0xff800000u);
  if (!all) {  // every slice has > CAP - 8 * C columns: enough for its sample
    const int r = sample_rank(K, C * BLOCK * kRowSample, end);
    bool ok;
    t0f = cluster_value_threshold<T, BLOCK, SUB, C>(cl, xs, send, r, cs, ok);
    if (!ok) {  // cluster-uniform: rank the samples by ordered keys
      const Seg ss = sample_keys<T, BLOCK, kRowSample, SUB>(xs, send, sm);
      const Sel s = cluster_list_select<BLOCK, SUB, C>(
          cl, [&](int i) { return sm.key[i]; }, ss, r, cs, 3, kPubSampleStats, stats_unknown(),
          32 - KB);
      t0f = threshold_float<KB>(s.take_all ? 1u : s.T);
    }
  }
  if (threadIdx.x == 0) sm.flag = 0;
  __syncthreads();  // sample keys read, flag clear
  WarpStats st;
  Seg sg = collect_filtered<T, BLOCK, SUB, ALIGN, kRowBatch>(xs, send, t0f, sm, st);
  int listed;
  block_warp_prefix<BLOCK>(sg.cnt, sm.sel.wtot[3], &listed);
  if (threadIdx.x == 0) {
    cs.pub[kPubFlag] = static_cast<uint32_t>(sm.flag);
    cs.pub[kPubCount] = static_cast<uint32_t>(listed);
  }
  cl.sync();  // every CTA's overflow flag and count published
  bool over = false;
  int total = 0;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    over = over || cluster_word(cl, &cs.pub[kPubFlag], c) != 0u;
    total += static_cast<int>(cluster_word(cl, &cs.pub[kPubCount], c));
  }
  if (!over && (all || total >= K)) {  // cluster-uniform
    cluster_topk_emit<BLOCK, SUB, C>(cl, cs, sg, K, col0, put, fill, st, 32 - KB);
  } else if (crank == 0) {  // the exact path, on CTA 0 over the whole row
    __syncthreads();
    sg = collect_exact<T, BLOCK, SUB, VECLOAD>(xr, end, K, sm);
    list_topk_emit<BLOCK, SUB>(
        sm, sg, K,
        [&](int pos, int i) {
          if ((unsigned)pos < (unsigned)K) put(pos, sm.key[i], static_cast<int>(sm.val[i]));
        },
        fill, stats_unknown(), 32 - KB);
  }
  cl.sync();  // no CTA leaves while another may still read its shared memory
}

}  // namespace satk
