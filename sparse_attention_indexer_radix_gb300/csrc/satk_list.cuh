// satk_list.cuh -- candidate lists in shared memory and the exact select
// over them.
//
// A row's candidates are first filtered into an ordered list that provably
// holds the row's K best, then the K best are selected exactly on the list.
// The list lives in per-warp segments: warp w owns entries
// [base_w, base_w + cnt_w) of the shared arrays key[] and val[], and the
// order of the row is (warp, entry): warp segments follow one another in
// row order and each segment is in row order.  key is the ordered score key
// (0 = no candidate) and val the id to emit (column, or global id).
//
// The select is a most-significant-digit radix select whose digits are
// taken relative to the list's own key range: with kmin and kmax the
// smallest and largest key, digits are cut from key - kmin over the
// bit-length of kmax - kmin.  A list gathered above a threshold spans a
// narrow range, so its top absolute bits are all equal; relative digits
// spread it over the bins, which keeps the shared-memory histogram atomics
// free of pile-ups without any warp aggregation.
#pragma once

#include "satk_device.cuh"

namespace satk {

template <int BLOCK, int SUB>
struct ListSmem {
  static constexpr int NW = BLOCK / 32;
  static constexpr int CAP = NW * SUB;
  SelectSmem<BLOCK> sel;
  uint32_t key[CAP];
  uint32_t val[CAP];
  int cnt[NW];
  int flag;
};

// This thread's share of the list: warp w's segment, lane-strided.  The
// loop bound rounds the segment up to whole warps so that every lane of a
// warp runs the same iterations (entries past the segment read as key 0).
struct Seg {
  int base;
  int cnt;
  __device__ __forceinline__ int rounds() const { return (cnt + 31) >> 5; }
};

// Count, smallest and largest key of one warp's list entries, when the
// pass that wrote them already knows them (warp-uniform values); n < 0
// means unknown.
struct WarpStats {
  int n;
  uint32_t mn, mx;
  __device__ __forceinline__ bool known() const { return n >= 0; }
};
__device__ __forceinline__ WarpStats stats_unknown() { return WarpStats{-1, 0u, 0u}; }

// Digit width of the list select: a pass costs one walk over the list plus
// one scan over the bins.  Short lists take 8-bit digits (cheap scans),
// longer ones 11-bit digits (fewer walks).
constexpr int kListDigitShort = 8;
constexpr int kListDigitLong = 11;
constexpr int kListLong = 1024;
// At most this many keys in the threshold digit are ranked directly.
constexpr int kListFinish = 64;

// Radix select of the K largest keys among the list entries gk(i) != 0 of
// this thread's segment.  Outcome as Sel (see satk_device.cuh); the
// threshold T is an absolute key.  gk may return 0 to drop an entry.
// With max_passes, the digit passes stop early and T is the start of the
// threshold digit (at least K keys are >= T).  With pre known, the warp's
// count and key range come from the caller instead of a walk over the list
// (gk must then be non-zero exactly on those entries).  With lz, the low lz
// bits of every key are known to be zero (bf16 keys: ord16 << 16), so the
// digits start above them.
template <int BLOCK, class GetKey>
__device__ Sel list_select(GetKey gk, const Seg &sg, int K, SelectSmem<BLOCK> &sm,
                           int max_passes = 8, WarpStats pre = stats_unknown(), int lz = 0) {
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
  // count, min and max in one reduction (one barrier): warp values go to
  // red / wtot[1] / wtot[2]; the next writer of those arrays (another
  // list_select, block_min) is behind later barriers
  if (lane == 0) {
    sm.red[warp_id()] = mn;
    sm.wtot[1][warp_id()] = static_cast<int>(mx);
    sm.wtot[2][warp_id()] = n;
  }
  __syncthreads();
  int total = 0;
  mn = 0xffffffffu;
  mx = 0u;
#pragma unroll
  for (int w = 0; w < BLOCK / 32; ++w) {
    mn = min(mn, sm.red[w]);
    mx = max(mx, static_cast<uint32_t>(sm.wtot[1][w]));
    total += sm.wtot[2][w];
  }
  Sel r;
  r.tie = false;
  r.take_all = false;
  r.total = total;
  const uint32_t span = (mx - mn) >> lz;
  const int b = span == 0u ? 0 : 32 - __clz(span);
  if (total < K || b == 0) __syncthreads();  // no pass barrier follows
  if (total < K) {
    r.take_all = true;
    r.T = 1u;
    r.need = 0;
    return r;
  }
  if (b == 0 && total == K) {  // exactly K keys, all equal: no tie to break
    r.T = mn;
    r.need = K;
    r.exact = true;
    return r;
  }
  int need = K;
  uint32_t prefix = 0u;
  int pbits = 0;
  const int digit = total > kListLong ? kListDigitLong : kListDigitShort;
  while (pbits < b) {
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
    __syncthreads();
    const PassOut p = digit == kListDigitLong
                          ? find_threshold<BLOCK, (1 << kListDigitLong)>(sm, need)
                          : find_threshold<BLOCK, (1 << kListDigitShort)>(sm, need);
    need -= p.above;
    prefix = (prefix << width) | static_cast<uint32_t>(p.d);
    pbits += width;
    if (p.cnt == need) {
      r.T = mn + ((prefix << shift) << lz);
      r.need = need;
      return r;
    }
    if (p.cnt <= kListFinish && pbits < b) {  // block-uniform
      // a few keys left in the threshold digit: rank them on one warp
      // instead of more digit passes over the whole list
      for (int j = 0; j < sg.rounds(); ++j) {
        const int i = j * 32 + lane;
        const uint32_t k = i < sg.cnt ? gk(sg.base + i) : 0u;
        if (k != 0u && (((k - mn) >> lz) >> shift) == prefix) {
          const int pos = atomicAdd(&sm.fcnt, 1);
          if (pos < kListFinish) sm.fin[pos] = k;
        }
      }
      __syncthreads();
      if (warp_id() == 0) {
        const int c = p.cnt;
        // lane l ranks fin[l] and fin[l + 32]: the need-th largest v has
        // gt(v) < need <= gt(v) + eq(v)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = lane + 32 * h;
          if (q < c) {
            const uint32_t x = sm.fin[q];
            int gt = 0, eq = 0;
            for (int i = 0; i < c; ++i) {
              const uint32_t f = sm.fin[i];
              gt += f > x ? 1 : 0;
              eq += f == x ? 1 : 0;
            }
            if (gt < need && need <= gt + eq) {  // every copy of v writes the same
              sm.scal[4] = static_cast<int>(x);
              sm.scal[5] = gt;
              sm.scal[6] = eq;
            }
          }
        }
        if (lane == 0) sm.fcnt = 0;
      }
      __syncthreads();
      const uint32_t v = static_cast<uint32_t>(sm.scal[4]);
      const int gt = sm.scal[5], eq = sm.scal[6];
      if (gt + eq == need) {  // exactly K keys >= v, v the smallest of them
        r.T = v;
        r.need = need;
        r.exact = true;
      } else {  // v is the K-th key, need - gt of its ties wanted
        r.T = v;
        r.need = need - gt;
        r.tie = true;
      }
      return r;
    }
    if (--max_passes == 0) {
      r.T = mn + ((prefix << shift) << lz);
      r.need = need;
      return r;
    }
  }
  // every key bit resolved: the K-th key is mn + prefix and `need` of the
  // keys equal to it are still wanted (more than need share it)
  r.T = mn + (prefix << lz);
  r.need = need;
  r.tie = true;
  return r;
}

// Ordered compaction over the list segments: cls(i) = 0 skip, 1 group A,
// 2 group B for absolute entry i; emitA/emitB(rank, i, tot) as in
// ordered_emit.  The counting walk keeps each round's two ballots (in the
// zero histogram, 64 words per warp, cleared again afterwards) so the
// writing walk need not classify again.  Two barriers.
template <int BLOCK, class Cls, class EmitA, class EmitB>
__device__ int2 list_emit(Cls cls, const Seg &sg, EmitA emitA, EmitB emitB, SelectSmem<BLOCK> &sm) {
  static_assert(BLOCK / 32 * 64 <= 2048, "ballot store exceeds the histogram");
  const int lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  uint32_t *bal = sm.hist + warp_id() * 64;
  const int R = sg.rounds();
  int ca = 0, cb = 0;
  for (int j = 0; j < R; ++j) {
    const int i = j * 32 + lane;
    const int c = i < sg.cnt ? cls(sg.base + i) : 0;
    const unsigned ba = __ballot_sync(kFull, c == 1);
    const unsigned bb = __ballot_sync(kFull, c == 2);
    if (lane == 0 && j < 32) {
      bal[2 * j] = ba;
      bal[2 * j + 1] = bb;
    }
    ca += __popc(ba);
    cb += __popc(bb);
  }
  int total;
  const unsigned base =
      (unsigned)block_warp_prefix<BLOCK>((ca << 16) | cb, sm.wtot[3], &total);
  const int2 tot = make_int2((int)((unsigned)total >> 16), (int)((unsigned)total & 0xffffu));
  int ra = (int)(base >> 16), rb = (int)(base & 0xffffu);
  for (int j = 0; j < R; ++j) {
    const int i = j * 32 + lane;
    unsigned ba, bb;
    if (j < 32) {
      ba = bal[2 * j];
      bb = bal[2 * j + 1];
    } else {
      const int c = i < sg.cnt ? cls(sg.base + i) : 0;
      ba = __ballot_sync(kFull, c == 1);
      bb = __ballot_sync(kFull, c == 2);
    }
    if ((ba >> lane) & 1u) emitA(ra + __popc(ba & lt), sg.base + i, tot);
    if ((bb >> lane) & 1u) emitB(rb + __popc(bb & lt), sg.base + i, tot);
    ra += __popc(ba);
    rb += __popc(bb);
  }
  __syncwarp();
  bal[lane] = 0u;
  bal[lane + 32] = 0u;
  __syncthreads();
  return tot;
}

// list_emit with one group: sel(i) chooses absolute entry i; emit(rank, i)
// receives each chosen entry's rank in list order.  Returns the count.
// Two barriers.
template <int BLOCK, class SelF, class Emit>
__device__ int list_emit1(SelF sel, const Seg &sg, Emit emit, SelectSmem<BLOCK> &sm) {
  static_assert(BLOCK / 32 * 32 <= 2048, "ballot store exceeds the histogram");
  const int lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  uint32_t *bal = sm.hist + warp_id() * 32;
  const int R = sg.rounds();
  int ca = 0;
  for (int j = 0; j < R; ++j) {
    const int i = j * 32 + lane;
    const unsigned ba = __ballot_sync(kFull, i < sg.cnt && sel(sg.base + i));
    if (lane == 0 && j < 32) bal[j] = ba;
    ca += __popc(ba);
  }
  int total;
  int ra = block_warp_prefix<BLOCK>(ca, sm.wtot[3], &total);
  for (int j = 0; j < R; ++j) {
    const int i = j * 32 + lane;
    const unsigned ba =
        j < 32 ? bal[j] : __ballot_sync(kFull, i < sg.cnt && sel(sg.base + i));
    if ((ba >> lane) & 1u) emit(ra + __popc(ba & lt), sg.base + i);
    ra += __popc(ba);
  }
  __syncwarp();
  bal[lane] = 0u;
  __syncthreads();
  return total;
}

// Row top-K layout from the list: entries above the K-th key in list order,
// then entries equal to it in list order up to K, then fill(pos) up to K.
// lz: low key bits known to be zero (list_select).
template <int BLOCK, int SUB, class Put, class Fill>
__device__ void list_topk_emit(ListSmem<BLOCK, SUB> &sm, const Seg &sg, int K, Put put,
                               Fill fill, WarpStats pre = stats_unknown(), int lz = 0) {
  auto gk = [&](int i) { return sm.key[i]; };
  const Sel sel = list_select<BLOCK>(gk, sg, K, sm.sel, 8, pre, lz);
  uint32_t v;
  if (sel.take_all) {
    v = 0u;
  } else if (sel.tie || sel.exact) {
    v = sel.T;
  } else {
    uint32_t m = 0xffffffffu;
    for (int j = 0; j < sg.rounds(); ++j) {
      const int i = j * 32 + lane_id();
      const uint32_t k = i < sg.cnt ? sm.key[sg.base + i] : 0u;
      if (k >= sel.T) m = min(m, k);
    }
    v = block_min<BLOCK>(m, sm.sel);
  }
  const bool all = sel.take_all;
  const int2 tot = list_emit<BLOCK>(
      [&](int i) -> int {
        const uint32_t k = sm.key[i];
        if (k == 0u) return 0;
        if (all) return 1;
        return k > v ? 1 : (k == v ? 2 : 0);
      },
      sg, [&](int rank, int i, int2) { put(rank, i); },
      [&](int rank, int i, int2 t) {
        if (rank < K - t.x) put(t.x + rank, i);
      },
      sm.sel);
  const int nsel = all ? max(0, min(tot.x, K)) : K;
  for (int q = nsel + (int)threadIdx.x; q < K; q += BLOCK) fill(q);
}

// Merge select on a list whose values are global ids: the K best entries
// under (key desc, id asc) -- a select on the key, then, when the K-th key
// is tied, a select on ~id among the tied entries -- emitted in list order
// as out(rank, id), then out(rank, -1) up to K.  When one (key, id) is
// repeated across the cut, all its copies are left out (fewer than K ids)
// and the call returns true.
struct ListMergeOut {
  bool dup;       // a repeated (key, id) sat on the cut
  int nsel;       // ids emitted before the -1 fill
  uint32_t kmin;  // smallest chosen key (with WANT_MIN; 0xffffffff when none)
};

template <int BLOCK, int SUB, bool WANT_MIN = false, class Out>
__device__ ListMergeOut list_merge_emit(ListSmem<BLOCK, SUB> &sm, const Seg &sg, int K, Out out,
                                        WarpStats pre = stats_unknown()) {
  const Sel s1 = list_select<BLOCK>([&](int i) { return sm.key[i]; }, sg, K, sm.sel, 8, pre);
  if (s1.take_all || !s1.tie) {  // block-uniform: no tie at the K-th key (the usual case)
    const bool all_keys = s1.take_all;
    const uint32_t T1 = s1.T;
    uint32_t kmin = 0xffffffffu;
    if (WANT_MIN && !all_keys && s1.exact) {
      kmin = T1;  // the select found the smallest chosen key itself
    } else if (WANT_MIN) {
      uint32_t m = 0xffffffffu;
      for (int j = 0; j < sg.rounds(); ++j) {
        const int i = j * 32 + lane_id();
        const uint32_t k = i < sg.cnt ? sm.key[sg.base + i] : 0u;
        if (k != 0u && (all_keys || k >= T1)) m = min(m, k);
      }
      kmin = block_min<BLOCK>(m, sm.sel);
    }
    const int n1 = list_emit1<BLOCK>(
        [&](int i) {
          const uint32_t k = sm.key[i];
          return k != 0u && (all_keys || k >= T1);
        },
        sg,
        [&](int rank, int i) {
          if ((unsigned)rank < (unsigned)K) out(rank, static_cast<int32_t>(sm.val[i]));
        },
        sm.sel);
    for (int q = max(0, n1) + (int)threadIdx.x; q < K; q += BLOCK) out(q, -1);
    return ListMergeOut{false, min(n1, K), kmin};
  }
  const Sel s2 = list_select<BLOCK>(
      [&](int i) { return sm.key[i] == s1.T ? 0xffffffffu - sm.val[i] : 0u; }, sg, s1.need,
      sm.sel);
  const uint32_t T1 = s1.T, t2 = s2.T;
  const bool tie2 = s2.tie;
  const int2 tot = list_emit<BLOCK>(
      [&](int i) -> int {
        const uint32_t k = sm.key[i];
        if (k == 0u) return 0;
        if (k != T1) return k > T1 ? 1 : 0;
        const uint32_t k2 = 0xffffffffu - sm.val[i];
        return (tie2 ? k2 > t2 : k2 >= t2) ? 1 : 0;
      },
      sg,
      [&](int rank, int i, int2) {
        if ((unsigned)rank < (unsigned)K) out(rank, static_cast<int32_t>(sm.val[i]));
      },
      [](int, int, int2) {}, sm.sel);
  for (int q = max(0, tot.x) + (int)threadIdx.x; q < K; q += BLOCK) out(q, -1);
  // with a tie the K-th key itself is chosen, unless its copies were all
  // left out as repeats (then fewer than K ids)
  return ListMergeOut{tie2, min(tot.x, K), WANT_MIN ? T1 : 0xffffffffu};
}

// ------------------------------------------------------ one warp alone --
//
// The select above at warp scale: no block barrier, only the calling warp
// (all 32 lanes) and a 256-bin histogram of its own.

// The digit d of a 256-bin histogram (descending) with
// above(d) < need <= above(d) + hist[d]; d = -1 when fewer than need keys
// were counted.  Zeroes every bin.  Lane l reads bins 255 - (32 j + l), so
// each of its eight reads is conflict-free.
struct WarpDigit {
  int d, above, cnt;
};
__device__ __forceinline__ WarpDigit warp_find_digit(uint32_t *hist, int need) {
  const int lane = lane_id();
  uint32_t c[8];
  int gs[8];
  int total = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int bin = 255 - (32 * j + lane);
    c[j] = hist[bin];
    hist[bin] = 0u;
    gs[j] = static_cast<int>(__reduce_add_sync(kFull, c[j]));
    total += gs[j];
  }
  WarpDigit r{-1, 0, 0};
  if (total < need) return r;
  int cum = 0, jc = 0;
  uint32_t cj = 0u;
  bool found = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {  // warp-uniform
    if (!found && cum + gs[j] >= need) {
      found = true;
      jc = j;
      cj = c[j];
    } else if (!found) {
      cum += gs[j];
    }
  }
  const int incl = warp_incl_scan(static_cast<int>(cj));
  const int before = cum + incl - static_cast<int>(cj);
  const unsigned hit = __ballot_sync(kFull, before < need && before + static_cast<int>(cj) >= need);
  const int src = __ffs(hit) - 1;
  r.d = 255 - (32 * jc + src);
  r.above = __shfl_sync(kFull, before, src);
  r.cnt = __shfl_sync(kFull, static_cast<int>(cj), src);
  return r;
}

// ------------------------------------------------------- thresholds ------

// The float whose ordered key is the smallest key >= T among the keys a
// dtype of KB bits can take (bf16 keys are multiples of 2**16); -inf when T
// is at or below the key of -inf, so that a float compare x >= result
// holds exactly for the non-NaN x with key(x) >= T.
template <int KB>
__device__ __forceinline__ float threshold_float(uint32_t T) {
  if (KB == 16) T = (T > 0xffff0000u) ? 0xffff0000u : ((T + 0xffffu) & 0xffff0000u);
  const uint32_t neg_inf_key = KB == 16 ? 0x007f0000u : 0x007fffffu;
  if (T <= neg_inf_key) return __uint_as_float(0xff800000u);
  // +0.0 and -0.0 compare equal as floats: a threshold at +0.0 moves to
  // -0.0 (one key lower), keeping the compare exact
  const uint32_t pos_zero = 0x80000000u;
  if (T == pos_zero) T = KB == 16 ? 0x7fff0000u : 0x7fffffffu;
  const uint32_t bits = (T & 0x80000000u) ? (T & 0x7fffffffu) : ~T;
  return __uint_as_float(bits);
}

}  // namespace satk
