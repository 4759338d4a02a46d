// satk_warp.cuh -- the row path with one warp per row, for short rows.
//
// Rows of a few thousand columns are bound by the latency of the per-row
// steps, not by the stream: a CTA per row leaves too few rows in flight.
// Here every warp owns one row and a small shared-memory workspace, and
// never waits on another warp, so an SM holds 28 rows at once.  The steps
// are those of the CTA path (satk_rows.cuh) at warp scale:
//  1. threshold from a sample of up to kWarpSample columns (runs of 256,
//     as few as keep the expected list within bounds for the row's length);
//  2. one filtered pass that records keys and columns of the columns at or
//     above it in the warp's list, in column order, with the copy engine
//     one batch ahead of the loads (bulk L2 prefetch);
//  3. exact select on the list (8-bit digits relative to the list's key
//     range, a 256-bin histogram per warp) and the ordered emit: ids with
//     key > v in ascending column order, then ids with key == v, -1 after.
// A list that would overflow, or a sample threshold that left fewer than K
// candidates, sends the row to an exact narrowing path over the row itself.
#pragma once

#include "satk_rows.cuh"

namespace satk {

constexpr int kWarpList = 1024;    // list entries per warp
constexpr int kWarpSample = 1536;  // sampled columns per row (kWarpSample / 32 runs)
constexpr int kWarpRowsPerCta = 4;

// Per-warp workspace.  buf holds the list (keys in buf[0, kWarpList), 16-bit
// columns after them) or, before the list exists, the sample's keys.
struct WarpRowSmem {
  uint32_t buf[kWarpList + kWarpList / 2];
  uint32_t hist[256];  // kept zero between passes
  __device__ __forceinline__ uint32_t *key() { return buf; }
  __device__ __forceinline__ uint16_t *col() {
    return reinterpret_cast<uint16_t *>(buf + kWarpList);
  }
};
static_assert(kWarpSample <= kWarpList + kWarpList / 2, "the sample must fit the list area");

// Count, smallest and largest key of a warp's list (warp-uniform).
struct WarpRange {
  int n;
  uint32_t mn, mx;
};

// Sample threshold of a row of end > kWarpList columns: the r-th largest key
// of the sampled columns -- runs of 32 8-column groups, one vector load per
// lane and run, spread evenly over the row, as many runs (at most
// kWarpSample / 256) as keep the expected list plus four standard
// deviations within kWarpList for this row's length --
// r = mu + 4 sqrt(mu) + 4 with mu = K * samples / end (as the CTA path);
// 1 when the sample holds fewer than r valid keys.  Two digit passes.
template <typename T, int ALIGN>
__device__ __forceinline__ uint32_t warp_sample_threshold(const T *__restrict__ xr, int end,
                                                          int K, WarpRowSmem &ws) {
  constexpr int MAXRUNS = kWarpSample / 256;
  const int lane = lane_id();
  const int ngroups = end / 8;  // >= 128: end > kWarpList
  // fewest runs of 256 columns whose expected list (K r / mu) plus four
  // standard deviations fits the list; shorter rows need fewer samples
  int nruns = MAXRUNS;
  for (int q = 1; q < MAXRUNS; ++q) {  // warp-uniform
    const float mu = static_cast<float>(K) * (256 * q) / static_cast<float>(end);
    const float r = ceilf(mu + 4.f * sqrtf(mu) + 4.f);
    const float list = static_cast<float>(K) * r / mu;
    if (list + 4.f * list * rsqrtf(r) <= static_cast<float>(kWarpList)) {
      nruns = q;
      break;
    }
  }
  const int S = 256 * nruns;
  uint32_t *sk = ws.buf;
  uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
  for (int q = 0; q < MAXRUNS; ++q) {
    if (q < nruns) {
      // 32-bit: q * ngroups < MAXRUNS * 2**13 for the rows this path takes
      const int g0 = min((q * ngroups) / nruns, ngroups - 32);
      Group8<T, ALIGN> grp;
      grp.load(xr + static_cast<size_t>(g0 + lane) * 8);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t k = key_of_raw<T>(grp.raw(e));
        sk[(q * 8 + e) * 32 + lane] = k;
        mn = min(mn, k);
        mx = max(mx, k);
      }
    }
  }
  mn = __reduce_min_sync(kFull, mn);
  mx = __reduce_max_sync(kFull, mx);
  __syncwarp();
  const float mu = static_cast<float>(K) * S / static_cast<float>(end);
  int r = static_cast<int>(ceilf(mu + 4.f * sqrtf(mu) + 4.f));
  r = r < 1 ? 1 : (r > S ? S : r);
  int m = S;
  if (mn == 0u) {  // NaN samples (key 0): compact the valid keys to the front
    m = 0;
    mn = 0xffffffffu;
    for (int i0 = 0; i0 < S; i0 += 32) {
      const uint32_t k = sk[i0 + lane];
      const unsigned b = __ballot_sync(kFull, k != 0u);
      __syncwarp();
      if (k != 0u) {
        sk[m + __popc(b & ((1u << lane) - 1u))] = k;
        mn = min(mn, k);
      }
      m += __popc(b);
      __syncwarp();
    }
    mn = __reduce_min_sync(kFull, mn);
  }
  if (m < r) return 1u;
  const WarpSel s = warp_list_select(sk, m, r, mn, mx, ws.hist, 2);
  return s.take_all ? 1u : s.T;
}

// The filtered pass over a whole row: columns whose score compares >= t0f
// go to the list in column order, with their keys.  Returns false when the
// list would overflow (the row then takes the exact path).
template <typename T, int ALIGN>
__device__ __forceinline__ bool warp_collect(const T *__restrict__ xr, int end, float t0f,
                                             WarpRowSmem &ws, WarpRange &out) {
  constexpr int U = 4;
  const int lane = lane_id();
  const int ngroups = end / 8;
  uint32_t *lk = ws.key();
  uint16_t *lc = ws.col();
  const ThresholdOf<T> thr(t0f);
  int cnt = 0;
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  bool over = false;
  for (int gb = 0; gb < ngroups; gb += 32 * U) {
    prefetch_groups<T, ALIGN>(xr, min(ngroups, gb + 32 * U), min(ngroups, gb + 2 * 32 * U));
    Group8<T, ALIGN> grp[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gi = gb + u * 32 + lane;
      if (gi < ngroups) grp[u].load(xr + static_cast<size_t>(gi) * 8);
    }
    uint32_t m[U];
    uint32_t pk[U / 2];
#pragma unroll
    for (int j = 0; j < U / 2; ++j) pk[j] = 0u;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gi = gb + u * 32 + lane;
      m[u] = gi < ngroups ? grp[u].mask(thr.arg()) : 0u;
      pk[u >> 1] |= static_cast<uint32_t>(__popc(m[u])) << (16 * (u & 1));
    }
    uint32_t incl[U / 2], tot[U / 2];
    int btot = 0;
#pragma unroll
    for (int j = 0; j < U / 2; ++j) {
      incl[j] = static_cast<uint32_t>(warp_incl_scan(static_cast<int>(pk[j])));
      tot[j] = __shfl_sync(kFull, incl[j], 31);
      btot += static_cast<int>((tot[j] & 0xffffu) + (tot[j] >> 16));
    }
    if (cnt + btot > kWarpList) {  // warp-uniform
      over = true;
      break;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t lcount = static_cast<uint32_t>(__popc(m[u]));
      int pos = cnt + static_cast<int>(((incl[u >> 1] >> (16 * (u & 1))) & 0xffffu) - lcount);
      uint32_t mm = m[u];
      const int c0 = (gb + u * 32 + lane) * 8;
      while (mm != 0u) {
        const int s = __ffs(mm) - 1;
        mm &= mm - 1u;
        const uint32_t k = key_of_num<T>(grp[u].raw(s));
        lk[pos] = k;
        lc[pos] = static_cast<uint16_t>(c0 + s);
        kmn = min(kmn, k);
        kmx = max(kmx, k);
        ++pos;
      }
      cnt += static_cast<int>((tot[u >> 1] >> (16 * (u & 1))) & 0xffffu);
    }
  }
  if (!over && ngroups * 8 < end) {  // the < 8 ragged columns
    const int c = ngroups * 8 + lane;
    const uint32_t rw = c < end ? load_raw(xr + c) : 0u;
    const bool keep = c < end && as_float<T>(rw) >= t0f;
    const unsigned b = __ballot_sync(kFull, keep);
    if (cnt + __popc(b) > kWarpList) {
      over = true;
    } else {
      if (keep) {
        const int pos = cnt + __popc(b & ((1u << lane) - 1u));
        const uint32_t k = key_of_num<T>(rw);
        lk[pos] = k;
        lc[pos] = static_cast<uint16_t>(c);
        kmn = min(kmn, k);
        kmx = max(kmx, k);
      }
      cnt += __popc(b);
    }
  }
  out = WarpRange{cnt, __reduce_min_sync(kFull, kmn), __reduce_max_sync(kFull, kmx)};
  __syncwarp();
  return !over;
}

// Exact path: narrows the K-th key over the row with 8-bit digits of the
// absolute key until the keys at or above the threshold prefix fit the list,
// then collects them in column order.  At full key resolution with a tie
// wider than the list, only the first `need` tied columns are kept.
template <typename T>
__device__ void warp_collect_exact(const T *__restrict__ xr, int end, int K, WarpRowSmem &ws,
                                   WarpRange &out) {
  constexpr int KB = KeyOf<T>::kBits;
  const int lane = lane_id();
  uint32_t prefix = 0u;
  int pbits = 0, need = K, above = 0;
  uint32_t thr = 1u;
  bool limited = false;
  while (true) {
    const int shift = 32 - pbits - 8;
    for (int c = lane; c < end; c += 32) {
      const uint32_t k = key_of_raw<T>(load_raw(xr + c));
      if (k != 0u && (pbits == 0 || (k >> (32 - pbits)) == prefix))
        atomicAdd(ws.hist + ((k >> shift) & 255u), 1u);
    }
    __syncwarp();
    const WarpDigit p = warp_find_digit(ws.hist, need);
    __syncwarp();
    if (p.d < 0) {  // fewer than K valid columns (first pass only): all of them
      thr = 1u;
      break;
    }
    above += p.above;
    need -= p.above;
    prefix = (prefix << 8) | static_cast<uint32_t>(p.d);
    pbits += 8;
    thr = prefix << (32 - pbits);
    if (above + p.cnt <= kWarpList) break;
    if (pbits == KB) {
      limited = true;
      break;
    }
  }
  if (thr == 0u) thr = 1u;  // key 0 is no column
  uint32_t *lk = ws.key();
  uint16_t *lc = ws.col();
  const unsigned lt = (1u << lane) - 1u;
  int n = 0, runB = 0;
  uint32_t kmn = 0xffffffffu, kmx = 0u;
  for (int c0 = 0; c0 < end; c0 += 32) {
    const int c = c0 + lane;
    const uint32_t k = c < end ? key_of_raw<T>(load_raw(xr + c)) : 0u;
    const bool a = limited ? k > thr : k >= thr;
    const bool b = limited && k == thr;
    const unsigned bb = __ballot_sync(kFull, b);
    const bool keep = a || (b && runB + __popc(bb & lt) < need);
    const unsigned kb = __ballot_sync(kFull, keep);
    if (keep) {
      const int pos = n + __popc(kb & lt);
      lk[pos] = k;
      lc[pos] = static_cast<uint16_t>(c);
      kmn = min(kmn, k);
      kmx = max(kmx, k);
    }
    n += __popc(kb);
    runB += __popc(bb);
  }
  out = WarpRange{n, __reduce_min_sync(kFull, kmn), __reduce_max_sync(kFull, kmx)};
  __syncwarp();
}

// Select on the warp's list and the ordered emit into o[0, K).
__device__ __forceinline__ void warp_emit(WarpRowSmem &ws, const WarpRange &lr, int K,
                                          int32_t *__restrict__ o) {
  const int lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  const uint32_t *lk = ws.key();
  const uint16_t *lc = ws.col();
  const int n = lr.n;
  const WarpSel s = warp_list_select(lk, n, K, lr.mn, lr.mx, ws.hist, 8);
  if (s.take_all) {  // fewer than K: every entry in list order, then -1
    for (int i = lane; i < n; i += 32) o[i] = static_cast<int32_t>(lc[i]);
    for (int q = n + lane; q < K; q += 32) o[q] = -1;
    return;
  }
  uint32_t v;
  int takeB;
  if (s.tie) {
    v = s.T;
    takeB = s.need;
  } else {  // exactly K keys >= T: v is the smallest of them
    uint32_t m = 0xffffffffu;
    int mc = 0;
    for (int i = lane; i < n; i += 32) {
      const uint32_t k = lk[i];
      if (k >= s.T) {
        if (k < m) {
          m = k;
          mc = 1;
        } else if (k == m) {
          ++mc;
        }
      }
    }
    v = __reduce_min_sync(kFull, m);
    takeB = static_cast<int>(__reduce_add_sync(kFull, m == v ? static_cast<unsigned>(mc) : 0u));
  }
  const int cgt = K - takeB;
  int runA = 0, runB = 0;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t k = i < n ? lk[i] : 0u;
    const unsigned ba = __ballot_sync(kFull, k > v);
    const unsigned bb = __ballot_sync(kFull, k == v);
    if ((ba >> lane) & 1u) o[runA + __popc(ba & lt)] = static_cast<int32_t>(lc[i]);
    if ((bb >> lane) & 1u) {
      const int pb = runB + __popc(bb & lt);
      if (pb < takeB) o[cgt + pb] = static_cast<int32_t>(lc[i]);
    }
    runA += __popc(ba);
    runB += __popc(bb);
  }
}

// The whole row on one warp.  The histogram must be zero on entry and is
// zero again on return.
template <typename T, int ALIGN>
__device__ void warp_topk_row(const T *__restrict__ xr, int end, int K, int32_t *__restrict__ o,
                              WarpRowSmem &ws) {
  constexpr int KB = KeyOf<T>::kBits;
  // the copy engine starts on the first batch of the filtered pass
  prefetch_groups<T, ALIGN>(xr, 0, min(end / 8, 32 * 4));
  const bool all = end <= kWarpList;
  float t0f = __uint_as_float(0xff800000u);  // -inf: every valid column
  if (!all) t0f = threshold_float<KB>(warp_sample_threshold<T, ALIGN>(xr, end, K, ws));
  __syncwarp();  // the sample's keys are read before the list overwrites them
  WarpRange lr;
  const bool fits = warp_collect<T, ALIGN>(xr, end, t0f, ws, lr);
  if (!fits || (!all && lr.n < K)) warp_collect_exact<T>(xr, end, K, ws, lr);
  warp_emit(ws, lr, K, o);
}

}  // namespace satk
