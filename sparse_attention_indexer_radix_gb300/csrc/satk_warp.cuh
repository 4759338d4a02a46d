// satk_warp.cuh -- the row path with one warp per row, for short rows.
//
// Rows of a few thousand columns are bound by instruction issue, not by the
// stream: every row pays fixed per-row steps, and a CTA per row leaves too
// few rows in flight.  Here every warp owns one row and a 7 KB shared-memory
// workspace and never waits on another warp, so an SM holds 28 rows at once.
// The steps (same semantics as the CTA path, satk_rows.cuh):
//  1. threshold from a sample of up to kWarpSample columns (runs of 256, as
//     few as keep the expected list within bounds for the row's length):
//     a value-linear 256-bin histogram over the sample's [min, max] picks the
//     bin of its r-th largest value (one finer pass inside that bin when it
//     is crowded), so for ordinary value ranges one pass over the sample
//     suffices; an unusable range (an infinity, a single value) takes the
//     ordered-key digits instead;
//  2. one filtered pass, coalesced 8-column groups per lane, that appends the
//     raw bits and column of every column at or above the threshold to the
//     warp's list in column order (per-lane counts through a warp prefix
//     scan, then predicated shared-memory stores), with the copy engine one
//     batch ahead of the loads (bulk L2 prefetch);
//  3. the list's raw bits turned into ordered keys in place, an exact select
//     (8-bit digits relative to the list's key range; once the threshold
//     digit holds at most 32 keys they are ranked on the warp directly) and
//     the ordered emit: ids with key > v in ascending column order, then ids
//     with key == v, -1 after.
// A list that would overflow, or a threshold that left fewer than K
// candidates, sends the row to an exact narrowing path over the row itself.
#pragma once

#include "satk_rows.cuh"

namespace satk {

constexpr int kWarpList = 1024;    // list entries per warp
constexpr int kWarpSample = 1536;  // sampled columns per row (kWarpSample / 256 runs)
constexpr int kWarpRowsPerCta = 4;

// Per-warp workspace.  buf holds the list (raw bits, then keys, in
// buf[0, kWarpList), 16-bit columns after them) or, before the list exists,
// the sampled values.
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

// Sampled columns of a row of end > kWarpList columns: runs of 32 8-column
// groups, one vector load per lane and run, spread evenly over the row, as
// many runs (at most kWarpSample / 256) as keep the expected list plus four
// standard deviations within kWarpList for this row's length.  The values
// go to buf: run q of lane l at words q*256 + h*128 + 4l (two 16-byte
// slots per lane and run, conflict-free).
template <typename T, int ALIGN>
__device__ __forceinline__ int warp_sample_runs(const T *__restrict__ xr, int end, int K,
                                                WarpRowSmem &ws, float &mn, float &mx) {
  constexpr int MAXRUNS = kWarpSample / 256;
  const int lane = lane_id();
  const int ngroups = end / 8;  // >= 128: end > kWarpList
  const float inv_end = __frcp_rn(static_cast<float>(end));
  int nruns = MAXRUNS;
  for (int q = 1; q < MAXRUNS; ++q) {  // warp-uniform
    const float mu = static_cast<float>(K * 256 * q) * inv_end;
    const float r = ceilf(mu + 4.f * (mu * rsqrtf(mu)) + 4.f);
    const float list = static_cast<float>(K) * r * __frcp_rn(mu);
    if (list + 4.f * list * rsqrtf(r) <= static_cast<float>(kWarpList)) {
      nruns = q;
      break;
    }
  }
  const float run_step = static_cast<float>(ngroups) * __frcp_rn(static_cast<float>(nruns));
  float *sv = reinterpret_cast<float *>(ws.buf);
  mn = __uint_as_float(0x7f800000u);
  mx = __uint_as_float(0xff800000u);
#pragma unroll
  for (int q = 0; q < MAXRUNS; ++q) {
    if (q < nruns) {
      const int g0 = min(static_cast<int>(static_cast<float>(q) * run_step), ngroups - 32);
      Group8<T, ALIGN> grp;
      grp.load(xr + static_cast<size_t>(g0 + lane) * 8);
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[e] = as_float<T>(grp.raw(e));
        mn = fminf(mn, v[e]);  // NaN ignored
        mx = fmaxf(mx, v[e]);
      }
      *reinterpret_cast<float4 *>(sv + q * 256 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4 *>(sv + q * 256 + 128 + 4 * lane) =
          make_float4(v[4], v[5], v[6], v[7]);
    }
  }
  mn = float_of_order(__reduce_min_sync(kFull, float_order(mn)));
  mx = float_of_order(__reduce_max_sync(kFull, float_order(mx)));
  __syncwarp();
  return nruns;
}

// The same rank by ordered-key digits (two range-relative 8-bit passes over
// the sampled values): for value ranges the bins cannot split.  Returns the
// threshold key (1: every valid column).
__device__ __forceinline__ uint32_t warp_sample_key_threshold(WarpRowSmem &ws, int nruns,
                                                              int r, bool bf16) {
  constexpr int MAXRUNS = kWarpSample / 256;
  const int lane = lane_id();
  const float *sv = reinterpret_cast<const float *>(ws.buf);
  auto key_at = [&](int q, int h, int e) -> uint32_t {
    const uint32_t b = __float_as_uint(sv[q * 256 + h * 128 + 4 * lane + e]);
    return bf16 ? key_bf16(b >> 16) : key_f32(b);
  };
  uint32_t mn = 0xffffffffu, mx = 0u;
  int nv = 0;
#pragma unroll
  for (int q = 0; q < MAXRUNS; ++q)
    if (q < nruns)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t k = key_at(q, h, e);
          mn = min(mn, k - 1u);  // key 0 (NaN) ignored
          mx = max(mx, k);
          nv += k != 0u;
        }
  mn = __reduce_min_sync(kFull, mn) + 1u;
  mx = __reduce_max_sync(kFull, mx);
  nv = static_cast<int>(__reduce_add_sync(kFull, static_cast<unsigned>(nv)));
  if (nv < r) return 1u;
  const uint32_t span = mx - mn;
  if (span == 0u) return mn;
  const int b = 32 - __clz(span);
  const int sh = b - (b < 8 ? b : 8);
#pragma unroll
  for (int q = 0; q < MAXRUNS; ++q)
    if (q < nruns)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t k = key_at(q, h, e);
          if (k != 0u) atomicAdd(ws.hist + ((k - mn) >> sh), 1u);
        }
  __syncwarp();
  const WarpDigit p = warp_find_digit(ws.hist, r);
  __syncwarp();
  uint32_t th = mn + (static_cast<uint32_t>(p.d) << sh);
  const int need = r - p.above;
  if (sh > 0 && p.cnt > need) {
    const int sh2 = sh - (sh < 8 ? sh : 8);
    const uint32_t dm = (1u << (sh - sh2)) - 1u;
    const uint32_t d = static_cast<uint32_t>(p.d);
#pragma unroll
    for (int q = 0; q < MAXRUNS; ++q)
      if (q < nruns)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t k = key_at(q, h, e);
            const uint32_t rel = k - mn;
            if (k != 0u && (rel >> sh) == d) atomicAdd(ws.hist + ((rel >> sh2) & dm), 1u);
          }
    __syncwarp();
    const WarpDigit p2 = warp_find_digit(ws.hist, need);
    __syncwarp();
    th += static_cast<uint32_t>(p2.d) << sh2;
  }
  return th;
}

// Sample threshold of a row of end > kWarpList columns: a float t such that,
// with a margin of about four standard deviations of the sampling error,
// at least K columns of the row score >= t; -inf when the sample holds
// fewer valid values than that (every valid column).  r = mu + 4 sqrt(mu)
// + 4 with mu = K * samples / end, as the CTA path.  On T's grid.
template <typename T, int ALIGN>
__device__ __forceinline__ float warp_sample_threshold(const T *__restrict__ xr, int end, int K,
                                                       WarpRowSmem &ws) {
  constexpr int MAXRUNS = kWarpSample / 256;
  constexpr int KB = KeyOf<T>::kBits;
  const int lane = lane_id();
  float mn, mx;
  const int nruns = warp_sample_runs<T, ALIGN>(xr, end, K, ws, mn, mx);
  const float ninf = __uint_as_float(0xff800000u);
  if (mx < mn) return ninf;  // no valid sample
  const int S = 256 * nruns;
  const float mu = static_cast<float>(K * S) * __frcp_rn(static_cast<float>(end));
  int r = static_cast<int>(ceilf(mu + 4.f * (mu * rsqrtf(mu)) + 4.f));
  r = r < 1 ? 1 : (r > S ? S : r);
  const float span = mx - mn;
  if (!(span > 0.f) || !(span < __uint_as_float(0x7f800000u)))
    return threshold_float<KB>(warp_sample_key_threshold(ws, nruns, r, KB == 16));
  const float *sv = reinterpret_cast<const float *>(ws.buf);
  const float sc = 256.f * __frcp_rn(span);
#pragma unroll
  for (int q = 0; q < MAXRUNS; ++q)
    if (q < nruns)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 v = *reinterpret_cast<const float4 *>(sv + q * 256 + h * 128 + 4 * lane);
        const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (vv[e] == vv[e]) atomicAdd(ws.hist + value_bin(vv[e], mn, sc), 1u);
      }
  __syncwarp();
  const WarpDigit p = warp_find_digit(ws.hist, r);
  __syncwarp();
  if (p.d < 0) return ninf;  // fewer than r valid samples
  float t = mn + static_cast<float>(p.d) * __frcp_rn(sc);
  if (p.cnt > 32 && p.d < 255) {  // crowded bin: one finer pass inside it
    const float sc2 = sc * 256.f;
    const float lo2 = t;
#pragma unroll
    for (int q = 0; q < MAXRUNS; ++q)
      if (q < nruns)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float4 v = *reinterpret_cast<const float4 *>(sv + q * 256 + h * 128 + 4 * lane);
          const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (vv[e] == vv[e] && value_bin(vv[e], mn, sc) == p.d)
              atomicAdd(ws.hist + value_bin(vv[e], lo2, sc2), 1u);
        }
    __syncwarp();
    const WarpDigit p2 = warp_find_digit(ws.hist, r - p.above);
    __syncwarp();
    t = lo2 + static_cast<float>(p2.d) * __frcp_rn(sc2);
  }
  // a little below the bin's edge, so rounding drops no counted sample
  return grid_floor<T>(t - fabsf(t) * 9.5367e-7f - 1e-37f);
}

// The filtered pass over a whole row: columns whose score compares >= t0f
// go to the list in column order, as raw bits and column.  Returns false
// when the list would overflow (the row then takes the exact path).
template <typename T, int ALIGN>
__device__ __forceinline__ bool warp_collect(const T *__restrict__ xr, int end, float t0f,
                                             WarpRowSmem &ws, int &n_out) {
  constexpr int U = 4;
  const int lane = lane_id();
  const int ngroups = end / 8;
  uint32_t *lk = ws.key();
  uint16_t *lc = ws.col();
  const ThresholdOf<T> thr(t0f);
  int cnt = 0;
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
      const int pos = cnt + static_cast<int>(((incl[u >> 1] >> (16 * (u & 1))) & 0xffffu) - lcount);
      // the lane's kept elements at pos, pos + 1, ...: each store predicated
      // on its mask bit, the two addresses advanced under the same predicate
      uint32_t ak = static_cast<uint32_t>(__cvta_generic_to_shared(lk + pos));
      uint32_t ac = static_cast<uint32_t>(__cvta_generic_to_shared(lc + pos));
      const int c0 = (gb + u * 32 + lane) * 8;
      const uint32_t mu = satk_check(pos + static_cast<int>(lcount) <= kWarpList, kDbgList)
                              ? m[u] : 0u;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "@p st.shared.b32 [%0], %2;\n\t"
            "@p st.shared.b16 [%1], %3;\n\t"
            "@p add.u32 %0, %0, 4;\n\t"
            "@p add.u32 %1, %1, 2;\n\t}"
            : "+r"(ak), "+r"(ac)
            : "r"(grp[u].raw(s)), "h"(static_cast<unsigned short>(c0 + s)),
              "r"(mu & (1u << s))
            : "memory");
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
        lk[pos] = rw;
        lc[pos] = static_cast<uint16_t>(c);
      }
      cnt += __popc(b);
    }
  }
  n_out = cnt;
  __syncwarp();
  return !over;
}

// The list's raw bits (none NaN: they passed a >= compare) -> ordered keys,
// in place; the list's count and key range.
template <typename T>
__device__ __forceinline__ WarpRange warp_list_keys(WarpRowSmem &ws, int n) {
  const int lane = lane_id();
  uint32_t *lk = ws.key();
  uint32_t mn = 0xffffffffu, mx = 0u;
  for (int i = lane; i < n; i += 32) {
    const uint32_t k = key_of_num<T>(lk[i]);
    lk[i] = k;
    mn = min(mn, k);
    mx = max(mx, k);
  }
  const WarpRange r{n, __reduce_min_sync(kFull, mn), __reduce_max_sync(kFull, mx)};
  __syncwarp();
  return r;
}

// Exact path: narrows the K-th key over the row with 8-bit digits of the
// absolute key until the keys at or above the threshold prefix fit the list,
// then collects them (as keys) in column order.  At full key resolution with
// a tie wider than the list, only the first `need` tied columns are kept.
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
    if (keep && satk_check(n + __popc(kb & lt) < kWarpList, kDbgList)) {
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

// Select on the warp's key list and the ordered emit (dst.put_entry(pos,
// list index, key, column) for positions [0, K), dst.fill past the last
// candidate): 8-bit
// digits relative to the list's key range; once the threshold digit holds
// at most 32 keys they are ranked on the warp directly (each lane counts
// the keys above and equal to its own) instead of more digit passes.
template <class Out>
__device__ __forceinline__ void warp_emit(WarpRowSmem &ws, const WarpRange &lr, int K,
                                          const Out &dst) {
  const int lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  const uint32_t *lk = ws.key();
  const uint16_t *lc = ws.col();
  const int n = lr.n;
  if (n < K) {  // fewer than K: every entry in list order, then the fill
    for (int i = lane; i < n; i += 32) dst.put_entry(i, i, lk[i], static_cast<int>(lc[i]));
    for (int q = n + lane; q < K; q += 32) dst.fill(q);
    return;
  }
  const uint32_t mn = lr.mn;
  const uint32_t span = lr.mx - mn;
  const int b = span == 0u ? 0 : 32 - __clz(span);
  int need = K;
  uint32_t prefix = 0u;
  int pbits = 0;
  uint32_t v = mn;   // the K-th key
  int takeB = need;  // keys == v to take
  bool found = false;
  while (pbits < b) {
    const int width = (b - pbits) < 8 ? (b - pbits) : 8;
    const int shift = b - pbits - width;
    const uint32_t dmask = (1u << width) - 1u;
    for (int i = lane; i < n; i += 32) {
      const uint32_t rel = lk[i] - mn;
      if (pbits == 0 || (rel >> (shift + width)) == prefix)
        atomicAdd(ws.hist + ((rel >> shift) & dmask), 1u);
    }
    __syncwarp();
    const WarpDigit p = warp_find_digit(ws.hist, need);
    __syncwarp();
    need -= p.above;
    prefix = (prefix << width) | static_cast<uint32_t>(p.d);
    pbits += width;
    if (pbits < b && p.cnt <= 32) {
      // the threshold digit's keys (hist[0, 32) as a buffer, zeroed again)
      int got = 0;
      for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t k = i < n ? lk[i] : 0u;
        const bool in = i < n && ((k - mn) >> shift) == prefix;
        const unsigned bb = __ballot_sync(kFull, in);
        if (in && satk_check(got + __popc(bb & lt) < 32, kDbgHist))
          ws.hist[got + __popc(bb & lt)] = k;
        got += __popc(bb);
      }
      __syncwarp();
      const uint32_t mine = lane < got ? ws.hist[lane] : 0u;
      __syncwarp();
      if (lane < got) ws.hist[lane] = 0u;
      int gt = 0, eq = 0;
      for (int j = 0; j < got; ++j) {
        const uint32_t x = __shfl_sync(kFull, mine, j);
        gt += x > mine;
        eq += x == mine;
      }
      const bool hit = lane < got && gt < need && need <= gt + eq;
      const int src = __ffs(__ballot_sync(kFull, hit)) - 1;
      v = __shfl_sync(kFull, mine, src);
      takeB = need - __shfl_sync(kFull, gt, src);
      found = true;
      __syncwarp();
      break;
    }
    if (p.cnt == need) {  // the whole digit is taken: v is its smallest key
      const uint32_t lo = prefix << shift;
      uint32_t m = 0xffffffffu;
      for (int i = lane; i < n; i += 32)
        if (lk[i] - mn >= lo) m = min(m, lk[i]);
      v = __reduce_min_sync(kFull, m);
      int c = 0;
      for (int i = lane; i < n; i += 32) c += lk[i] == v;
      takeB = static_cast<int>(__reduce_add_sync(kFull, static_cast<unsigned>(c)));
      found = true;
      break;
    }
  }
  if (!found) {  // every bit resolved: v = mn + prefix, `need` of its ties
    v = mn + prefix;
    takeB = need;
  }
  const int cgt = K - takeB;
  int runA = 0, runB = 0;
  for (int i0 = 0; i0 < n; i0 += 32) {
    const int i = i0 + lane;
    const uint32_t k = i < n ? lk[i] : 0u;
    const unsigned ba = __ballot_sync(kFull, k > v);
    const unsigned bb = __ballot_sync(kFull, k == v && i < n);
    if ((ba >> lane) & 1u) dst.put_entry(runA + __popc(ba & lt), i, k, static_cast<int>(lc[i]));
    if ((bb >> lane) & 1u) {
      const int pb = runB + __popc(bb & lt);
      if (pb < takeB) dst.put_entry(cgt + pb, i, k, static_cast<int>(lc[i]));
    }
    runA += __popc(ba);
    runB += __popc(bb);
  }
}

// The whole row on one warp.  The histogram must be zero on entry and is
// zero again on return.
template <typename T, int ALIGN, class Out>
__device__ void warp_topk_row(const T *__restrict__ xr, int end, int K, const Out &dst,
                              WarpRowSmem &ws) {
  // the copy engine starts on the first batch of the filtered pass
  prefetch_groups<T, ALIGN>(xr, 0, min(end / 8, 32 * 4));
  const bool all = end <= kWarpList;
  float t0f = __uint_as_float(0xff800000u);  // -inf: every valid column
  if (!all) t0f = warp_sample_threshold<T, ALIGN>(xr, end, K, ws);
  __syncwarp();  // the sampled values are read before the list overwrites them
  int n;
  WarpRange lr;
  const bool fits = warp_collect<T, ALIGN>(xr, end, t0f, ws, n);
  if (fits && (all || n >= K))
    lr = warp_list_keys<T>(ws, n);
  else
    warp_collect_exact<T>(xr, end, K, ws, lr);
  warp_emit(ws, lr, K, dst);
}

}  // namespace satk
