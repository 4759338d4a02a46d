// satk_rows.cuh -- exact top-K of one row of fp32 or bf16 logits.
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
// One CTA per row, three steps:
//  1. threshold: a sample of the row (4 columns per thread) is ranked (to
//     24 bits of its key range) and a key T0 picked so that, with a margin of about four
//     standard deviations of the sampling error, at least K columns of the
//     row score at or above it.  Rows no longer than the list capacity skip
//     this and take every valid column.
//  2. collection: the row is streamed from HBM once, each warp over its own
//     contiguous stretch of columns; a column is kept when its score
//     compares >= T0 as a float (one compare per element; NaN never
//     passes).  Kept columns are ballot-compacted, in column order, into
//     the warp's segment of the shared-memory list.
//  3. select: the exact K-th key on the list, then the ordered emit.
// The collection is exact, never approximate: it fails only when the list
// is too short (T0 above the K-th key) or a warp's segment overflows, and
// then the row is redone by the two-pass method below, which always fits:
// a digit histogram of the whole row picks the threshold digit (narrowed by
// more digit passes until its candidates fit the list), then an ordered
// collection pass gathers the candidates.
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "satk_list.cuh"

namespace satk {

template <typename T>
__device__ __forceinline__ float as_float(uint32_t raw) {  // one element's bits
  if constexpr (std::is_same<T, float>::value)
    return __uint_as_float(raw);
  else
    return __uint_as_float(raw << 16);
}
template <typename T>
__device__ __forceinline__ uint32_t key_of_raw(uint32_t raw) {
  if constexpr (std::is_same<T, float>::value)
    return key_f32(raw);
  else
    return key_bf16(raw);
}
template <typename T>
__device__ __forceinline__ uint32_t key_of_num(uint32_t raw) {  // raw not NaN
  if constexpr (std::is_same<T, float>::value)
    return key_f32_num(raw);
  else
    return key_bf16_num(raw);
}
template <typename T>
__device__ __forceinline__ uint32_t load_raw(const T *p) {
  if constexpr (std::is_same<T, float>::value)
    return __float_as_uint(__ldg(p));
  else
    return __ldg(reinterpret_cast<const unsigned short *>(p));
}

// ------------------------------------------------------------ threshold --

// A float as an int with the same order (for warp and block minima and maxima).
__device__ __forceinline__ int float_order(float f) {
  const int i = __float_as_int(f);
  return i ^ ((i >> 31) & 0x7fffffff);
}
__device__ __forceinline__ float float_of_order(int i) {
  return __int_as_float(i ^ ((i >> 31) & 0x7fffffff));
}

// Bin of x in a value-linear histogram of 256 bins starting at lo, sc bins
// per unit; values below lo go to bin 0, above the top to bin 255.
__device__ __forceinline__ int value_bin(float x, float lo, float sc) {
  return min(255, max(0, __float2int_rz((x - lo) * sc)));
}

// The largest value of T's grid at or below t (bf16 thresholds compare
// exactly as floats only on the bf16 grid).
template <typename T>
__device__ __forceinline__ float grid_floor(float t) {
  if constexpr (std::is_same<T, float>::value) {
    return t;
  } else {
    uint32_t b = __float_as_uint(t);
    b = (b & 0x80000000u) ? ((b + 0xffffu) & 0xffff0000u) : (b & 0xffff0000u);
    return __uint_as_float(b);
  }
}


// Loads the sample of a row: BLOCK*SPT columns in BLOCK*SPT/32 runs of 32
// consecutive columns spread evenly over [0, end), one coalesced load per
// warp and run, so the sample touches few memory sectors.  Their keys go to
// the first 32*SPT entries of each warp's list segment.  Needs
// end >= BLOCK * SPT.
template <typename T, int BLOCK, int SPT, int SUB>
__device__ __forceinline__ Seg sample_keys(const T *__restrict__ xr, int end,
                                           ListSmem<BLOCK, SUB> &sm) {
  static_assert(SPT * 32 <= SUB, "samples must fit a warp segment");
  constexpr int NRUNS = BLOCK * SPT / 32;
  const int lane = lane_id(), warp = warp_id();
  uint32_t raw[SPT];
#pragma unroll
  for (int q = 0; q < SPT; ++q) {
    const int run = warp * SPT + q;
    const int start = static_cast<int>((static_cast<int64_t>(run) * end) / NRUNS) & ~31;
    raw[q] = load_raw(xr + start + lane);
  }
#pragma unroll
  for (int q = 0; q < SPT; ++q) sm.key[warp * SUB + q * 32 + lane] = key_of_raw<T>(raw[q]);
  __syncwarp();
  return Seg{warp * SUB, 32 * SPT};
}

// The rank r of the sample's key that is T0: with mu = K * samples / end
// columns of the top K expected in the sample, r = mu + 4 sqrt(mu) + 4 makes
// P(fewer than K columns of the row have key >= T0) negligible under random
// sampling.
__device__ __forceinline__ int sample_rank(int K, int samples, int end) {
  const float mu = static_cast<float>(K) * samples / static_cast<float>(end);
  const int r = static_cast<int>(ceilf(mu + 4.f * sqrtf(mu) + 4.f));
  return r < 1 ? 1 : (r > samples ? samples : r);
}

// T0 of a row: the r-th largest key of its sample (sample_keys,
// sample_rank); 1 (every valid column) when the sample holds fewer than r
// valid keys.
template <typename T, int BLOCK, int SPT, int SUB>
__device__ uint32_t sample_threshold(const T *__restrict__ xr, int end, int K,
                                     ListSmem<BLOCK, SUB> &sm) {
  const Seg sg = sample_keys<T, BLOCK, SPT, SUB>(xr, end, sm);
  const int r = sample_rank(K, BLOCK * SPT, end);
  const Sel s = list_select<BLOCK>([&](int i) { return sm.key[i]; }, sg, r, sm.sel, 3);
  return s.take_all ? 1u : s.T;
}

// The threshold of a block's sample of SPT values per thread (NaN: no
// candidate) for rank r: a value-linear histogram of 256 bins over the
// sample's [min, max], the r-th largest value's bin edge (one finer pass
// inside a bin holding more than 32 samples), a little below the edge so
// that rounding drops no counted sample.  One pass and three block
// barriers where the ordered-key digits take up to three passes.  -inf when
// fewer than r values are valid; ok = false when the range is not usable
// (an infinity, a single value): the caller then ranks by ordered keys.
template <int BLOCK, int SPT>
__device__ float block_value_threshold(const float (&v)[SPT], int r, SelectSmem<BLOCK> &sel,
                                       bool &ok) {
  constexpr int NW = BLOCK / 32;
  const int lane = lane_id(), warp = warp_id();
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
  int imn = sel.wtot[1][0], imx = sel.wtot[2][0];
#pragma unroll
  for (int w = 1; w < NW; ++w) {
    imn = min(imn, sel.wtot[1][w]);
    imx = max(imx, sel.wtot[2][w]);
  }
  mn = float_of_order(imn);
  mx = float_of_order(imx);
  ok = true;
  const float ninf = __uint_as_float(0xff800000u);
  if (mx < mn) return ninf;  // no valid sample (block-uniform)
  const float span = mx - mn;
  if (!(span > 0.f) || !(span < __uint_as_float(0x7f800000u))) {
    // block-uniform; the caller's fallback select writes wtot[1] and
    // wtot[2] next, so every warp must have read them first
    __syncthreads();
    ok = false;
    return 0.f;
  }
  const float sc = 256.f * __frcp_rn(span);
#pragma unroll
  for (int q = 0; q < SPT; ++q)
    if (v[q] == v[q]) atomicAdd(sel.hist + value_bin(v[q], mn, sc), 1u);
  __syncthreads();
  const PassOut p = find_threshold<BLOCK, 256>(sel, r);
  if (p.d < 0) return ninf;  // fewer than r valid samples
  float t = mn + static_cast<float>(p.d) * __frcp_rn(sc);
  if (p.cnt > 32 && p.d < 255) {  // block-uniform: a crowded bin, a finer pass inside it
    const float sc2 = sc * 256.f;
    const float lo2 = t;
#pragma unroll
    for (int q = 0; q < SPT; ++q)
      if (v[q] == v[q] && value_bin(v[q], mn, sc) == p.d)
        atomicAdd(sel.hist + value_bin(v[q], lo2, sc2), 1u);
    __syncthreads();
    const PassOut p2 = find_threshold<BLOCK, 256>(sel, r - p.above);
    t = lo2 + static_cast<float>(p2.d) * __frcp_rn(sc2);
  }
  return t - fabsf(t) * 9.5367e-7f - 1e-37f;
}

// T0 of a row from block_value_threshold over the same sample as
// sample_threshold (the values kept in registers).  On T's grid.
template <typename T, int BLOCK, int SPT, int SUB>
__device__ float value_sample_threshold(const T *__restrict__ xr, int end, int K,
                                        ListSmem<BLOCK, SUB> &sm, bool &ok) {
  constexpr int NRUNS = BLOCK * SPT / 32;
  const int lane = lane_id(), warp = warp_id();
  float v[SPT];
#pragma unroll
  for (int q = 0; q < SPT; ++q) {
    const int run = warp * SPT + q;
    const int start = static_cast<int>((static_cast<int64_t>(run) * end) / NRUNS) & ~31;
    v[q] = as_float<T>(load_raw(xr + start + lane));
  }
  const float t = block_value_threshold<BLOCK, SPT>(v, sample_rank(K, BLOCK * SPT, end), sm.sel,
                                                    ok);
  return grid_floor<T>(t);
}

// ---------------------------------------------------- single-pass filter --

// 8 consecutive elements of one lane: loads and the kept-column mask (bit s
// set when element s compares >= the threshold; NaN never does).
// ALIGN 32: one 32-byte load (fp32, rows 32-byte aligned); 16: two 16-byte
// loads (fp32) or one (bf16); 0: scalar loads.
template <typename T, int ALIGN>
struct Group8;

template <int ALIGN>
struct Group8<float, ALIGN> {
  uint32_t w[8];
  // raw bits of element s (s not a compile-time constant: a select tree)
  __device__ __forceinline__ uint32_t raw(int s) const {
    const uint32_t a0 = (s & 1) ? w[1] : w[0], a1 = (s & 1) ? w[3] : w[2];
    const uint32_t a2 = (s & 1) ? w[5] : w[4], a3 = (s & 1) ? w[7] : w[6];
    const uint32_t b0 = (s & 2) ? a1 : a0, b1 = (s & 2) ? a3 : a2;
    return (s & 4) ? b1 : b0;
  }
  __device__ __forceinline__ void load(const float *p) {
    if constexpr (ALIGN == 32) {
      asm volatile(
          "ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
          : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
            "=r"(w[7])
          : "l"(p));
    } else if constexpr (ALIGN == 16) {
      const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
      const uint4 b = __ldg(reinterpret_cast<const uint4 *>(p) + 1);
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
      w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
    } else {
#pragma unroll
      for (int s = 0; s < 8; ++s) w[s] = __float_as_uint(__ldg(p + s));
    }
  }
  __device__ __forceinline__ uint32_t mask(float t) const {
    uint32_t m = 0;
#pragma unroll
    for (int s = 0; s < 8; ++s) m |= (__uint_as_float(w[s]) >= t ? 1u : 0u) << s;
    return m;
  }
  // the raw words to / from 32 bytes of shared memory (16-byte aligned)
  __device__ __forceinline__ void stash(uint32_t *p) const {
    reinterpret_cast<uint4 *>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4 *>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
  __device__ __forceinline__ void unstash(const uint32_t *p) {
    const uint4 a = reinterpret_cast<const uint4 *>(p)[0];
    const uint4 b = reinterpret_cast<const uint4 *>(p)[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
  // whether some element compares >= t (the maximum ignores NaN)
  __device__ __forceinline__ bool any(float t) const {
    const float a = fmaxf(fmaxf(__uint_as_float(w[0]), __uint_as_float(w[1])),
                          fmaxf(__uint_as_float(w[2]), __uint_as_float(w[3])));
    const float b = fmaxf(fmaxf(__uint_as_float(w[4]), __uint_as_float(w[5])),
                          fmaxf(__uint_as_float(w[6]), __uint_as_float(w[7])));
    return fmaxf(a, b) >= t;
  }
};

template <int ALIGN>
struct Group8<uint16_t, ALIGN> {
  uint32_t w[4];  // two bf16 per word, element 2j in the low half
  __device__ __forceinline__ uint32_t raw(int s) const {
    const uint32_t a0 = (s & 2) ? w[1] : w[0], a1 = (s & 2) ? w[3] : w[2];
    const uint32_t b = (s & 4) ? a1 : a0;
    return (s & 1) ? (b >> 16) : (b & 0xffffu);
  }
  __device__ __forceinline__ void load(const uint16_t *p) {
    if constexpr (ALIGN != 0) {
      const uint4 a = ldg_stream(p);
      w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    } else {
      const unsigned short *q = reinterpret_cast<const unsigned short *>(p);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        w[j] = static_cast<uint32_t>(__ldg(q + 2 * j)) |
               (static_cast<uint32_t>(__ldg(q + 2 * j + 1)) << 16);
    }
  }
  __device__ __forceinline__ uint32_t mask(__nv_bfloat162 t2) const {
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t h = __hge2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w[j]), t2);
      m |= ((h & 1u) | ((h >> 15) & 2u)) << (2 * j);
    }
    return m;
  }
  // the raw words to / from 16 bytes of shared memory (16-byte aligned)
  __device__ __forceinline__ void stash(uint32_t *p) const {
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  __device__ __forceinline__ void unstash(const uint32_t *p) {
    const uint4 a = *reinterpret_cast<const uint4 *>(p);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  }
  // whether some element compares >= t (the maximum ignores NaN)
  __device__ __forceinline__ bool any(__nv_bfloat162 t2) const {
    const __nv_bfloat162 *v = reinterpret_cast<const __nv_bfloat162 *>(w);
    const __nv_bfloat162 m = __hmax2(__hmax2(v[0], v[1]), __hmax2(v[2], v[3]));
    return __hge2_mask(m, t2) != 0u;
  }
};

template <typename T>
struct ThresholdOf;
template <>
struct ThresholdOf<float> {
  float t;
  __device__ __forceinline__ explicit ThresholdOf(float f) : t(f) {}
  __device__ __forceinline__ float arg() const { return t; }
};
template <>
struct ThresholdOf<uint16_t> {
  __nv_bfloat162 t2;
  __device__ __forceinline__ explicit ThresholdOf(float f) {
    // f is a bf16 value, or has only low-half bits below one (negative
    // thresholds carry 0xffff there): round toward -inf to the bf16 grid,
    // which admits exactly the same bf16 inputs
    uint32_t b = __float_as_uint(f) >> 16;
    const __nv_bfloat16 h = *reinterpret_cast<const __nv_bfloat16 *>(&b);
    t2 = __halves2bfloat162(h, h);
  }
  __device__ __forceinline__ __nv_bfloat162 arg() const { return t2; }
};

// The warp's stretch of 8-element groups: [g0, g1) of end / 8 groups.
template <int BLOCK>
__device__ __forceinline__ void warp_stretch(int end, int &g0, int &g1) {
  constexpr int NW = BLOCK / 32;
  const int ngroups = end / 8;
  const int per = (ngroups + NW - 1) / NW;
  g0 = min(ngroups, warp_id() * per);
  g1 = min(ngroups, g0 + per);
}

// L2 prefetch of groups [ga, gb) of the warp's stretch (16-byte rows only),
// issued by lane 0, split in pieces of at most 64 KB.
template <typename T, int ALIGN>
__device__ __forceinline__ void prefetch_groups(const T *__restrict__ xr, int ga, int gb) {
  if constexpr (ALIGN != 0) {
    if (lane_id() == 0 && ga < gb) {
      constexpr uint32_t GB = 8 * sizeof(T);  // bytes per group (16 or 32)
      const char *p = reinterpret_cast<const char *>(xr) + static_cast<size_t>(ga) * GB;
      uint32_t left = static_cast<uint32_t>(gb - ga) * GB;
      while (left != 0u) {
        const uint32_t piece = left < 65536u ? left : 65536u;
        prefetch_l2(p, piece);
        p += piece;
        left -= piece;
      }
    }
  }
}

// Groups per lane per batch of the filtered pass, and samples per thread of
// the cluster path's threshold step (a slice there is only known to exceed
// CAP - 8 columns, and the sample needs BLOCK * samples of them).
constexpr int kRowBatch = 4;
constexpr int kRowSample = 4;

// Samples per thread of the CTA path's threshold step (its rows exceed CAP
// >= BLOCK * 16 columns): a larger sample tightens the threshold, so the
// list shrinks toward K, at the cost of its loads and histogram.  Measured
// best: 8 for fp32 rows (4096 x 51200, K 512: 167 -> 164 us against 4; 16
// was slower at 25600 columns) and 16 for bf16 rows (the decode top-384 pack
// of 65536 columns: 50 -> 46 us against 4), whose small K per column left
// the 4-sample threshold loosest.
template <typename T>
__host__ __device__ constexpr int row_sample() {
  return sizeof(T) == 2 ? 16 : 8;
}

// L2 prefetch of the first two batches of every warp's stretch of a row of
// `end` columns: what the filtered pass reads first.
template <typename T, int BLOCK, int ALIGN>
__device__ __forceinline__ void prefetch_row_head(const T *__restrict__ xr, int end) {
  int g0, g1;
  warp_stretch<BLOCK>(end, g0, g1);
  prefetch_groups<T, ALIGN>(xr, g0, min(g1, g0 + 2 * 32 * kRowBatch));
}

// Every warp streams its own contiguous stretch of 8-element groups (one
// group per lane, U per lane in flight) and records the columns whose score
// compares >= the threshold, with their keys, in its list segment, in
// column order.  The copy engine keeps the L2 PF batches ahead of the
// warp's loads (the first ones were requested before the threshold step).  Per-lane counts of each batch go
// through one packed warp prefix scan.  The < 8 ragged columns at the end
// go to the last warp.  Returns the segment; sets sm.flag on overflow.
// (The element-wise form of collect_filtered, for stretches whose groups
// mostly pass.)
template <typename T, int BLOCK, int SUB, int ALIGN, int U>
__device__ __forceinline__ Seg collect_filtered_elems(const T *__restrict__ xr, int end,
                                                      float t0f, ListSmem<BLOCK, SUB> &sm,
                                                      WarpStats &st) {
  static_assert(U % 2 == 0, "counts are packed two per word");
  constexpr int NW = BLOCK / 32;
  constexpr int PF = 1;  // batches prefetched ahead (more is evicted before use)
  const int lane = lane_id(), warp = warp_id();
  const int ngroups = end / 8;
  int g0, g1;
  warp_stretch<BLOCK>(end, g0, g1);
  uint32_t *lk = sm.key + warp * SUB;
  uint32_t *lv = sm.val + warp * SUB;
  const ThresholdOf<T> thr(t0f);
  int cnt = 0;
  uint32_t kmn = 0xffffffffu, kmx = 0u;  // range of the keys written
  for (int gb = g0; gb < g1; gb += 32 * U) {
    prefetch_groups<T, ALIGN>(xr, min(g1, gb + PF * 32 * U), min(g1, gb + (PF + 1) * 32 * U));
    Group8<T, ALIGN> grp[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gi = gb + u * 32 + lane;
      if (gi < g1) grp[u].load(xr + static_cast<size_t>(gi) * 8);
    }
    uint32_t m[U];
    uint32_t pk[U / 2];
#pragma unroll
    for (int j = 0; j < U / 2; ++j) pk[j] = 0u;
    uint32_t any = 0u;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gi = gb + u * 32 + lane;
      m[u] = gi < g1 ? grp[u].mask(thr.arg()) : 0u;
      pk[u >> 1] |= static_cast<uint32_t>(__popc(m[u])) << (16 * (u & 1));
      any |= m[u];
    }
    if (!__any_sync(kFull, any != 0u)) continue;
    uint32_t incl[U / 2], tot[U / 2];
    int btot = 0;
#pragma unroll
    for (int j = 0; j < U / 2; ++j) {
      incl[j] = static_cast<uint32_t>(warp_incl_scan(static_cast<int>(pk[j])));
      tot[j] = __shfl_sync(kFull, incl[j], 31);
      btot += static_cast<int>((tot[j] & 0xffffu) + (tot[j] >> 16));
    }
    if (cnt + btot > SUB) {  // warp-uniform: the segment overflows
      cnt += btot;
      break;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint32_t lc = static_cast<uint32_t>(__popc(m[u]));
      int pos = cnt + static_cast<int>(((incl[u >> 1] >> (16 * (u & 1))) & 0xffffu) - lc);
      uint32_t mm = m[u];
      const int c0 = (gb + u * 32 + lane) * 8;
      while (mm != 0u) {
        const int s = __ffs(mm) - 1;
        mm &= mm - 1u;
        const uint32_t k = key_of_num<T>(grp[u].raw(s));
        if (satk_check(pos < SUB, kDbgList)) {
          lk[pos] = k;
          lv[pos] = static_cast<uint32_t>(c0 + s);
        }
        kmn = min(kmn, k);
        kmx = max(kmx, k);
        ++pos;
      }
      cnt += static_cast<int>((tot[u >> 1] >> (16 * (u & 1))) & 0xffffu);
    }
  }
  if (warp == NW - 1 && ngroups * 8 < end && cnt <= SUB) {  // ragged columns
    const int c = ngroups * 8 + lane;
    const uint32_t rw = c < end ? load_raw(xr + c) : 0u;
    const bool keep = c < end && as_float<T>(rw) >= t0f;
    const unsigned b = __ballot_sync(kFull, keep);
    const int pos = cnt + __popc(b & ((1u << lane) - 1u));
    if (keep && pos < SUB) {
      const uint32_t k = key_of_num<T>(rw);
      lk[pos] = k;
      lv[pos] = static_cast<uint32_t>(c);
      kmn = min(kmn, k);
      kmx = max(kmx, k);
    }
    cnt += __popc(b);
  }
  if (cnt > SUB && lane == 0) sm.flag = 1;
  st.n = min(cnt, SUB);
  st.mn = __reduce_min_sync(kFull, kmn);
  st.mx = __reduce_max_sync(kFull, kmx);
  return Seg{warp * SUB, min(cnt, SUB)};
}

// The filtered pass for thresholds that keep few columns.  Every warp
// streams its stretch of 8-element groups (one group per lane, U per lane
// in flight, the copy engine a batch ahead) and tests each group by its
// maximum against the threshold; a ballot stages the groups that pass --
// their raw words in the warp's share of the idle histogram, their indices
// in the last 32 entries of its list segment -- and each time 32 are
// staged the warp takes them one per lane: the columns that compare >= the
// threshold go, with their keys, to the list segment in column order
// (per-lane counts through a warp prefix scan).  So the per-column work
// runs only on passing groups, and nothing is read twice.  fp32 rows and an
// unbounded threshold (every group passes) take collect_filtered_elems
// instead.
// The < 8 ragged columns at the end go to the last warp.  Returns the
// segment; sets sm.flag on overflow.  The histogram is zero on entry and
// on return.
template <typename T, int BLOCK, int SUB, int ALIGN, int U>
__device__ __forceinline__ Seg collect_filtered(const T *__restrict__ xr, int end, float t0f,
                                                ListSmem<BLOCK, SUB> &sm, WarpStats &st) {
  using G = Group8<T, ALIGN>;
  constexpr int NW = BLOCK / 32;
  constexpr int GW = sizeof(G::w) / sizeof(uint32_t);  // words per group
  static_assert(32 * GW <= 2048 / NW, "32 staged groups per warp fit its histogram share");
  constexpr int LCAP = SUB - 32;  // list entries; the last 32 hold staged indices
  constexpr int PF = 1;           // batches prefetched ahead
  const int lane = lane_id(), warp = warp_id();
  const unsigned lt = (1u << lane) - 1u;
  // fp32 rows stay on the element path: their 32-byte groups leave the
  // staging loop short of registers (measured slower at 25600 - 102400
  // columns), while bf16 rows gain
  if (std::is_same<T, float>::value || !(t0f > __uint_as_float(0xff800000u)))
    return collect_filtered_elems<T, BLOCK, SUB, ALIGN, U>(xr, end, t0f, sm, st);
  const int ngroups = end / 8;
  int g0, g1;
  warp_stretch<BLOCK>(end, g0, g1);
  uint32_t *stw = sm.sel.hist + warp * (2048 / NW);  // staged groups' words
  uint32_t *lk = sm.key + warp * SUB;
  uint32_t *lv = sm.val + warp * SUB;
  uint32_t *sgi = lv + LCAP;  // staged groups' indices
  const ThresholdOf<T> thr(t0f);
  int cnt = 0, staged = 0;
  bool over = false;  // warp-uniform: the list segment overflowed
  uint32_t kmn = 0xffffffffu, kmx = 0u;  // range of the keys written
  auto flush = [&]() {  // warp-uniform; the staged groups, one per lane
    __syncwarp();
    G grp;
    uint32_t m = 0u;
    int gi = 0;
    if (lane < staged) {
      grp.unstash(stw + lane * GW);
      gi = static_cast<int>(sgi[lane]);
      m = grp.mask(thr.arg());
    }
    const int lc = __popc(m);
    const int incl = warp_incl_scan(lc);
    const int tot = __shfl_sync(kFull, incl, 31);
    if (cnt + tot > LCAP) {
      over = true;
    } else {
      int pos = cnt + incl - lc;
      const int c0 = gi * 8;
      while (m != 0u) {
        const int s = __ffs(m) - 1;
        m &= m - 1u;
        const uint32_t k = key_of_num<T>(grp.raw(s));
        if (satk_check(pos < LCAP, kDbgList)) {
          lk[pos] = k;
          lv[pos] = static_cast<uint32_t>(c0 + s);
        }
        kmn = min(kmn, k);
        kmx = max(kmx, k);
        ++pos;
      }
    }
    cnt += tot;
    staged = 0;
    __syncwarp();
  };
  for (int gb = g0; gb < g1 && !over; gb += 32 * U) {
    prefetch_groups<T, ALIGN>(xr, min(g1, gb + PF * 32 * U), min(g1, gb + (PF + 1) * 32 * U));
    G grp[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gi = gb + u * 32 + lane;
      if (gi < g1) grp[u].load(xr + static_cast<size_t>(gi) * 8);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int gi = gb + u * 32 + lane;
      const bool p = gi < g1 && grp[u].any(thr.arg());
      const unsigned b = __ballot_sync(kFull, p);
      if (b != 0u) {  // warp-uniform
        const int c = __popc(b);
        if (staged + c > 32) flush();
        if (p) {
          const int slot = staged + __popc(b & lt);
          grp[u].stash(stw + slot * GW);
          sgi[slot] = static_cast<uint32_t>(gi);
        }
        staged += c;
      }
    }
  }
  if (staged != 0 && !over) flush();
  __syncwarp();
#pragma unroll
  for (int w = lane; w < 32 * GW; w += 32) stw[w] = 0u;  // the histogram zero again
  if (warp == NW - 1 && ngroups * 8 < end && !over) {  // ragged columns
    const int c = ngroups * 8 + lane;
    const uint32_t rw = c < end ? load_raw(xr + c) : 0u;
    const bool keep = c < end && as_float<T>(rw) >= t0f;
    const unsigned b = __ballot_sync(kFull, keep);
    const int pos = cnt + __popc(b & lt);
    if (keep && pos < LCAP) {
      const uint32_t k = key_of_num<T>(rw);
      lk[pos] = k;
      lv[pos] = static_cast<uint32_t>(c);
      kmn = min(kmn, k);
      kmx = max(kmx, k);
    }
    cnt += __popc(b);
    over = cnt > LCAP;
  }
  if (over && lane == 0) sm.flag = 1;
  st.n = min(cnt, LCAP);
  st.mn = __reduce_min_sync(kFull, kmn);
  st.mx = __reduce_max_sync(kFull, kmx);
  return Seg{warp * SUB, min(cnt, LCAP)};
}

// ------------------------------------------------------ exact (fallback) --

// Visits the row [0, end) tile by tile with a warp-contiguous mapping: in a
// tile of BLOCK*U vectors, warp w owns vectors [w*32*U, (w+1)*32*U) and
// lane l reads vector w*32*U + u*32 + l at step u (coalesced per step).
// body(kk, col) gets the lane's U*VEC keys (0 past the end) and the column
// of kk[u*VEC] in col[u]; every thread makes the same calls, so body may
// use warp collectives and barriers.  A last call to tail(k, c) covers the
// < VEC ragged columns (warp 0, one per lane).
template <typename T, int BLOCK, int U, bool VECLOAD, class Body, class TailBody>
__device__ __forceinline__ void for_row_tiles(const T *__restrict__ xr, int end, Body body,
                                              TailBody tail) {
  constexpr int VEC = VECLOAD ? KeyOf<T>::kVec : 1;
  const int lane = lane_id(), warp = warp_id();
  const int nvec = end / VEC;
  for (int tile = 0; tile < nvec; tile += BLOCK * U) {
    uint32_t kk[U * VEC];
    int col[U];
    if constexpr (VECLOAD) {
      uint4 raw[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int vi = tile + warp * (32 * U) + u * 32 + lane;
        col[u] = vi * VEC;
        if (vi < nvec) raw[u] = ldg_stream(xr + static_cast<size_t>(vi) * VEC);
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

// The two-pass method: digit histogram(s) of the whole row, then an ordered
// collection of every candidate at or above the threshold digit into the
// list [0, CAP).  At full key resolution with a tie wider than the list,
// only the first `need` tied columns are kept, so the list never exceeds K
// there.  Returns this warp's share of the list.
template <typename T, int BLOCK, int SUB, bool VECLOAD>
__device__ Seg collect_exact(const T *__restrict__ xr, int end, int K,
                             ListSmem<BLOCK, SUB> &sm) {
  constexpr int VEC = VECLOAD ? KeyOf<T>::kVec : 1;
  constexpr int U = VECLOAD ? 8 / VEC : 8;  // 8 keys per lane per tile
  constexpr int KB = KeyOf<T>::kBits;
  constexpr int CAP = ListSmem<BLOCK, SUB>::CAP;
  constexpr int NK = U * VEC;
  constexpr int NW = BLOCK / 32;
  static_assert(BLOCK * U * VEC < 65536, "tile counts must fit 16 bits");
  SelectSmem<BLOCK> &ss = sm.sel;
  const int lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;

  // ---- pass 1: top-digit histogram
  for_row_tiles<T, BLOCK, U, VECLOAD>(
      xr, end,
      [&](const uint32_t *kk, const int *) {
#pragma unroll
        for (int j = 0; j < NK; ++j) hist_add<true>(ss.hist, kk[j] >> 21, kk[j] != 0u);
      },
      [&](uint32_t k, int) { hist_add<true>(ss.hist, k >> 21, k != 0u); });
  __syncthreads();
  PassOut p = find_threshold<BLOCK, 2048>(ss, K);

  uint32_t thr;
  bool limited = false;
  int need = K;
  if (p.d < 0) {
    thr = 1u;  // fewer than K valid: every valid column
  } else {
    uint32_t prefix = static_cast<uint32_t>(p.d);
    int pbits = 11;
    int above = p.above;
    int cnt = p.cnt;
    need = K - above;
    while (above + cnt > CAP && pbits < KB) {  // narrow the threshold digit
      const int width = (KB - pbits >= 11) ? 11 : (KB - pbits);
      const int shift = 32 - pbits - width;
      const uint32_t dmask = (1u << width) - 1u;
      const int pb = pbits;
      const uint32_t pf = prefix;
      auto visit = [&](uint32_t k) {
        hist_add<true>(ss.hist, (k >> shift) & dmask, k != 0u && (k >> (32 - pb)) == pf);
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
      prefix = (prefix << width) | static_cast<uint32_t>(p.d);
      pbits += width;
    }
    thr = prefix << (32 - pbits);
    limited = above + cnt > CAP;  // full resolution, tie too wide: keep `need`
  }

  // ---- ordered collection into the list
  int runA = 0, runB = 0;
  int par = 0;
  auto collect = [&](const uint32_t *kk, const int *col, auto nk_tag, auto vec_tag) {
    constexpr int NKT = decltype(nk_tag)::value;
    constexpr int VT = decltype(vec_tag)::value;
    int ca = 0, cb = 0;
#pragma unroll
    for (int j = 0; j < NKT; ++j) {
      const uint32_t k = kk[j];
      ca += __popc(__ballot_sync(kFull, limited ? (k > thr) : (k >= thr)));
      cb += __popc(__ballot_sync(kFull, limited && k == thr));
    }
    int tot;
    const unsigned base =
        (unsigned)block_warp_prefix<BLOCK>((ca << 16) | cb, ss.wtot[par], &tot);
    par ^= 1;
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
          sm.key[pos] = k;
          sm.val[pos] = static_cast<uint32_t>(col[u] + s);
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
  const int chunk = (nlist + NW - 1) / NW;
  const int b0 = min(nlist, warp_id() * chunk);
  return Seg{b0, min(nlist, b0 + chunk) - b0};
}

// ----------------------------------------------------------------- a row --

// The whole row: threshold, collection (exact fallback when needed), select
// and emit.  put(pos, i) stores list entry i at output position pos;
// fill(pos) pads [n, K).  The histogram must be zero on entry and is zero
// again on return.
template <typename T, int BLOCK, int SUB, int ALIGN, class Put, class Fill>
__device__ void topk_row(const T *__restrict__ xr, int end, int K, Put put, Fill fill,
                         ListSmem<BLOCK, SUB> &sm) {
  constexpr int KB = KeyOf<T>::kBits;
  constexpr int CAP = ListSmem<BLOCK, SUB>::CAP;
  constexpr bool VECLOAD = ALIGN != 0;
  constexpr int U = kRowBatch;
  static_assert(CAP >= BLOCK * row_sample<T>(), "a sampled row (end > CAP) holds the sample");
  const bool all = end <= CAP;
  // start the copy engine on the first batches of this warp's stretch
  prefetch_row_head<T, BLOCK, ALIGN>(xr, end);
  float t0f;
  if (all) {
    t0f = __uint_as_float(0xff800000u);  // -inf: every valid column
  } else {
    bool ok;
    t0f = value_sample_threshold<T, BLOCK, row_sample<T>(), SUB>(xr, end, K, sm, ok);
    if (!ok)  // block-uniform
      t0f = threshold_float<KB>(sample_threshold<T, BLOCK, row_sample<T>(), SUB>(xr, end, K, sm));
  }
  if (threadIdx.x == 0) sm.flag = 0;
  __syncthreads();  // sample keys read, flag clear
  WarpStats st;
  Seg sg = collect_filtered<T, BLOCK, SUB, ALIGN, U>(xr, end, t0f, sm, st);
  // wtot[3]: its next writer (the list emit) is behind the select's barriers
  int total;
  block_warp_prefix<BLOCK>(sg.cnt, sm.sel.wtot[3], &total);
  const bool ok = sm.flag == 0 && (all || total >= K);
  if (!ok) {  // block-uniform
    __syncthreads();
    sg = collect_exact<T, BLOCK, SUB, VECLOAD>(xr, end, K, sm);
  }
  // bf16 keys are ord16 << 16: their low 16 bits are zero
  list_topk_emit<BLOCK, SUB>(sm, sg, K, put, fill, ok ? st : stats_unknown(), 32 - KB);
}

}  // namespace satk
