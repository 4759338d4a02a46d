// satk_device.cuh -- device building blocks of the exact top-K kernels.
//
// Ordered keys.  Every candidate becomes an unsigned 32-bit key whose
// integer order is the score order, with 0 reserved for "no candidate"
// (NaN, past the row end, an empty slot):
//   fp32 : the IEEE bits, negatives bit-inverted, non-negatives with the
//          sign bit set (so -0.0 sits just below +0.0 and +-inf are the
//          ends of the range);
//   bf16 : the 16-bit version of the same map placed in the top half
//          (vLLM API page vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge
//          .kernels, section _ord16), low half zero.
// A NaN pattern would map to 0 or above +inf, so NaNs are tested first and
// given key 0.
//
// Select.  A most-significant-digit radix select over those keys finds the
// K-th key (11-bit digits, shared-memory histograms, one block-wide scan
// per digit; the same page, _make_radix_select, uses 9-bit digits over a
// 512-thread block).  Candidates live in registers: thread t of warp w holds
// slot i at flat position w*32*KPT + (i/VEC)*32*VEC + lane*VEC + i%VEC, so
// a warp owns a contiguous run of positions and ballots give a stable,
// position-ordered compaction without atomics ordering anything.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace satk {

constexpr unsigned kFull = 0xffffffffu;

// ----------------------------------------------------------- debug checks --
//
// Built with -DSATK_DEBUG (libsatk_debug.so), device code checks the bound
// of every shared-memory list index, output position, histogram bin and
// scratch index that it relies on an invariant for, before the access: a
// failed check skips the access and ORs a bit into the library's debug word
// (read and cleared by satk_debug_flags), and never traps.  In the normal
// build satk_check is the constant true and the checks compile away.
constexpr unsigned kDbgList = 1u;     // a shared-memory list index
constexpr unsigned kDbgOut = 2u;      // an output position
constexpr unsigned kDbgHist = 4u;     // a histogram bin
constexpr unsigned kDbgScratch = 8u;  // a scratch or plane-word index
#ifdef SATK_DEBUG
extern __device__ unsigned int satk_debug_word;
__device__ __forceinline__ bool satk_check(bool ok, unsigned bit) {
  if (!ok) atomicOr(&satk_debug_word, bit);
  return ok;
}
#else
__device__ __forceinline__ constexpr bool satk_check(bool, unsigned) { return true; }
#endif

// ------------------------------------------------------------------ keys --

__device__ __forceinline__ uint32_t key_f32(uint32_t b) {
  if ((b & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// bf16 pattern in the low 16 bits -> ord16 << 16 (0 for NaN).
// The same keys for values known not to be NaN (they passed a >= compare):
// flip every bit of a negative value, only the sign bit of the others.
__device__ __forceinline__ uint32_t key_f32_num(uint32_t b) {
  return b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
}
__device__ __forceinline__ uint32_t key_bf16_num(uint32_t h) {
  return key_f32_num(h << 16) & 0xffff0000u;
}

__device__ __forceinline__ uint32_t key_bf16(uint32_t h) {
  h &= 0xffffu;
  if ((h & 0x7fffu) > 0x7f80u) return 0u;  // NaN
  uint32_t o = (h & 0x8000u) ? (~h & 0xffffu) : (h | 0x8000u);
  return o << 16;
}

template <typename T>
struct KeyOf;
template <>
struct KeyOf<float> {
  static constexpr int kBits = 32;
  static constexpr int kVec = 4;  // elements per 16-byte load
  __device__ __forceinline__ static uint32_t scalar(const float *p) {
    return key_f32(__float_as_uint(__ldg(p)));
  }
  // one 16-byte vector -> kVec keys
  __device__ __forceinline__ static void vec(const uint4 &v, uint32_t *k) {
    k[0] = key_f32(v.x);
    k[1] = key_f32(v.y);
    k[2] = key_f32(v.z);
    k[3] = key_f32(v.w);
  }
};
template <>
struct KeyOf<uint16_t> {  // raw bfloat16
  static constexpr int kBits = 16;
  static constexpr int kVec = 8;
  __device__ __forceinline__ static uint32_t scalar(const uint16_t *p) {
    return key_bf16(__ldg(reinterpret_cast<const unsigned short *>(p)));
  }
  __device__ __forceinline__ static void vec(const uint4 &v, uint32_t *k) {
    k[0] = key_bf16(v.x);
    k[1] = key_bf16(v.x >> 16);
    k[2] = key_bf16(v.y);
    k[3] = key_bf16(v.y >> 16);
    k[4] = key_bf16(v.z);
    k[5] = key_bf16(v.z >> 16);
    k[6] = key_bf16(v.w);
    k[7] = key_bf16(v.w >> 16);
  }
};

// 16-byte streaming load through the read-only path, not kept in L1.
__device__ __forceinline__ uint4 ldg_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Bulk prefetch of [p, p + bytes) into L2 by the copy engine: no registers,
// no completion to wait for.  p 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ------------------------------------------------------------ block scan --

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = lane_id();
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive block-wide prefix sum of v; *total gets the block sum.  wtot is
// shared scratch of BLOCK/32 ints; one __syncthreads inside.  A caller that
// reuses the same wtot must separate the calls by another barrier.
template <int BLOCK>
__device__ __forceinline__ int block_excl_scan(int v, int *wtot, int *total) {
  constexpr int NW = BLOCK / 32;
  static_assert(NW <= 32, "block too large");
  const int lane = lane_id(), warp = warp_id();
  const int incl = warp_incl_scan(v);
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  const int w = lane < NW ? wtot[lane] : 0;
  const int wi = warp_incl_scan(w);
  *total = __shfl_sync(kFull, wi, NW - 1);
  const int wex = __shfl_sync(kFull, wi - w, warp);
  return wex + incl - v;
}

// Exclusive prefix over the warps of a warp-uniform value wv (one value per
// warp, identical on its lanes): warp w gets the sum over warps < w and
// *total the block sum.  One __syncthreads inside; wtot as above.
template <int BLOCK>
__device__ __forceinline__ int block_warp_prefix(int wv, int *wtot, int *total) {
  constexpr int NW = BLOCK / 32;
  const int lane = lane_id(), warp = warp_id();
  if (lane == 0) wtot[warp] = wv;
  __syncthreads();
  const int w = lane < NW ? wtot[lane] : 0;
  const int wi = warp_incl_scan(w);
  *total = __shfl_sync(kFull, wi, NW - 1);
  return __shfl_sync(kFull, wi - w, warp);
}

// ------------------------------------------------------------- workspace --

template <int BLOCK>
struct SelectSmem {
  uint32_t hist[2048];      // digit histogram, kept zero between passes
  int wtot[4][BLOCK / 32];  // scan scratch: [0] thresholds, [1]-[3] by caller
  int scal[8];              // broadcast scalars
  uint32_t red[BLOCK / 32]; // reductions
  uint32_t fin[64];         // the few keys of a threshold digit (list select)
  int fcnt;                 // their count, kept zero between uses
};

template <int BLOCK>
__device__ __forceinline__ void zero_hist(SelectSmem<BLOCK> &sm) {
  for (int i = threadIdx.x; i < 2048; i += BLOCK) sm.hist[i] = 0u;
  if (threadIdx.x == 0) sm.fcnt = 0;
}

// Histogram add of digit d for lanes with m set.  With AGG, lanes holding
// the same digit combine first (one atomic per distinct digit per warp), so
// a row whose values pile into one bin costs one atomic per warp instead
// of 32 serialised ones.
template <bool AGG>
__device__ __forceinline__ void hist_add(uint32_t *hist, uint32_t d, bool m) {
  if constexpr (!AGG) {
    if (m) atomicAdd(hist + d, 1u);
  } else {
    const unsigned act = __ballot_sync(kFull, m);
    if (m) {
      const unsigned peers = __match_any_sync(act, d);
      if (lane_id() == __ffs(peers) - 1) atomicAdd(hist + d, (unsigned)__popc(peers));
    }
  }
}

struct PassOut {
  int d;      // threshold digit, -1 when fewer than `need` keys matched
  int above;  // keys in digits above d
  int cnt;    // keys in digit d
  int total;  // keys that matched the prefix
};

// Scans the NB-bin histogram from the top digit down and finds the digit d
// with above(d) < need <= above(d) + hist[d].  Zeroes every bin it reads,
// so the histogram is clean for the next pass.  Ends with a barrier.
//
// Bins are read in groups of 32, one per lane in descending order (no bank
// conflicts), warp w taking groups [w*GPW, (w+1)*GPW); group sums come from
// a warp reduction, warp offsets from one block prefix, and only the warp
// holding the crossing scans its group lane by lane.
template <int BLOCK, int NB>
__device__ __forceinline__ PassOut find_threshold(SelectSmem<BLOCK> &sm, int need) {
  static_assert(NB % 32 == 0, "bins come in groups of 32");
  constexpr int NW = BLOCK / 32;
  constexpr int NG = NB / 32;
  constexpr int GPW = (NG + NW - 1) / NW;
  const int lane = lane_id(), warp = warp_id();
  uint32_t c[GPW];
  int gs[GPW];
  int wsum = 0;
#pragma unroll
  for (int q = 0; q < GPW; ++q) {
    const int g = warp * GPW + q;
    c[q] = 0u;
    if (g < NG) {
      const int bin = NB - 1 - (g * 32 + lane);
      c[q] = sm.hist[bin];
      sm.hist[bin] = 0u;
    }
    gs[q] = static_cast<int>(__reduce_add_sync(kFull, c[q]));
    wsum += gs[q];
  }
  int total;
  const int wbase = block_warp_prefix<BLOCK>(wsum, sm.wtot[0], &total);
  if (total >= need && wbase < need && wbase + wsum >= need) {  // warp-uniform
    int cum = wbase;
#pragma unroll
    for (int q = 0; q < GPW; ++q) {
      if (cum < need && cum + gs[q] >= need) {  // warp-uniform
        const int incl = warp_incl_scan(static_cast<int>(c[q]));
        const int before = cum + incl - static_cast<int>(c[q]);
        if (before < need && before + static_cast<int>(c[q]) >= need) {
          sm.scal[0] = NB - 1 - ((warp * GPW + q) * 32 + lane);
          sm.scal[1] = before;
          sm.scal[2] = static_cast<int>(c[q]);
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

// One digit pass over KPT register keys: keys whose top `pbits` bits equal
// `prefix` add digit (key >> shift) & (NB-1).
template <int BLOCK, int KPT, int NB, bool AGG, class GetKey>
__device__ __forceinline__ PassOut reg_pass(GetKey gk, int shift, uint32_t prefix, int pbits,
                                            int need, SelectSmem<BLOCK> &sm) {
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const uint32_t k = gk(i);
    const bool m = (k != 0u) && (pbits == 0 || (k >> (32 - pbits)) == prefix);
    hist_add<AGG>(sm.hist, (k >> shift) & (NB - 1), m);
  }
  __syncthreads();
  return find_threshold<BLOCK, NB>(sm, need);
}

// Outcome of a select over keys with K wanted:
//  take_all : fewer than K non-zero keys; every non-zero key is chosen.
//  !tie     : exactly the keys >= T are chosen (K of them).
//  tie      : the K-th key is T itself and `need` of the keys equal to T
//             must still be chosen (keys > T are all chosen).
struct Sel {
  uint32_t T;
  int need;
  int total;  // non-zero keys (valid when take_all)
  bool tie;
  bool take_all;
  bool exact = false;  // !tie: T is itself a key, the smallest chosen one
};

// Radix select over register keys: 11-bit digits from the top; KEYBITS 32
// takes digits 11/11/10, KEYBITS 16 (bf16 keys: low half zero, except the
// key 1 of a zero score field) 11/5.
template <int BLOCK, int KPT, int KEYBITS, bool AGG, class GetKey>
__device__ Sel radix_select(GetKey gk, int K, SelectSmem<BLOCK> &sm) {
  Sel r;
  r.tie = false;
  r.take_all = false;
  r.total = 0;
  int need = K;
  PassOut p = reg_pass<BLOCK, KPT, 2048, AGG>(gk, 21, 0u, 0, need, sm);
  if (p.d < 0) {
    r.take_all = true;
    r.total = p.total;
    r.T = 1u;
    r.need = 0;
    return r;
  }
  need -= p.above;
  uint32_t prefix = (uint32_t)p.d;
  if (p.cnt == need) {
    r.T = prefix << 21;
    r.need = need;
    return r;
  }
  if constexpr (KEYBITS == 32) {
    p = reg_pass<BLOCK, KPT, 2048, AGG>(gk, 10, prefix, 11, need, sm);
    need -= p.above;
    prefix = (prefix << 11) | (uint32_t)p.d;
    if (p.cnt == need) {
      r.T = prefix << 10;
      r.need = need;
      return r;
    }
    p = reg_pass<BLOCK, KPT, 1024, AGG>(gk, 0, prefix, 22, need, sm);
    need -= p.above;
    prefix = (prefix << 10) | (uint32_t)p.d;
    r.T = prefix;
    r.need = need;
    r.tie = p.cnt != need;
    return r;
  } else {
    p = reg_pass<BLOCK, KPT, 32, AGG>(gk, 16, prefix, 11, need, sm);
    need -= p.above;
    prefix = (prefix << 5) | (uint32_t)p.d;
    // the score-0 digit holds only the key 1 (a B' word with a zero score
    // field); T is that key, so that keys == T are exactly its ties
    r.T = prefix == 0u ? 1u : prefix << 16;
    r.need = need;
    r.tie = p.cnt != need;
    return r;
  }
}

// Block-wide minimum of v (uniform result).  Two barriers.
template <int BLOCK>
__device__ __forceinline__ uint32_t block_min(uint32_t v, SelectSmem<BLOCK> &sm) {
  v = __reduce_min_sync(kFull, v);
  if (lane_id() == 0) sm.red[warp_id()] = v;
  __syncthreads();
  uint32_t m = 0xffffffffu;
#pragma unroll
  for (int w = 0; w < BLOCK / 32; ++w) m = min(m, sm.red[w]);
  __syncthreads();
  return m;
}

// ------------------------------------------------ ordered compaction ------

// Stable compaction of register slots into two ordered groups.  cls(i)
// returns 0 (skip), 1 (group A) or 2 (group B) for slot i; emitA(rank, i,
// tot) and emitB(rank, i, tot) receive each member's rank inside its group
// in flat position order, and the block totals (A in tot.x, B in tot.y).
// Returns the totals.  Each group's count per block must stay below 65536.  Uses
// sm.wtot[1]; two barriers.
template <int BLOCK, int KPT, int VEC, class Cls, class EmitA, class EmitB>
__device__ int2 ordered_emit(Cls cls, EmitA emitA, EmitB emitB, SelectSmem<BLOCK> &sm) {
  static_assert(KPT % VEC == 0, "KPT must be a multiple of VEC");
  const int lane = lane_id();
  const unsigned lt = (1u << lane) - 1u;
  int ca = 0, cb = 0;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const int c = cls(i);
    ca += __popc(__ballot_sync(kFull, c == 1));
    cb += __popc(__ballot_sync(kFull, c == 2));
  }
  // (A << 16) | B with A, B < 65536: unpacked as unsigned
  int total;
  const unsigned base =
      (unsigned)block_warp_prefix<BLOCK>((ca << 16) | cb, sm.wtot[1], &total);
  const int2 tot = make_int2((int)((unsigned)total >> 16), (int)((unsigned)total & 0xffffu));
  int ra = (int)(base >> 16), rb = (int)(base & 0xffffu);
#pragma unroll
  for (int g = 0; g < KPT / VEC; ++g) {
    unsigned ba[VEC], bb[VEC];
    int c[VEC];
    int pa = 0, pb = 0;
#pragma unroll
    for (int s = 0; s < VEC; ++s) {
      c[s] = cls(g * VEC + s);
      ba[s] = __ballot_sync(kFull, c[s] == 1);
      bb[s] = __ballot_sync(kFull, c[s] == 2);
      pa += __popc(ba[s] & lt);
      pb += __popc(bb[s] & lt);
    }
#pragma unroll
    for (int s = 0; s < VEC; ++s) {
      if (c[s] == 1) emitA(ra + pa, g * VEC + s, tot);
      if (c[s] == 2) emitB(rb + pb, g * VEC + s, tot);
      pa += (c[s] == 1);
      pb += (c[s] == 2);
    }
#pragma unroll
    for (int s = 0; s < VEC; ++s) {
      ra += __popc(ba[s]);
      rb += __popc(bb[s]);
    }
  }
  __syncthreads();  // sm.wtot[1] free again
  return tot;
}

// Flat position of register slot i.
template <int KPT, int VEC>
__device__ __forceinline__ int flat_pos(int i) {
  return warp_id() * (32 * KPT) + (i / VEC) * (32 * VEC) + lane_id() * VEC + (i % VEC);
}

}  // namespace satk
