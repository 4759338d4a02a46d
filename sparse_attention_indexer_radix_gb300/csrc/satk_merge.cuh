// satk_merge.cuh -- the merge select shared by the round-1 select and the
// rescue re-select (vLLM API page
// vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels, sections
// DCPTopkSelectKernel, DCPTopkRescueKernel, _make_radix_select).
//
// The candidates of one row sit in registers, one per slot, keyed by their
// score (0 = empty); the global id of slot i is gid(i).  The chosen set is
// the K best under (score desc, global id asc): a radix select on the score
// key, and, when the K-th score is tied, a second radix select on
// ~global-id among the tied candidates.  A (score, id) pair repeated across
// the cut (only an out-of-contract producer sends one) is left out, as the
// page's select does, so fewer than K ids come out and the status gets
// SATK_STATUS_DUPLICATE_KEYS.  The ids are written in ascending flat
// position order.
#pragma once

#include "satk_device.cuh"

namespace satk {

struct MergeOut {
  int nsel;       // ids written before the -1 fill
  uint32_t kmin;  // smallest chosen score key (0xffffffff when none)
  bool dup;       // a repeated candidate sat on the cut
};

template <int BLOCK, int KPT, int KEYBITS, class GidOf, class Out>
__device__ MergeOut merge_core(const uint32_t (&keys)[KPT], GidOf gid, Out out, int K,
                               bool want_min, SelectSmem<BLOCK> &sm) {
  auto gk = [&](int i) { return keys[i]; };
  const Sel s = radix_select<BLOCK, KPT, KEYBITS, true>(gk, K, sm);
  uint32_t t2 = 0u;
  bool use2 = false, tie2 = false;
  if (!s.take_all && s.tie) {
    auto gk2 = [&](int i) { return keys[i] == s.T ? 0xffffffffu - gid(i) : 0u; };
    const Sel s2 = radix_select<BLOCK, KPT, 32, true>(gk2, s.need, sm);
    use2 = true;
    t2 = s2.T;
    tie2 = s2.tie;
  }
  auto chosen = [&](int i) -> bool {
    const uint32_t k = keys[i];
    if (k == 0u) return false;
    if (s.take_all) return true;
    if (!use2) return k >= s.T;
    if (k != s.T) return k > s.T;
    const uint32_t k2 = 0xffffffffu - gid(i);
    return tie2 ? k2 > t2 : k2 >= t2;
  };
  const int2 tot = ordered_emit<BLOCK, KPT, 1>(
      [&](int i) { return chosen(i) ? 1 : 0; },
      [&](int rank, int i, int2) { out(rank, static_cast<int32_t>(gid(i))); },
      [](int, int, int2) {}, sm);
  for (int q = max(0, tot.x) + (int)threadIdx.x; q < K; q += BLOCK) out(q, -1);
  MergeOut r;
  r.nsel = tot.x;
  r.dup = tie2;
  r.kmin = 0xffffffffu;
  if (want_min) {
    uint32_t m = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < KPT; ++i)
      if (chosen(i)) m = min(m, keys[i]);
    r.kmin = block_min<BLOCK>(m, sm);
  }
  return r;
}

// B' word of slot j (plane word holds bit local[16] at j % 32) -> score key
// and local id.  Only the word 0 is empty (vLLM API page
// vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels, _decode_key): a
// non-zero word keys as ord16 << 16, or as 1 when its score field is 0 --
// below every other score, above the empty key.  Every 16-bit select treats
// 1 as the one key of score 0 (radix_select<..., 16> returns T = 1 for it).
__device__ __forceinline__ uint32_t bprime_key(uint32_t w) {
  const uint32_t k = w & 0xffff0000u;
  return k != 0u ? k : (w != 0u ? 1u : 0u);
}
// The same word's key in the shared-memory list engine: ord16 + 1 (0 for
// the empty word only), so that the list select's range-relative digits
// cover the score's 16 bits and nothing else (ord16 << 16 would leave 16
// bits that are always zero, and every key of their digit passes would
// land in one histogram bin).  Order is that of bprime_key.
__device__ __forceinline__ uint32_t bprime_list_key(uint32_t w) {
  return w == 0u ? 0u : (w >> 16) + 1u;
}
__device__ __forceinline__ uint32_t bprime_local(uint32_t w, uint32_t plane, int j) {
  return (0xffffu - (w & 0xffffu)) | (((plane >> (j & 31)) & 1u) << 16);
}

}  // namespace satk
