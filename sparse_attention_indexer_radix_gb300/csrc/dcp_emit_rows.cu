// dcp_emit_rows.cu -- satk_dcp_emit_rows: this rank's physical KV rows of
// the selected tokens (emit_rows of the DCP top-K merge: vLLM API page
// vllm.models.kimi_k3.nvidia.ops.dcp_topk_merge.kernels, DCPTopkSelectKernel
// docstring and dcp_topk_merge_rows).
//
// One CTA per row walks the row's ids in tiles of BLOCK x 8: each thread
// classifies eight consecutive ids (owned by this rank, block inside the
// table), one block-wide scan places the owned ones after those of earlier
// threads and tiles, so rows_out keeps the order of the ids.  Pure integer
// work; HBM-bound on the ids read and the rows written (the block-table
// gathers hit L2).
#include "satk_host.hpp"
#include "satk_device.cuh"

namespace satk {
namespace {

constexpr int kEmitBlock = 256;
constexpr int kEmitPerThread = 8;

struct EmitArgs {
  const int32_t *ids;
  int64_t T, ld_ids;
  int k, W, rank;
  const int32_t *req_id, *block_table;
  int64_t table_rows, ld_table;
  int max_blocks, block_size;
  int64_t stride_rows;
  int32_t *rows_out;
  int64_t ld_rows;
  int32_t *valid_out, *status;
  int w_shift, b_shift;  // log2 of W and block_size when powers of two, else -1
  bool vec_ids;          // every row of ids starts 16-byte aligned
};

__global__ void __launch_bounds__(kEmitBlock) emit_rows_kernel(EmitArgs a) {
  __shared__ int wtot[2][kEmitBlock / 32];
  const int64_t t = blockIdx.x;
  const int32_t *id = a.ids + t * a.ld_ids;
  int32_t *out = a.rows_out + t * a.ld_rows;
  const int req = a.req_id[t];
  const bool req_ok = req >= 0 && static_cast<int64_t>(req) < a.table_rows;
  const int32_t *table = a.block_table + (req_ok ? static_cast<int64_t>(req) * a.ld_table : 0);
  int n = 0;  // rows emitted by earlier tiles (block-uniform)
  int par = 0;
  if (req_ok) {
    for (int base = 0; base < a.k; base += kEmitBlock * kEmitPerThread) {
      const int j0 = base + static_cast<int>(threadIdx.x) * kEmitPerThread;
      int32_t phys[kEmitPerThread];
      int g8[kEmitPerThread];
      unsigned own = 0u;
      if (a.vec_ids && j0 + kEmitPerThread <= a.k) {  // two 16-byte loads
        const int4 u = __ldg(reinterpret_cast<const int4 *>(id + j0));
        const int4 v = __ldg(reinterpret_cast<const int4 *>(id + j0) + 1);
        g8[0] = u.x; g8[1] = u.y; g8[2] = u.z; g8[3] = u.w;
        g8[4] = v.x; g8[5] = v.y; g8[6] = v.z; g8[7] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < kEmitPerThread; ++e) g8[e] = j0 + e < a.k ? id[j0 + e] : -1;
      }
#pragma unroll
      for (int e = 0; e < kEmitPerThread; ++e) {
        const int g = g8[e];
        phys[e] = 0;
        const int owner = a.w_shift >= 0 ? (g & ((1 << a.w_shift) - 1)) : g % a.W;
        if (g >= 0 && owner == a.rank) {
          const int local = a.w_shift >= 0 ? (g >> a.w_shift) : g / a.W;
          const int b = a.b_shift >= 0 ? (local >> a.b_shift) : local / a.block_size;
          const int in_block = a.b_shift >= 0 ? (local & ((1 << a.b_shift) - 1))
                                              : local % a.block_size;
          if (b < a.max_blocks) {
            const int64_t p = static_cast<int64_t>(table[b]) * a.stride_rows + in_block;
            phys[e] = static_cast<int32_t>(static_cast<uint32_t>(static_cast<uint64_t>(p)));
            own |= 1u << e;
          }
        }
      }
      int total;
      int pos = n + block_excl_scan<kEmitBlock>(__popc(own), wtot[par], &total);
      par ^= 1;
#pragma unroll
      for (int e = 0; e < kEmitPerThread; ++e)
        if ((own >> e) & 1u) {
          if (satk_check(pos < a.k, kDbgOut)) out[pos] = phys[e];
          ++pos;
        }
      n += total;
    }
  }
  for (int q = n + static_cast<int>(threadIdx.x); q < a.k; q += kEmitBlock) out[q] = -1;
  if (threadIdx.x == 0) {
    a.valid_out[t] = n;
    if (!req_ok && a.status != nullptr) atomicOr(a.status, SATK_STATUS_BAD_REQUEST);
  }
}

}  // namespace
}  // namespace satk

extern "C" int satk_dcp_emit_rows(const int32_t *ids, int64_t T, int32_t k, int64_t ld_ids,
                                  int32_t W, int32_t dcp_rank, const int32_t *req_id,
                                  const int32_t *block_table, int64_t table_rows,
                                  int64_t ld_block_table, int32_t max_blocks,
                                  int32_t block_size, int64_t stride_rows, int32_t *rows_out,
                                  int64_t ld_rows_out, int32_t *valid_out, int32_t *status,
                                  satk_stream_t stream) {
  using namespace satk;
  if (ids == nullptr || req_id == nullptr || block_table == nullptr || rows_out == nullptr ||
      valid_out == nullptr || T < 0 || k < 1 || ld_ids < k || W < 1 || dcp_rank < 0 ||
      dcp_rank >= W || table_rows < 0 || max_blocks < 0 || ld_block_table < max_blocks ||
      block_size < 1 || ld_rows_out < k || T > INT32_MAX)
    return SATK_EINVAL;
  if (T == 0) return SATK_OK;
  auto log2_or = [](int v) {
    if (v <= 0 || (v & (v - 1)) != 0) return -1;
    int s = 0;
    while ((1 << s) < v) ++s;
    return s;
  };
  const bool vec_ids = (reinterpret_cast<uintptr_t>(ids) & 15u) == 0 && ld_ids % 4 == 0;
  EmitArgs a{ids,        T,           ld_ids,     k,           W,         dcp_rank,
             req_id,     block_table, table_rows, ld_block_table, max_blocks, block_size,
             stride_rows, rows_out,   ld_rows_out, valid_out,  status,
             log2_or(W), log2_or(block_size), vec_ids};
  emit_rows_kernel<<<dim3(static_cast<unsigned>(T)), kEmitBlock, 0, as_stream(stream)>>>(a);
  return launch_status();
}

extern "C" int dcp_emit_rows(const int32_t *ids, int64_t T, int32_t k, int64_t ld_ids,
                             int32_t W, int32_t dcp_rank, const int32_t *req_id,
                             const int32_t *block_table, int64_t table_rows,
                             int64_t ld_block_table, int32_t max_blocks, int32_t block_size,
                             int64_t stride_rows, int32_t *rows_out, int64_t ld_rows_out,
                             int32_t *valid_out, int32_t *status, satk_stream_t stream) {
  return satk_dcp_emit_rows(ids, T, k, ld_ids, W, dcp_rank, req_id, block_table, table_rows,
                            ld_block_table, max_blocks, block_size, stride_rows, rows_out,
                            ld_rows_out, valid_out, status, stream);
}
