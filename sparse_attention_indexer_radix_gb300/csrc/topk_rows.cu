// topk_rows.cu -- satk_topk_rows, satk_topk_rows_sorted and
// satk_dcp_topk_pack: exact per-row
// top-K over fp32 or bf16 logits with causal row ends, -1 padding and a
// strided output ([Perf][DSA] Use DeepSelect for eligible sparse-indexer
// prefill chunks, vLLM PR #57206: Purpose, Test Plan).
//
// The entry points check their arguments and pick the translation unit of
// the row's type and alignment; the kernels and the choice of path are in
// topk_rows_impl.cuh.
#include <climits>

#include "satk_host.hpp"
#include "topk_rows_impl.cuh"

namespace satk {
namespace {

// Widest load every row start allows: 32 or 16 bytes, else element loads.
inline int row_alignment(const void *x, int64_t ld_bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(x);
  if ((a & 31u) == 0 && ld_bytes % 32 == 0) return 32;
  if ((a & 15u) == 0 && ld_bytes % 16 == 0) return 16;
  return 0;
}

}  // namespace
}  // namespace satk


extern "C" int satk_topk_rows_sorted(const void *logits, int dtype, int64_t rows, int64_t cols,
                                     int64_t ld_logits, const int32_t *row_ends, int32_t k,
                                     int32_t *out, int64_t ld_out, satk_stream_t stream) {
  using namespace satk;
  if (logits == nullptr || out == nullptr || rows < 0 || cols < 0 || ld_logits < cols ||
      k < 1 || k > SATK_TOPK_MAX_K || ld_out < k || cols > INT_MAX || rows > INT_MAX ||
      (dtype != SATK_F32 && dtype != SATK_BF16))
    return SATK_EINVAL;
  if (rows == 0) return SATK_OK;
  const cudaStream_t st = as_stream(stream);
  const int c = static_cast<int>(cols);
  if (dtype == SATK_F32) {
    const float *x = static_cast<const float *>(logits);
    switch (row_alignment(x, ld_logits * 4)) {
      case 32:
        return topk_rows_launch_f32_a32(x, rows, c, ld_logits, row_ends, k, out, ld_out, true, st);
      case 16:
        return topk_rows_launch_f32_a16(x, rows, c, ld_logits, row_ends, k, out, ld_out, true, st);
      default:
        return topk_rows_launch_f32_a0(x, rows, c, ld_logits, row_ends, k, out, ld_out, true, st);
    }
  }
  const uint16_t *x = static_cast<const uint16_t *>(logits);
  if (row_alignment(x, ld_logits * 2) != 0)
    return topk_rows_launch_bf16_a16(x, rows, c, ld_logits, row_ends, k, out, ld_out, true, st);
  return topk_rows_launch_bf16_a0(x, rows, c, ld_logits, row_ends, k, out, ld_out, true, st);
}

extern "C" int satk_topk_rows(const void *logits, int dtype, int64_t rows, int64_t cols,
                              int64_t ld_logits, const int32_t *row_ends, int32_t k,
                              int32_t *out, int64_t ld_out, satk_stream_t stream) {
  using namespace satk;
  if (logits == nullptr || out == nullptr || rows < 0 || cols < 0 || ld_logits < cols ||
      k < 1 || k > SATK_TOPK_MAX_K || ld_out < k || cols > INT_MAX || rows > INT_MAX ||
      (dtype != SATK_F32 && dtype != SATK_BF16))
    return SATK_EINVAL;
  if (rows == 0) return SATK_OK;
  const cudaStream_t st = as_stream(stream);
  const int c = static_cast<int>(cols);
  if (dtype == SATK_F32) {
    const float *x = static_cast<const float *>(logits);
    switch (row_alignment(x, ld_logits * 4)) {
      case 32:
        return topk_rows_launch_f32_a32(x, rows, c, ld_logits, row_ends, k, out, ld_out, false, st);
      case 16:
        return topk_rows_launch_f32_a16(x, rows, c, ld_logits, row_ends, k, out, ld_out, false, st);
      default:
        return topk_rows_launch_f32_a0(x, rows, c, ld_logits, row_ends, k, out, ld_out, false, st);
    }
  }
  const uint16_t *x = static_cast<const uint16_t *>(logits);
  if (row_alignment(x, ld_logits * 2) != 0)
    return topk_rows_launch_bf16_a16(x, rows, c, ld_logits, row_ends, k, out, ld_out, false, st);
  return topk_rows_launch_bf16_a0(x, rows, c, ld_logits, row_ends, k, out, ld_out, false, st);
}

extern "C" int satk_dcp_topk_pack(const uint16_t *logits_bf16, int64_t rows, int64_t S,
                                  int64_t ld_logits, const int32_t *row_ends, int32_t n,
                                  int32_t *packed, satk_stream_t stream) {
  using namespace satk;
  if (logits_bf16 == nullptr || packed == nullptr || rows < 0 || S < 0 || ld_logits < S ||
      n < 32 || n % 32 != 0 || n > SATK_TOPK_MAX_K || S > INT_MAX || rows > INT_MAX)
    return SATK_EINVAL;
  if (rows == 0) return SATK_OK;
  const cudaStream_t st = as_stream(stream);
  const int c = static_cast<int>(S);
  if (row_alignment(logits_bf16, ld_logits * 2) != 0)
    return topk_pack_launch_bf16_a16(logits_bf16, rows, c, ld_logits, row_ends, n, packed, st);
  return topk_pack_launch_bf16_a0(logits_bf16, rows, c, ld_logits, row_ends, n, packed, st);
}
