// topk_pack_bf16_a16.cu -- the local top-K of bf16 rows written as B' rows
// (satk_dcp_topk_pack), rows with 16-byte aligned starts
// (one translation unit per alignment, see topk_rows_impl.cuh).
#include "topk_rows_impl.cuh"

namespace satk {

int topk_pack_launch_bf16_a16(const uint16_t *x, int64_t rows, int cols, int64_t ld,
                             const int32_t *row_ends, int K, int32_t *packed, cudaStream_t st) {
  return launch_rows<uint16_t, 16, PackedOut>(x, rows, cols, ld, row_ends, K, packed,
                                             K + K / 32, st);
}

}  // namespace satk
