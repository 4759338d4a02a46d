// topk_rows_bf16_a16.cu -- the row kernels for bf16 rows with 16-byte aligned starts
// (one translation unit per type and alignment, see topk_rows_impl.cuh).
#include "topk_rows_impl.cuh"

namespace satk {

int topk_rows_launch_bf16_a16(const uint16_t *x, int64_t rows, int cols, int64_t ld,
                              const int32_t *row_ends, int K, int32_t *out, int64_t ld_out,
                              bool sorted, cudaStream_t st) {
  return sorted ? launch_rows_sorted<uint16_t, 16>(x, rows, cols, ld, row_ends, K, out, ld_out, st)
                : launch_rows<uint16_t, 16>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
}

}  // namespace satk
