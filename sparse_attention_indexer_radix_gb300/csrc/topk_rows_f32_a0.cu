// topk_rows_f32_a0.cu -- the row kernels for fp32 rows of any alignment (element loads)
// (one translation unit per type and alignment, see topk_rows_impl.cuh).
#include "topk_rows_impl.cuh"

namespace satk {

int topk_rows_launch_f32_a0(const float *x, int64_t rows, int cols, int64_t ld,
                            const int32_t *row_ends, int K, int32_t *out, int64_t ld_out,
                            bool sorted, cudaStream_t st) {
  return sorted ? launch_rows_sorted<float, 0>(x, rows, cols, ld, row_ends, K, out, ld_out, st)
                : launch_rows<float, 0>(x, rows, cols, ld, row_ends, K, out, ld_out, st);
}

}  // namespace satk
