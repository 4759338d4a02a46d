// topk_rows.cu -- satk_topk_rows: exact per-row top-K over fp32 or bf16
// logits with causal row ends, -1 padding and a strided output
// ([Perf][DSA] Use DeepSelect for eligible sparse-indexer prefill chunks,
// vLLM PR #57206: Purpose, Test Plan).
//
// One CTA per row.  Rows that fit the CTA's registers (BLOCK * KPT columns)
// take the register path; longer rows the streaming path (see
// satk_rows.cuh).  Both read each valid column from HBM once.
#include <climits>

#include "satk_host.hpp"
#include "satk_rows.cuh"

namespace satk {
namespace {

__device__ __forceinline__ int row_end_of(const int32_t *row_ends, int64_t row, int cols) {
  if (row_ends == nullptr) return cols;
  const int e = row_ends[row];
  return e < 0 ? 0 : (e > cols ? cols : e);
}

template <typename T, int BLOCK, int KPT, bool VECLOAD, bool AGG>
__global__ void __launch_bounds__(BLOCK) topk_rows_reg_kernel(const T *__restrict__ x, int64_t ld,
                                                              int cols,
                                                              const int32_t *__restrict__ row_ends,
                                                              int K, int32_t *__restrict__ out,
                                                              int64_t ld_out) {
  __shared__ SelectSmem<BLOCK> sm;
  const int64_t row = blockIdx.x;
  const int end = row_end_of(row_ends, row, cols);
  zero_hist(sm);
  __syncthreads();
  int32_t *o = out + row * ld_out;
  topk_reg_row<T, BLOCK, KPT, VECLOAD, AGG>(
      x + row * ld, end, K, [&](int pos, uint32_t, int col) {
        if ((unsigned)pos < (unsigned)K) o[pos] = col;
      },
      [&](int pos) { o[pos] = -1; }, sm);
}

template <typename T, int BLOCK, int LKPT, bool VECLOAD, bool AGG>
__global__ void __launch_bounds__(BLOCK) topk_rows_stream_kernel(
    const T *__restrict__ x, int64_t ld, int cols, const int32_t *__restrict__ row_ends, int K,
    int32_t *__restrict__ out, int64_t ld_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<StreamSmem<BLOCK, BLOCK * LKPT> *>(smem_raw);
  const int64_t row = blockIdx.x;
  const int end = row_end_of(row_ends, row, cols);
  zero_hist(sm.sel);
  __syncthreads();
  int32_t *o = out + row * ld_out;
  topk_stream_row<T, BLOCK, LKPT, VECLOAD, AGG>(
      x + row * ld, end, K, [&](int pos, uint32_t, int col) {
        if ((unsigned)pos < (unsigned)K) o[pos] = col;
      },
      [&](int pos) { o[pos] = -1; }, sm);
}

constexpr int kBlock = 512;
constexpr int kStreamLkpt = 8;  // list of 4096 candidates

template <typename T, bool VECLOAD>
int launch_rows(const T *x, int64_t rows, int cols, int64_t ld, const int32_t *row_ends, int K,
                int32_t *out, int64_t ld_out, cudaStream_t st) {
  constexpr int VEC = VECLOAD ? KeyOf<T>::kVec : 1;
  const dim3 grid(static_cast<unsigned>(rows));
  // register path: BLOCK * KPT columns, KPT a multiple of the vector width
  constexpr int K1 = VEC > 4 ? VEC : 4;
  if (cols <= kBlock * K1) {
    topk_rows_reg_kernel<T, kBlock, K1, VECLOAD, true>
        <<<grid, kBlock, 0, st>>>(x, ld, cols, row_ends, K, out, ld_out);
  } else if (cols <= kBlock * 2 * K1) {
    topk_rows_reg_kernel<T, kBlock, 2 * K1, VECLOAD, true>
        <<<grid, kBlock, 0, st>>>(x, ld, cols, row_ends, K, out, ld_out);
  } else if (cols <= kBlock * 16 && 16 % VEC == 0 && 16 > 2 * K1) {
    topk_rows_reg_kernel<T, kBlock, 16, VECLOAD, true>
        <<<grid, kBlock, 0, st>>>(x, ld, cols, row_ends, K, out, ld_out);
  } else {
    auto kern = topk_rows_stream_kernel<T, kBlock, kStreamLkpt, VECLOAD, true>;
    const size_t smem = sizeof(StreamSmem<kBlock, kBlock * kStreamLkpt>);
    if (!allow_smem(kern, smem)) return SATK_ECUDA;
    kern<<<grid, kBlock, smem, st>>>(x, ld, cols, row_ends, K, out, ld_out);
  }
  return launch_status();
}

}  // namespace
}  // namespace satk

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
    if (aligned16(x) && (ld_logits * 4) % 16 == 0)
      return launch_rows<float, true>(x, rows, c, ld_logits, row_ends, k, out, ld_out, st);
    return launch_rows<float, false>(x, rows, c, ld_logits, row_ends, k, out, ld_out, st);
  }
  const uint16_t *x = static_cast<const uint16_t *>(logits);
  if (aligned16(x) && (ld_logits * 2) % 16 == 0)
    return launch_rows<uint16_t, true>(x, rows, c, ld_logits, row_ends, k, out, ld_out, st);
  return launch_rows<uint16_t, false>(x, rows, c, ld_logits, row_ends, k, out, ld_out, st);
}
