// abi.cu -- status strings, the short-name aliases of the C ABI, and the
// host helpers that keep state (the resident-CTA cache).
#include <mutex>
#include <unordered_map>

#include "satk_device.cuh"
#include "satk_host.hpp"

namespace satk {

int64_t resident_ctas(const void *kernel, int block, size_t smem) {
  static std::mutex mu;
  static std::unordered_map<const void *, int64_t> cache[64];  // per device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  {
    std::lock_guard<std::mutex> g(mu);
    auto it = cache[dev].find(kernel);
    if (it != cache[dev].end()) return it->second;
  }
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, smem) != cudaSuccess)
    return 0;
  const int64_t n = static_cast<int64_t>(sms) * (per_sm < 1 ? 1 : per_sm);
  std::lock_guard<std::mutex> g(mu);
  cache[dev][kernel] = n;
  return n;
}

}  // namespace satk

#ifdef SATK_DEBUG
__device__ unsigned int satk::satk_debug_word;
#endif

extern "C" uint32_t satk_debug_flags(int clear) {
#ifdef SATK_DEBUG
  unsigned int h = 0u;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpyFromSymbol(&h, satk::satk_debug_word, sizeof h) != cudaSuccess)
    return 0xffffffffu;
  if (clear) {
    const unsigned int z = 0u;
    if (cudaMemcpyToSymbol(satk::satk_debug_word, &z, sizeof z) != cudaSuccess) return 0xffffffffu;
  }
  return h;
#else
  (void)clear;
  return 0u;
#endif
}

extern "C" const char *satk_status_string(int rc) {
  switch (rc) {
    case SATK_OK:
      return "ok";
    case SATK_EINVAL:
      return "invalid argument (pointer, size, stride or alignment)";
    case SATK_EUNSUPPORTED:
      return "valid but outside the instantiated range";
    case SATK_ECUDA:
      return "CUDA launch failed";
    default:
      return "unknown status";
  }
}

extern "C" int topk_rows(const void *logits, int dtype, int64_t rows, int64_t cols,
                         int64_t ld_logits, const int32_t *row_ends, int32_t k, int32_t *out,
                         int64_t ld_out, satk_stream_t stream) {
  return satk_topk_rows(logits, dtype, rows, cols, ld_logits, row_ends, k, out, ld_out, stream);
}

extern "C" int topk_rows_sorted(const void *logits, int dtype, int64_t rows, int64_t cols,
                                int64_t ld_logits, const int32_t *row_ends, int32_t k,
                                int32_t *out, int64_t ld_out, satk_stream_t stream) {
  return satk_topk_rows_sorted(logits, dtype, rows, cols, ld_logits, row_ends, k, out, ld_out,
                               stream);
}

extern "C" int dcp_pack(const uint16_t *logits_bf16, int64_t rows, int64_t S, int64_t ld_logits,
                        const int32_t *local_idx, int64_t ld_idx, int32_t n,
                        const int32_t *row_ends, int32_t *packed, satk_stream_t stream) {
  return satk_dcp_pack(logits_bf16, rows, S, ld_logits, local_idx, ld_idx, n, row_ends, packed,
                       stream);
}

extern "C" int dcp_merge_select(const void *cand, int format, int32_t W, int64_t T, int32_t n,
                                int32_t k, int32_t *ids_out, int64_t ld_out, int32_t *sat_word,
                                int32_t *status, satk_stream_t stream) {
  return satk_dcp_merge_select(cand, format, W, T, n, k, ids_out, ld_out, sat_word, status,
                               stream);
}

extern "C" int dcp_rescue_select(const int32_t *packed, int32_t W, int64_t T, int32_t n,
                                 int32_t k, const uint16_t *logits_bf16, int64_t S,
                                 int64_t ld_logits, const int32_t *row_ends,
                                 const int32_t *sat_word, int32_t *recv, int32_t *ids_out,
                                 int64_t ld_out, int32_t *status, satk_stream_t stream) {
  return satk_dcp_rescue_select(packed, W, T, n, k, logits_bf16, S, ld_logits, row_ends,
                                sat_word, recv, ids_out, ld_out, status, stream);
}

extern "C" int dcp_topk_pack(const uint16_t *logits_bf16, int64_t rows, int64_t S,
                             int64_t ld_logits, const int32_t *row_ends, int32_t n,
                             int32_t *packed, satk_stream_t stream) {
  return satk_dcp_topk_pack(logits_bf16, rows, S, ld_logits, row_ends, n, packed, stream);
}
