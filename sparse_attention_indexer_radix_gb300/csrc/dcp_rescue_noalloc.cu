// dcp_rescue_noalloc.cu -- satk_dcp_rescue_select_noalloc: the rescue round
// for callers that cannot allocate device memory.
//
// satk_dcp_rescue_select needs a scratch buffer (`recv`) for the pushed
// lists, and asks its caller for it.  Some callers have no way to provide
// one: code that runs where no allocator may be called (inside a framework
// hook that forbids cudaMalloc, a plugin that only receives pointers to its
// inputs and outputs, a process whose memory pool is already handed out).
// This entry point serves them: its scratch is a fixed array in the
// library's own device memory, so the call allocates nothing.
//
// The array is a file-scope __device__ variable.  Host code cannot use its
// name as a device address (on the host the name only stands for a shadow
// object), so the address is looked up with cudaGetSymbolAddress once per
// device, with that device current, on the first call made on that device,
// and then passed to the kernels like any caller-owned buffer.  The kept
// address is valid as long as the device's primary context lives: a device
// reset after the first call is not supported (the module, and with it the
// array, would be loaded again at another address).
#include <climits>
#include <mutex>

#include "satk_host.hpp"

namespace {

// Every GPU that loads the library keeps this array until the process
// exits: 8 MiB per device.
__device__ __align__(256) int32_t g_rescue_scratch[SATK_RESCUE_NOALLOC_MAX_WORDS];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
int32_t *g_addr[kMaxDevices] = {};

// The scratch's device address on the current device (nullptr on error).
int32_t *scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_rescue_scratch) != cudaSuccess) return nullptr;
    g_addr[dev] = static_cast<int32_t *>(p);
  }
  return g_addr[dev];
}

}  // namespace

extern "C" int satk_dcp_rescue_select_noalloc(const int32_t *packed, int32_t W, int64_t T,
                                              int32_t n, int32_t k,
                                              const uint16_t *logits_bf16, int64_t S,
                                              int64_t ld_logits, const int32_t *row_ends,
                                              const int32_t *sat_word, int32_t *ids_out,
                                              int64_t ld_out, int32_t *status,
                                              satk_stream_t stream) {
  if (T < 0 || n < 1 || k < 1) return SATK_EINVAL;
  if (satk_rescue_recv_words(T, n, k) > static_cast<size_t>(SATK_RESCUE_NOALLOC_MAX_WORDS))
    return SATK_EUNSUPPORTED;  // the fixed scratch is too small for this call
  int32_t *scratch = scratch_on_current_device();
  if (scratch == nullptr) return SATK_ECUDA;
  return satk_dcp_rescue_select(packed, W, T, n, k, logits_bf16, S, ld_logits, row_ends,
                                sat_word, scratch, ids_out, ld_out, status, stream);
}
