// satk_host.hpp -- host-side helpers shared by the entry points of
// libsatk.so: argument checks, launch-status mapping, stream cast.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "satk.h"

namespace satk {

inline cudaStream_t as_stream(satk_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Maps the result of the launches just issued to an SATK return code.
inline int launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SATK_OK : SATK_ECUDA;
}

// Raises the dynamic shared-memory limit of a kernel once per process.
template <class K>
inline bool allow_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return true;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes)) == cudaSuccess;
}

// CTAs of `kernel` (block threads, smem dynamic bytes) the current device
// holds at once: SMs x resident CTAs per SM, computed once per kernel and
// device.  0 on error.
int64_t resident_ctas(const void *kernel, int block, size_t smem);

}  // namespace satk
