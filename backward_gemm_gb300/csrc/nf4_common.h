// nf4_common.h -- host-side helpers shared by the library's translation units:
// status codes, argument checks and stream conversion.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "nf4bwd.h"

namespace nf4 {

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Checks shared by every call that reads an NF4 weight of K x N.
inline int check_weight(const float* scales, const uint8_t* data, int K, int N) {
  if (scales == nullptr || data == nullptr) return NF4_ERR_INVALID;
  if (K <= 0 || N < 0 || K % 64 != 0) return NF4_ERR_INVALID;
  if (!aligned(data, 16) || !aligned(scales, 4)) return NF4_ERR_ALIGN;
  return NF4_OK;
}

inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}

}  // namespace nf4
