// Helpers shared by the C-ABI files (api.cu, int4_api.cu): status reporting, the device guard,
// argument checks and device allocation.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <string>

#include "svdq_internal.h"

namespace svdq {

// The calling thread's message for its last failed call (svdq_last_error), defined in api.cu.
std::string& last_error_slot();

inline svdq_status_t fail(svdq_status_t s, const std::string& msg) {
  last_error_slot() = msg;
  return s;
}
inline svdq_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(SVDQ_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// Makes `dev` current for the scope of a call and restores the caller's device afterwards.
struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) changed = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

// SVDQ_ERR_ARCH unless the device is compute capability 10.3 (api.cu).
svdq_status_t check_arch(int device);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte.
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

inline void* dalloc(size_t bytes, cudaError_t* e) {
  void* p = nullptr;
  *e = cudaMalloc(&p, bytes ? bytes : 256);
  return *e == cudaSuccess ? p : nullptr;
}

}  // namespace svdq
