// Shared helpers of libcpthd: status handling and the device error record.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "cpthd.h"

#define CPTHD_TRY_CUDA(expr)                      \
  do {                                            \
    cudaError_t cpthd_e_ = (expr);                \
    if (cpthd_e_ != cudaSuccess) return CPTHD_ERR_CUDA; \
  } while (0)

namespace cpthd {

// Record the first data-dependent error of a launch in the caller's
// err[0..1] pair: err[0] = status code, err[1] = detail. Later errors are
// dropped. Never traps.
__device__ __forceinline__ void record_error(int32_t* err, int code, long long detail) {
  if (err != nullptr) {
    if (atomicCAS(reinterpret_cast<int*>(err), 0, code) == 0) {
      atomicExch(reinterpret_cast<int*>(err + 1), static_cast<int>(detail));
    }
  }
}

// Largest j in [0, n) with a[j] <= x, for a non-decreasing a[0..n]
// (a[0] <= x assumed; clamps to [0, n-1] on malformed input).
__device__ __forceinline__ int upper_bound_doc(const int32_t* __restrict__ a, int n, long long x) {
  int lo = 0, hi = n;  // invariant: answer in [lo, hi)
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (static_cast<long long>(__ldg(a + mid)) <= x) lo = mid; else hi = mid;
  }
  return lo;
}

inline int grid_for(long long work, int per_block, int max_blocks) {
  long long b = (work + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > max_blocks) b = max_blocks;
  return static_cast<int>(b);
}

}  // namespace cpthd
