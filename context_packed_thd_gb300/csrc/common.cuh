// Shared helpers of libcpthd: status handling and the device error record.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

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

// Programmatic dependent launch. The forward path's kernels are launched
// with programmatic stream serialization, so that a kernel's launch and
// first instructions overlap the tail of the kernel before it on the
// stream. Every such kernel calls grid_dependency_wait() first, before it
// reads or writes global memory: it returns once the preceding kernel has
// completed and its writes are visible (immediately when the launch had no
// programmatic dependency), so ordering on the stream is as strict as with
// a plain launch. grid_dependents_launch() then lets the next kernel start
// launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KernelArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KernelArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Number of SMs of the current device (looked up once per device).
inline int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

inline int grid_for(long long work, int per_block, int max_blocks) {
  long long b = (work + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > max_blocks) b = max_blocks;
  return static_cast<int>(b);
}

}  // namespace cpthd
