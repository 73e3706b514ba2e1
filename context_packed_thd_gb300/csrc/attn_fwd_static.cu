// thd_causal_attn_fwd for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: code running
// inside a host framework that owns every allocation and exposes none of it,
// plugins that must not call cudaMalloc (it synchronises the device and can
// fail or fragment memory mid-step), or hot paths that must never enter the
// allocator at all. For them this file keeps the attention's scratch
// (per-row key bounds, per-group key intervals, the group schedule) in a
// fixed-size array that lives in device memory for as long as the library is
// loaded, so the call itself allocates nothing.
//
// The array's name is only a host-side stand-in for the device object: host
// code must not pass it to a kernel. The first call on each device asks the
// runtime for the array's device address (cudaGetSymbolAddress, with that
// device current), checks the result and caches it; every call then passes
// that address down as the workspace of the regular entry point, which runs
// unchanged.
#include <mutex>

#include "common.cuh"

namespace cpthd {

// 4 MiB: the scratch of a slice of up to about 250,000 query rows (16 bytes
// per row plus 28 bytes per row group). Every GPU that loads the library
// holds this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;

static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
static void* g_scratch_addr[kMaxDevices] = {};
static std::mutex g_scratch_mutex;

// Device address of g_attn_scratch on the current device (looked up once per
// device). Returns nullptr when the runtime cannot provide it.
static void* static_scratch_address(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = CPTHD_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_attn_scratch) != cudaSuccess || ptr == nullptr) {
      *status = CPTHD_ERR_CUDA;
      return nullptr;
    }
    g_scratch_addr[dev] = ptr;
  }
  *status = CPTHD_OK;
  return g_scratch_addr[dev];
}

}  // namespace cpthd

extern "C" int thd_causal_attn_fwd_static_scratch(const int32_t* q_slice_idx_dev, int64_t t_local,
                                                  const void* q_dev, const void* k_dev, const void* v_dev,
                                                  int64_t T, const int32_t* cu_seqlens_dev,
                                                  const int32_t* cu_seqlens_padded_dev, int num_docs, int Hq,
                                                  int Hkv, int d, float softmax_scale, void* out_dev,
                                                  float* lse_dev, int32_t* err_dev, cpthd_stream_t stream) {
  size_t need = 0;
  const int st = thd_causal_attn_workspace_size(t_local, Hq, Hkv, d, &need);
  if (st != CPTHD_OK) return st;
  if (need > cpthd::kStaticScratchBytes) return CPTHD_ERR_SCRATCH_LIMIT;
  if (t_local == 0) return CPTHD_OK;
  int status = CPTHD_OK;
  void* scratch = cpthd::static_scratch_address(&status);
  if (scratch == nullptr) return status;
  // The regular entry point's metadata kernel writes every scratch byte the
  // attention kernel later reads, so the previous call's contents need no
  // clearing.
  return thd_causal_attn_fwd(q_slice_idx_dev, t_local, q_dev, k_dev, v_dev, T, cu_seqlens_dev,
                             cu_seqlens_padded_dev, num_docs, Hq, Hkv, d, softmax_scale, out_dev, lse_dev, scratch,
                             cpthd::kStaticScratchBytes, err_dev, stream);
}
