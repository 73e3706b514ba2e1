// thd_causal_attn_fwd for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: code running
// inside a host framework that owns every allocation and exposes none of it,
// plugins that must not call cudaMalloc (it synchronises the device and can
// fail or fragment memory mid-step), or hot paths that must never enter the
// allocator at all. For them this file keeps the attention's scratch
// (per-row key bounds, the query tiles, per-group key intervals, the
// schedule, the partial results of cut items) in a
// fixed-size array that lives in device memory for as long as the library is
// loaded, so the call itself allocates nothing.
//
// The array's name is only a host-side stand-in for the device object: host
// code must not pass it to a kernel. A call asks the runtime for the array's
// device address on the current device (cudaGetSymbolAddress, with that
// device current), checks the result, and passes that address down as the
// workspace of the regular entry point, which runs unchanged. The address is
// looked up again on every call whose stream is not capturing, so a device
// reset or another context made current is picked up; a call inside a stream
// capture uses the address the last uncaptured call on that device found,
// which is why the first call on a device must come before any capture.
#include <mutex>

#include "attn_common.cuh"

namespace cpthd {

// 32 MiB: the attention's fixed part (about 20 MiB at d = 128: the partial
// results of the items that the schedule cuts at CTA share boundaries, one
// slot per boundary and tile) and the plan of a slice of up to about 350,000
// query rows (about 33 bytes per row: per-row bounds and document, the
// document runs, and per tile and group its key intervals). Every GPU that
// loads the library holds this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
static void* g_scratch_addr[kMaxDevices] = {};
static std::mutex g_scratch_mutex;

// Device address of g_attn_scratch on the current device. Outside a stream
// capture it is looked up afresh (and remembered for the device); inside one
// the remembered address is used. Returns nullptr (and a status) when the
// runtime cannot provide it, or when a capture comes before any uncaptured
// call on this device.
static void* static_scratch_address(cudaStream_t stream, int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = CPTHD_ERR_CUDA;
    return nullptr;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
    *status = CPTHD_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_attn_scratch) != cudaSuccess || ptr == nullptr) {
      *status = CPTHD_ERR_CUDA;
      return nullptr;
    }
    g_scratch_addr[dev] = ptr;
  }
  *status = (g_scratch_addr[dev] != nullptr) ? CPTHD_OK : CPTHD_ERR_CUDA;
  return g_scratch_addr[dev];
}

}  // namespace cpthd

extern "C" int thd_causal_attn_fwd_static_scratch(const int32_t* q_slice_idx_dev, int64_t t_local,
                                                  const void* q_dev, const void* k_dev, const void* v_dev,
                                                  int64_t T, const int32_t* cu_seqlens_dev,
                                                  const int32_t* cu_seqlens_padded_dev, int num_docs, int Hq,
                                                  int Hkv, int d, float softmax_scale, void* out_dev,
                                                  float* lse_dev, int32_t* err_dev, cpthd_stream_t stream) {
  using namespace cpthd;
  // the same host checks, in the same order, as thd_causal_attn_fwd; then
  // the scratch limit
  int st = check_attn_shape(t_local, T, num_docs, Hq, Hkv);
  if (st != CPTHD_OK) return st;
  if (d != 64 && d != 128) return CPTHD_ERR_UNSUPPORTED;
  if (t_local == 0) return CPTHD_OK;
  size_t need = 0;
  st = thd_causal_attn_workspace_size(t_local, Hq, Hkv, d, &need);
  if (st != CPTHD_OK) return st;
  if (need > kStaticScratchBytes) return CPTHD_ERR_SCRATCH_LIMIT;
  int status = CPTHD_OK;
  void* scratch = static_scratch_address(reinterpret_cast<cudaStream_t>(stream), &status);
  if (scratch == nullptr) return status;
  // The regular entry point's metadata kernel writes every scratch byte the
  // attention kernel later reads, so the previous call's contents need no
  // clearing.
  return thd_causal_attn_fwd(q_slice_idx_dev, t_local, q_dev, k_dev, v_dev, T, cu_seqlens_dev,
                             cu_seqlens_padded_dev, num_docs, Hq, Hkv, d, softmax_scale, out_dev, lse_dev, scratch,
                             kStaticScratchBytes, err_dev, stream);
}
