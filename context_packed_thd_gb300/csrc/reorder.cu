// Reorder (row gather) kernels: dst[i, :] = src[idx[i], :], bit exact.
//
// This is the slicing of THD tensors into a context-parallel rank's token
// order (TransformerEngine PR #3221, "How to use": get_batch_on_this_cp_rank
// over input_ids, labels, position_ids; the same gather applies to
// activations). It is a pure copy, bound by HBM bandwidth for wide rows and
// by launch latency for the 8-byte id rows.
//
// Layout: wide rows are cut into units of 32 x UNROLL vectors (2 KB with
// 16-byte vectors), and the warps of the grid take units in turn: a warp's
// lanes move one unit per step with UNROLL independent loads in flight
// before the stores, so the SMs keep enough bytes outstanding to cover HBM
// latency, and every warp gets nearly the same number of units whatever the
// row count (one row per warp left up to half of the warps idle for the
// last row). Vectors are 16 bytes (8 or 4 when the row or a base pointer is
// less aligned, bytes otherwise). Narrow rows (fewer than 32 vectors) use
// one thread per vector instead. Loads and stores use the streaming cache
// hints: every byte is touched once.
//
// The fused form (cp_partition_reorder_multi) takes the source rows from
// the partition formulas instead of an index list: each row's physical slot
// is computed where it is gathered, and the blocks of the first tensor also
// write the rank's index list and check the offset table, so one launch
// replaces the partition-index launch and the gather.
#include "partition_math.cuh"

namespace cpthd {

struct ReorderTensor {
  const void* src;
  void* dst;
  long long row_bytes;
  int vec;  // bytes per vector: 16, 8, 4 or 1
};

struct ReorderBatch {
  ReorderTensor t[8];
};

template <typename V>
__device__ __forceinline__ V load_stream(const V* p) { return __ldcs(p); }
template <>
__device__ __forceinline__ uint8_t load_stream<uint8_t>(const uint8_t* p) { return *p; }
template <typename V>
__device__ __forceinline__ void store_stream(V* p, V v) { __stcs(p, v); }
template <>
__device__ __forceinline__ void store_stream<uint8_t>(uint8_t* p, uint8_t v) { *p = v; }

constexpr int kUnroll = 4;

constexpr int kUnitVecs = 32 * kUnroll;  // vectors per unit of work

template <typename V>
__device__ __forceinline__ void gather_wide(const V* __restrict__ src, long long src_rows, long long vpr,
                                            const IndexGen& ig, long long n_rows,
                                            V* __restrict__ dst, int32_t* err, long long warp,
                                            long long nwarps, int lane) {
  const long long upr = (vpr + kUnitVecs - 1) / kUnitVecs;  // units per row
  const long long units = n_rows * upr;
  for (long long unit = warp; unit < units; unit += nwarps) {
    const long long row = unit / upr;
    const long long c0 = (unit - row * upr) * kUnitVecs;
    const int32_t s = ig.at(row);
    if (s < 0 || s >= src_rows) {
      if (lane == 0 && c0 == 0) record_error(err, CPTHD_ERR_INDEX_RANGE, row);
      continue;
    }
    const V* sp = src + static_cast<long long>(s) * vpr;
    V* dp = dst + row * vpr;
    if (c0 + kUnitVecs <= vpr) {
      V tmp[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) tmp[u] = load_stream(sp + c0 + lane + u * 32);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) store_stream(dp + c0 + lane + u * 32, tmp[u]);
    } else {
      for (long long c = c0 + lane; c < vpr; c += 32) store_stream(dp + c, load_stream(sp + c));
    }
  }
}

template <typename V>
__device__ __forceinline__ void gather_narrow(const V* __restrict__ src, long long src_rows, int vpr,
                                              const IndexGen& ig, long long n_rows,
                                              V* __restrict__ dst, int32_t* err, long long tid,
                                              long long nthreads) {
  const long long total = n_rows * vpr;
  for (long long v = tid; v < total; v += nthreads) {
    const long long row = (vpr == 1) ? v : v / vpr;
    const int col = static_cast<int>(v - row * vpr);
    const int32_t s = ig.at(row);
    if (s < 0 || s >= src_rows) {
      if (col == 0) record_error(err, CPTHD_ERR_INDEX_RANGE, row);
      continue;
    }
    dst[v] = src[static_cast<long long>(s) * vpr + col];
  }
}

template <typename V>
__device__ __forceinline__ void gather_one(const ReorderTensor& t, long long src_rows,
                                           const IndexGen& ig, long long n_rows, int32_t* err) {
  const long long vpr = t.row_bytes / static_cast<long long>(sizeof(V));
  const V* src = static_cast<const V*>(t.src);
  V* dst = static_cast<V*>(t.dst);
  if (vpr >= 32) {
    const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    gather_wide<V>(src, src_rows, vpr, ig, n_rows, dst, err, warp, nwarps, threadIdx.x & 31);
  } else {
    const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const long long nthreads = (long long)gridDim.x * blockDim.x;
    gather_narrow<V>(src, src_rows, static_cast<int>(vpr), ig, n_rows, dst, err, tid, nthreads);
  }
}

// blockIdx.y selects the tensor of the batch. With a computed index, the
// blocks of blockIdx.y == 0 also write the index list (idx_out) and check
// the offset table.
__global__ void __launch_bounds__(256) reorder_kernel(ReorderBatch batch, long long src_rows, IndexGen ig,
                                                      long long n_rows, int32_t* __restrict__ idx_out,
                                                      int32_t* err) {
  // every block waits, even one with nothing to copy, so that this grid never
  // completes before the kernel it depends on
  grid_dependency_wait();
  grid_dependents_launch();
  if (ig.idx == nullptr && blockIdx.y == 0) {
    const long long first = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    const long long stride = (long long)gridDim.x * blockDim.x;
    check_offsets_range(ig.cup, ig.num_docs, ig.T, ig.cp, ig.strategy == CPTHD_DUAL_CHUNK_SWAP, err, first,
                        stride);
    for (long long row = first; row < n_rows; row += stride) idx_out[row] = ig.at(row);
  }
  const ReorderTensor& t = batch.t[blockIdx.y];
  if (t.row_bytes == 0) return;
  switch (t.vec) {
    case 16: gather_one<uint4>(t, src_rows, ig, n_rows, err); break;
    case 8: gather_one<uint2>(t, src_rows, ig, n_rows, err); break;
    case 4: gather_one<uint32_t>(t, src_rows, ig, n_rows, err); break;
    default: gather_one<uint8_t>(t, src_rows, ig, n_rows, err); break;
  }
}

static int vector_bytes(const void* src, const void* dst, long long row_bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                      static_cast<uintptr_t>(row_bytes);
  if ((a & 15) == 0) return 16;
  if ((a & 7) == 0) return 8;
  if ((a & 3) == 0) return 4;
  return 1;
}

// computed = false: ig.idx is the caller's index list (required when there
// is anything to copy). computed = true: the partition index of ig's rank,
// written to idx_out.
static int launch_reorder(int n, const void* const* src, void* const* dst, const int64_t* row_bytes,
                          int64_t src_rows, const IndexGen& ig, bool computed, int64_t n_rows, int32_t* idx_out,
                          int32_t* err, cudaStream_t s) {
  if (n < 1 || n > 8 || src_rows < 0 || n_rows < 0) return CPTHD_ERR_INVALID_ARG;
  if (src_rows > INT32_MAX) return CPTHD_ERR_INVALID_ARG;
  ReorderBatch b{};
  long long max_bytes = 0;
  for (int i = 0; i < n; ++i) {
    if (row_bytes[i] < 0) return CPTHD_ERR_INVALID_ARG;
    if (row_bytes[i] > 0 && n_rows > 0 && (src[i] == nullptr || dst[i] == nullptr)) return CPTHD_ERR_INVALID_ARG;
    b.t[i].src = src[i];
    b.t[i].dst = dst[i];
    b.t[i].row_bytes = row_bytes[i];
    b.t[i].vec = vector_bytes(src[i], dst[i], row_bytes[i]);
    max_bytes = row_bytes[i] > max_bytes ? row_bytes[i] : max_bytes;
  }
  if (n_rows == 0 || (max_bytes == 0 && !computed)) return CPTHD_OK;
  if (!computed && ig.idx == nullptr) return CPTHD_ERR_INVALID_ARG;
  if (computed && (ig.idx != nullptr || idx_out == nullptr)) return CPTHD_ERR_INVALID_ARG;
  // Wide rows: a warp per unit (32 x kUnroll vectors) for large gathers, a
  // warp per row for small ones (the warps then share the rows' units); a
  // thread per vector for narrow rows; capped at 8 resident 256-thread
  // blocks on each SM of the device. Sized by units, the small Q gather of a
  // rank slice held more SMs for longer and the attention launch after it
  // started later; sized by rows, the large activation gathers left SMs
  // idle (82% vs 79% of the copy bandwidth on [131072, 8192] bf16).
  long long total_bytes = 0;
  for (int i = 0; i < n; ++i) total_bytes += n_rows * b.t[i].row_bytes;
  const bool by_units = total_bytes >= (32LL << 20);
  long long work = computed ? n_rows : 0;  // the index list is written by one thread per row
  for (int i = 0; i < n; ++i) {
    const long long vpr = b.t[i].row_bytes / b.t[i].vec;
    const long long upr = by_units ? (vpr + kUnitVecs - 1) / kUnitVecs : 1;
    const long long w = (vpr >= 32) ? n_rows * upr * 32 : n_rows * vpr;
    work = w > work ? w : work;
  }
  const int sms = sm_count();
  if (sms < 1) return CPTHD_ERR_CUDA;
  const int grid = grid_for(work, 256, sms * 8);
  dim3 g(grid, n);
  CPTHD_TRY_CUDA(launch_pdl(reorder_kernel, g, dim3(256), 0, s, b, static_cast<long long>(src_rows), ig,
                            static_cast<long long>(n_rows), idx_out, err));
  return CPTHD_OK;
}

}  // namespace cpthd

extern "C" int cp_reorder(const void* src_dev, int64_t src_rows, int64_t row_bytes, const int32_t* idx_dev,
                          int64_t n_rows, void* dst_dev, int32_t* err_dev, cpthd_stream_t stream) {
  const void* srcs[1] = {src_dev};
  void* dsts[1] = {dst_dev};
  const int64_t rb[1] = {row_bytes};
  return cpthd::launch_reorder(1, srcs, dsts, rb, src_rows, cpthd::index_list(idx_dev), false, n_rows, nullptr,
                               err_dev, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int cp_reorder_multi(int n_tensors, const void* const* src_dev_host, void* const* dst_dev_host,
                                const int64_t* row_bytes_host, int64_t src_rows, const int32_t* idx_dev,
                                int64_t n_rows, int32_t* err_dev, cpthd_stream_t stream) {
  if (src_dev_host == nullptr || dst_dev_host == nullptr || row_bytes_host == nullptr)
    return CPTHD_ERR_INVALID_ARG;
  return cpthd::launch_reorder(n_tensors, src_dev_host, dst_dev_host, row_bytes_host, src_rows,
                               cpthd::index_list(idx_dev), false, n_rows, nullptr, err_dev,
                               reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int cp_partition_reorder_multi(int strategy, const int32_t* cu_seqlens_padded_dev, int num_docs,
                                          int64_t T, int cp_size, int rank, int n_tensors,
                                          const void* const* src_dev_host, void* const* dst_dev_host,
                                          const int64_t* row_bytes_host, int32_t* idx_out_dev, int32_t* err_dev,
                                          cpthd_stream_t stream) {
  int64_t t_local = 0;
  const int st = cp_local_tokens(strategy, T, cp_size, &t_local);
  if (st != CPTHD_OK) return st;
  if (rank < 0 || rank >= cp_size || num_docs < 0 || T > INT32_MAX) return CPTHD_ERR_INVALID_ARG;
  if (src_dev_host == nullptr || dst_dev_host == nullptr || row_bytes_host == nullptr) return CPTHD_ERR_INVALID_ARG;
  if (t_local > 0 && (cu_seqlens_padded_dev == nullptr || num_docs == 0 || idx_out_dev == nullptr))
    return CPTHD_ERR_INVALID_ARG;
  const cpthd::IndexGen g =
      cpthd::index_formula(strategy, cu_seqlens_padded_dev, num_docs, T, cp_size, rank, t_local);
  return cpthd::launch_reorder(n_tensors, src_dev_host, dst_dev_host, row_bytes_host, T, g, true, t_local,
                               idx_out_dev, err_dev, reinterpret_cast<cudaStream_t>(stream));
}
