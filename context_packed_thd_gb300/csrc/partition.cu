// Partition index kernels: which physical THD tokens a context-parallel rank
// owns.
//
// TransformerEngine PR #3221 ("Why", "What changed"): the default
// DualChunkSwap partition cuts every document into 2*cp_size chunks and
// rank r owns chunks r and 2*cp_size-1-r (the head-tail split, torchtitan
// PR #2144 "Summary"); NO_LOAD_BALANCE cuts the complete physical buffer into
// cp_size contiguous chunks, rank-major. Within a DualChunkSwap rank the
// documents keep pack order and chunk r precedes chunk 2*cp_size-1-r, so the
// rank-local offsets are cu_seqlens_padded / cp_size: output position t is
// found by a binary search over those local offsets. The PR's interim
// "packed super-sequence" partition (PACKED_MIRRORED) is DualChunkSwap of the
// whole buffer taken as one sequence. The restore index inverts the
// rank-major concatenation of all ranks' lists, which is what an all-gather
// of the ranks' K/V slices produces.
#include "partition_math.cuh"

namespace cpthd {

__device__ __forceinline__ void check_offsets(const int32_t* __restrict__ cup, int num_docs, long long T, int cp,
                                              int dcs, int32_t* err) {
  check_offsets_range(cup, num_docs, T, cp, dcs, err, blockIdx.x * (long long)blockDim.x + threadIdx.x,
                      (long long)gridDim.x * blockDim.x);
}

__global__ void dual_chunk_swap_index_kernel(const int32_t* __restrict__ cup, int num_docs, long long T, int cp,
                                             int rank, long long t_local, long long total,
                                             int32_t* __restrict__ idx, int32_t* err) {
  grid_dependency_wait();
  grid_dependents_launch();
  check_offsets(cup, num_docs, T, cp, 1, err);
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    int r = rank;
    long long t = o;
    if (rank < 0) { r = static_cast<int>(o / t_local); t = o - (long long)r * t_local; }
    const long long p = dcs_slot(cup, num_docs, cp, r, t);
    idx[o] = static_cast<int32_t>(p);
  }
}

__global__ void no_load_balance_index_kernel(const int32_t* __restrict__ cup, int num_docs, long long T, int cp,
                                             int rank, long long t_local, long long total,
                                             int32_t* __restrict__ idx, int32_t* err) {
  grid_dependency_wait();
  grid_dependents_launch();
  check_offsets(cup, num_docs, T, cp, 0, err);
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    const long long p = (rank < 0) ? o : nlb_slot(rank, t_local, o);
    idx[o] = static_cast<int32_t>(p);
  }
}

__global__ void packed_mirrored_index_kernel(const int32_t* __restrict__ cup, int num_docs, long long T, int cp,
                                             int rank, long long t_local, long long total,
                                             int32_t* __restrict__ idx, int32_t* err) {
  grid_dependency_wait();
  grid_dependents_launch();
  check_offsets(cup, num_docs, T, cp, 0, err);
  for (long long o = blockIdx.x * (long long)blockDim.x + threadIdx.x; o < total;
       o += (long long)gridDim.x * blockDim.x) {
    int r = rank;
    long long t = o;
    if (rank < 0) { r = static_cast<int>(o / t_local); t = o - (long long)r * t_local; }
    const long long p = mirrored_slot(T, cp, r, t);
    idx[o] = static_cast<int32_t>(p);
  }
}

// restore[p] = row of the rank-major gathered buffer holding physical slot p.
__global__ void restore_index_kernel(int strategy, const int32_t* __restrict__ cup, int num_docs, long long T,
                                     int cp, int32_t* __restrict__ restore, int32_t* err) {
  grid_dependency_wait();
  grid_dependents_launch();
  check_offsets(cup, num_docs, T, cp, strategy == CPTHD_DUAL_CHUNK_SWAP, err);
  const long long t_local = T / cp;
  for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < T;
       p += (long long)gridDim.x * blockDim.x) {
    long long g = p;
    if (strategy != CPTHD_NO_LOAD_BALANCE) {
      long long start = 0, len = T;
      if (strategy == CPTHD_DUAL_CHUNK_SWAP) {
        const int j = upper_bound_doc(cup, num_docs, p);
        start = __ldg(cup + j);
        len = static_cast<long long>(__ldg(cup + j + 1)) - start;
      }
      const long long chunk = len / (2LL * cp);
      const long long u = p - start;
      if (chunk > 0 && u >= 0 && u < len) {
        const long long c = u / chunk;
        const long long r = (c < cp) ? c : 2LL * cp - 1 - c;
        const long long within = (c < cp) ? (u - c * chunk) : (chunk + u - c * chunk);
        g = r * t_local + start / cp + within;
      } else {
        g = 0;  // malformed offsets; recorded by check_offsets
      }
    }
    restore[p] = static_cast<int32_t>(g);
  }
}

}  // namespace cpthd

extern "C" int cp_local_tokens(int strategy, int64_t T, int cp_size, int64_t* t_local_host) {
  if (t_local_host == nullptr || cp_size < 1 || T < 0) return CPTHD_ERR_INVALID_ARG;
  if (strategy != CPTHD_DUAL_CHUNK_SWAP && strategy != CPTHD_NO_LOAD_BALANCE && strategy != CPTHD_PACKED_MIRRORED)
    return CPTHD_ERR_INVALID_ARG;
  if (T % cp_size != 0) return CPTHD_ERR_NOT_DIVISIBLE;
  if (strategy == CPTHD_PACKED_MIRRORED && T % (2LL * cp_size) != 0) return CPTHD_ERR_NOT_DIVISIBLE;
  *t_local_host = T / cp_size;
  return CPTHD_OK;
}

extern "C" int cp_partition_index(int strategy, const int32_t* cu_seqlens_padded_dev, int num_docs,
                                  int64_t T, int cp_size, int rank, int32_t* idx_out_dev,
                                  int32_t* err_dev, cpthd_stream_t stream) {
  int64_t t_local = 0;
  int st = cp_local_tokens(strategy, T, cp_size, &t_local);
  if (st != CPTHD_OK) return st;
  if (rank < -1 || rank >= cp_size) return CPTHD_ERR_INVALID_ARG;
  if (num_docs < 0 || T > INT32_MAX) return CPTHD_ERR_INVALID_ARG;
  if (cu_seqlens_padded_dev == nullptr) return CPTHD_ERR_INVALID_ARG;
  const long long total = (rank < 0) ? (long long)cp_size * t_local : t_local;
  if (total > 0 && idx_out_dev == nullptr) return CPTHD_ERR_INVALID_ARG;
  if (total > 0 && num_docs == 0) return CPTHD_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool dcs = (strategy == CPTHD_DUAL_CHUNK_SWAP);
  const long long work = total > num_docs + 1 ? total : num_docs + 1;
  const int sms = cpthd::sm_count();
  if (sms < 1) return CPTHD_ERR_CUDA;
  const int grid = cpthd::grid_for(work, 256, sms * 16);
  auto kernel = dcs ? cpthd::dual_chunk_swap_index_kernel
                    : (strategy == CPTHD_NO_LOAD_BALANCE ? cpthd::no_load_balance_index_kernel
                                                         : cpthd::packed_mirrored_index_kernel);
  CPTHD_TRY_CUDA(cpthd::launch_pdl(kernel, dim3(grid), dim3(256), 0, s, cu_seqlens_padded_dev, num_docs,
                                   static_cast<long long>(T), cp_size, rank, static_cast<long long>(t_local), total,
                                   idx_out_dev, err_dev));
  return CPTHD_OK;
}

extern "C" int cp_restore_index(int strategy, const int32_t* cu_seqlens_padded_dev, int num_docs, int64_t T,
                                int cp_size, int32_t* restore_idx_out_dev, int32_t* err_dev, cpthd_stream_t stream) {
  int64_t t_local = 0;
  int st = cp_local_tokens(strategy, T, cp_size, &t_local);
  if (st != CPTHD_OK) return st;
  if (num_docs < 0 || T > INT32_MAX || cu_seqlens_padded_dev == nullptr) return CPTHD_ERR_INVALID_ARG;
  if (T > 0 && (restore_idx_out_dev == nullptr || num_docs == 0)) return CPTHD_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long work = T > num_docs + 1 ? T : num_docs + 1;
  const int sms = cpthd::sm_count();
  if (sms < 1) return CPTHD_ERR_CUDA;
  CPTHD_TRY_CUDA(cpthd::launch_pdl(cpthd::restore_index_kernel, dim3(cpthd::grid_for(work, 256, sms * 16)),
                                   dim3(256), 0, s, strategy, cu_seqlens_padded_dev, num_docs,
                                   static_cast<long long>(T), cp_size, restore_idx_out_dev, err_dev));
  return CPTHD_OK;
}
