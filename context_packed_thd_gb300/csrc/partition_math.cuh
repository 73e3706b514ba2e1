// Closed forms of the partition index, shared by the index kernels, the
// fused partition-and-gather kernel and the attention metadata kernel.
//
// TransformerEngine PR #3221 ("Why", "What changed"): DualChunkSwap cuts
// every document into 2*cp_size chunks and rank r owns chunks r and
// 2*cp_size-1-r (the head-tail split, torchtitan PR #2144 "Summary"); within
// a rank, documents keep pack order and chunk r precedes chunk
// 2*cp_size-1-r, so the rank-local offsets are cu_seqlens_padded / cp_size.
// NO_LOAD_BALANCE cuts the whole physical buffer into cp_size contiguous
// chunks, rank-major. The packed mirrored partition is DualChunkSwap of the
// whole buffer taken as one sequence.
#pragma once

#include "common.cuh"

namespace cpthd {

// Offset-table checks: cup starts at 0, never decreases and ends at T; under
// DualChunkSwap every padded length is a multiple of 2*cp_size. Grid-stride
// over documents with (first, stride) supplied by the caller.
__device__ __forceinline__ void check_offsets_range(const int32_t* __restrict__ cup, int num_docs, long long T,
                                                    int cp, int dcs, int32_t* err, long long first,
                                                    long long stride) {
  for (long long j = first; j <= num_docs; j += stride) {
    const int32_t a = cup[j];
    if (j == 0 && a != 0) record_error(err, CPTHD_ERR_BAD_OFFSETS, 0);
    if (j == num_docs && a != T) record_error(err, CPTHD_ERR_BAD_OFFSETS, j);
    if (j < num_docs) {
      const int32_t b = cup[j + 1];
      if (b < a) record_error(err, CPTHD_ERR_BAD_OFFSETS, j);
      else if (dcs && ((b - a) % (2 * cp)) != 0) record_error(err, CPTHD_ERR_NOT_DIVISIBLE, j);
    }
  }
}

// Physical slot of rank r's local slot t under DualChunkSwap: find the
// document j whose local range [cup[j] / cp, cup[j+1] / cp) holds t, then
// map t into chunk r or chunk 2*cp-1-r of that document.
__device__ __forceinline__ long long dcs_slot(const int32_t* __restrict__ cup, int num_docs, int cp, int r,
                                              long long t) {
  int lo = 0, hi = num_docs;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<long long>(__ldg(cup + mid) / cp) <= t) lo = mid; else hi = mid;
  }
  const long long start = __ldg(cup + lo);
  const long long chunk = (static_cast<long long>(__ldg(cup + lo + 1)) - start) / (2 * cp);
  const long long u = t - start / cp;
  return (u < chunk) ? start + r * chunk + u : start + (2LL * cp - 1 - r) * chunk + (u - chunk);
}

// NO_LOAD_BALANCE: rank-major contiguous chunks of t_local slots.
__device__ __forceinline__ long long nlb_slot(int r, long long t_local, long long t) { return r * t_local + t; }

// Packed mirrored: DualChunkSwap of [0, T) as one sequence, chunk = T / (2 cp).
__device__ __forceinline__ long long mirrored_slot(long long T, int cp, int r, long long t) {
  const long long chunk = T / (2LL * cp);
  return (t < chunk) ? r * chunk + t : (2LL * cp - 1 - r) * chunk + (t - chunk);
}

// Where row t of a rank's slice lives in the physical buffer: read from an
// index list, or computed from one of the closed forms above.
struct IndexGen {
  const int32_t* idx;  // non-null: read the list
  int strategy;
  const int32_t* cup;
  int num_docs;
  long long T;
  int cp;
  int rank;
  long long t_local;
  __device__ __forceinline__ int32_t at(long long row) const {
    if (idx != nullptr) return __ldg(idx + row);
    long long slot;
    if (strategy == CPTHD_DUAL_CHUNK_SWAP) slot = dcs_slot(cup, num_docs, cp, rank, row);
    else if (strategy == CPTHD_NO_LOAD_BALANCE) slot = nlb_slot(rank, t_local, row);
    else slot = mirrored_slot(T, cp, rank, row);
    return static_cast<int32_t>(slot);
  }
};

inline IndexGen index_list(const int32_t* idx) {
  IndexGen g{};
  g.idx = idx;
  return g;
}

inline IndexGen index_formula(int strategy, const int32_t* cup, int num_docs, long long T, int cp, int rank,
                              long long t_local) {
  IndexGen g{};
  g.idx = nullptr;
  g.strategy = strategy;
  g.cup = cup;
  g.num_docs = num_docs;
  g.T = T;
  g.cp = cp;
  g.rank = rank;
  g.t_local = t_local;
  return g;
}

}  // namespace cpthd
