// Per-row and per-group metadata of the causal packed-THD attention.
//
// Document isolation and causality (TransformerEngine PR #3221, "Scope and
// constraints": causal, window_size = (-1, 0); "What changed": logical
// document boundaries kept through THD metadata) reduce, for a query row with
// physical index p in document j, to one contiguous interval of allowed key
// slots: [cu_seqlens_padded[j], p]. Pad keys of document j lie beyond every
// real query of j, so they never fall inside an interval. A pad query row
// gets the empty interval.
//
// The attention kernel gives each CTA two 128-row query tiles that read the
// same K/V blocks: either one row tile under two query heads of the same KV
// head (a "row group" of 128 rows), or two consecutive row tiles under one
// head (a row group of 256 rows). For every row group the metadata kernel
// stores the union of its rows' intervals (one interval per document present,
// sorted by document), the number of kBlockN-key blocks that covers them (the
// group's cost), and for each 128-row tile the largest interval start and
// smallest interval end over its real rows: a key block inside
// [max_lo, min_hi] needs no mask. A second kernel orders the groups by
// decreasing cost, so that a grid launched in that order hands the longest
// work to the SMs first.
#pragma once

#include "partition_math.cuh"

namespace cpthd {

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // keys per key block
constexpr int kMaxSortGroups = 8192;

struct GroupInfo {
  int n_intervals;
  int n_blocks;
  int max_lo[2];  // per tile, over real rows; INT_MIN when the tile has none
  int min_hi[2];  // per tile, over real rows; INT_MAX when the tile has none
};

struct AttnWorkspace {
  int32_t* row_lo;        // [ngroups * group_rows]
  int32_t* row_hi;        // [ngroups * group_rows]
  GroupInfo* group_info;  // [ngroups]
  int2* intervals;        // [ngroups * group_rows] (start, end) inclusive
  int32_t* order;         // [ngroups]
};

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

inline size_t attn_workspace_bytes(long long ngroups, int group_rows) {
  const long long rows = ngroups * group_rows;
  size_t b = 0;
  b += align256(sizeof(int32_t) * rows);
  b += align256(sizeof(int32_t) * rows);
  b += align256(sizeof(GroupInfo) * ngroups);
  b += align256(sizeof(int2) * rows);
  b += align256(sizeof(int32_t) * ngroups);
  return b;
}

inline AttnWorkspace carve_workspace(void* base, long long ngroups, int group_rows) {
  const long long rows = ngroups * group_rows;
  char* p = static_cast<char*>(base);
  AttnWorkspace w;
  w.row_lo = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * rows);
  w.row_hi = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * rows);
  w.group_info = reinterpret_cast<GroupInfo*>(p); p += align256(sizeof(GroupInfo) * ngroups);
  w.intervals = reinterpret_cast<int2*>(p); p += align256(sizeof(int2) * rows);
  w.order = reinterpret_cast<int32_t*>(p);
  return w;
}

// One block of ROWS threads per row group; thread t owns local row
// group * ROWS + t, whose physical slot comes from the slice's index list or
// from the partition formulas. The blocks also check the document table
// (offsets start at 0 and never decrease, padded offsets end at T,
// L_j <= P_j, and under a computed DualChunkSwap slice every padded length
// is a multiple of 2*cp_size) in a grid-stride loop over documents.
template <int ROWS>
static __global__ void __launch_bounds__(ROWS) attn_group_meta_kernel(
    IndexGen slots, long long t_local, const int32_t* __restrict__ cu,
    const int32_t* __restrict__ cup, int num_docs, long long T, AttnWorkspace ws, int32_t* err) {
  constexpr int kWarps = ROWS / 32;
  __shared__ unsigned long long xbuf[2][ROWS];
  __shared__ int warp_sum[kWarps];
  __shared__ int red_blocks[kWarps];
  __shared__ int red_lo[kWarps];
  __shared__ int red_hi[kWarps];
  grid_dependency_wait();
  grid_dependents_launch();
  const int t = threadIdx.x;
  const int lane = t & 31, wid = t >> 5;
  const long long group = blockIdx.x;
  const long long row = group * ROWS + t;
  const int p = (row < t_local) ? slots.at(row) : 0;  // issued before anything waits

  for (long long j = blockIdx.x * (long long)ROWS + t; j <= num_docs; j += (long long)gridDim.x * ROWS) {
    if (j == 0 && (cu[0] != 0 || cup[0] != 0)) record_error(err, CPTHD_ERR_BAD_OFFSETS, 0);
    if (j == num_docs && cup[j] != T) record_error(err, CPTHD_ERR_BAD_OFFSETS, j);
    if (j < num_docs) {
      const int L = cu[j + 1] - cu[j];
      const int P = cup[j + 1] - cup[j];
      if (L < 0 || P < 0) record_error(err, CPTHD_ERR_BAD_OFFSETS, j);
      else if (L > P) record_error(err, CPTHD_ERR_PAD_LENGTH, j);
      else if (slots.idx == nullptr && slots.strategy == CPTHD_DUAL_CHUNK_SWAP && P % (2 * slots.cp) != 0)
        record_error(err, CPTHD_ERR_NOT_DIVISIBLE, j);
    }
  }

  int lo = 1, hi = 0;  // empty interval
  bool valid = false;
  int doc = 0;
  if (row < t_local) {
    if (p < 0 || p >= T) {
      record_error(err, CPTHD_ERR_INDEX_RANGE, row);
    } else {
      doc = upper_bound_doc(cup, num_docs, p);
      const int start = cup[doc];
      const int L = cu[doc + 1] - cu[doc];
      const int pos = p - start;
      // start >= 0 is re-checked so that malformed offsets can never widen
      // an interval beyond [0, T)
      if (pos >= 0 && pos < L && start >= 0) { valid = true; lo = start; hi = p; }
    }
  }
  ws.row_lo[row] = lo;
  ws.row_hi[row] = hi;
  // bitonic sort of the (document, end) keys, ascending, one key per
  // thread: partners closer than 32 rows are in the same warp and exchange
  // through shuffles; farther partners go through shared memory (double
  // buffered, one barrier per such stage)
  unsigned long long key = valid ? ((static_cast<unsigned long long>(doc) << 32) | static_cast<unsigned>(hi)) : ~0ull;
  int buf = 0;
  for (int k = 2; k <= ROWS; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      unsigned long long other;
      if (j >= 32) {
        xbuf[buf][t] = key;
        __syncthreads();
        other = xbuf[buf][t ^ j];
        buf ^= 1;
      } else {
        other = __shfl_xor_sync(0xffffffffu, key, j);
      }
      const bool up = ((t & k) == 0);
      const bool lower = ((t & j) == 0);
      key = (lower == up) ? (key < other ? key : other) : (key > other ? key : other);
    }
  }
  xbuf[buf][t] = key;
  __syncthreads();
  const unsigned long long nxt = (t + 1 < ROWS) ? xbuf[buf][t + 1] : ~0ull;
  const bool last = (key != ~0ull) && ((nxt >> 32) != (key >> 32));
  int my_lo = 0, my_hi = -1, my_blocks = 0;
  if (last) {
    const int d = static_cast<int>(key >> 32);
    my_lo = max(cup[d], 0);
    my_hi = static_cast<int>(key & 0xffffffffu);
    my_blocks = (my_hi - my_lo + kBlockN) / kBlockN;
  }
  // compact the intervals in document order; reduce cost and per-warp bounds
  const unsigned ballot = __ballot_sync(0xffffffffu, last);
  if (lane == 0) warp_sum[wid] = __popc(ballot);
  int blocks = my_blocks;
  int vlo = valid ? lo : INT_MIN;
  int vhi = valid ? hi : INT_MAX;
  for (int o = 16; o > 0; o >>= 1) {
    blocks += __shfl_xor_sync(0xffffffffu, blocks, o);
    vlo = max(vlo, __shfl_xor_sync(0xffffffffu, vlo, o));
    vhi = min(vhi, __shfl_xor_sync(0xffffffffu, vhi, o));
  }
  if (lane == 0) { red_blocks[wid] = blocks; red_lo[wid] = vlo; red_hi[wid] = vhi; }
  __syncthreads();
  int base = 0;
  for (int w = 0; w < wid; ++w) base += warp_sum[w];
  if (last) {
    const int slot = base + __popc(ballot & ((1u << lane) - 1u));
    ws.intervals[group * ROWS + slot] = make_int2(my_lo, my_hi);
  }
  if (t == 0) {
    GroupInfo gi;
    gi.n_intervals = 0;
    gi.n_blocks = 0;
    for (int x = 0; x < 2; ++x) { gi.max_lo[x] = INT_MIN; gi.min_hi[x] = INT_MAX; }
    for (int w = 0; w < kWarps; ++w) {
      gi.n_intervals += warp_sum[w];
      gi.n_blocks += red_blocks[w];
      const int x = (w * 32) / kBlockM;  // tile of this warp's rows
      gi.max_lo[x] = max(gi.max_lo[x], red_lo[w]);
      gi.min_hi[x] = min(gi.min_hi[x], red_hi[w]);
    }
    if (ROWS == kBlockM) { gi.max_lo[1] = gi.max_lo[0]; gi.min_hi[1] = gi.min_hi[0]; }
    ws.group_info[group] = gi;
  }
}

// One block of 1024 threads: order[] = groups by decreasing block count
// (ties by group index, so equal-cost groups keep their natural order).
// cost[i * cost_stride] is group i's block count. Larger group counts keep
// the natural order.
static __global__ void __launch_bounds__(1024) attn_group_order_kernel(int ngroups, const int* __restrict__ cost,
                                                                       int cost_stride, int32_t* __restrict__ order) {
  __shared__ unsigned keys[kMaxSortGroups];
  grid_dependency_wait();
  grid_dependents_launch();
  const int t = threadIdx.x;
  if (ngroups > kMaxSortGroups) {
    for (int i = t; i < ngroups; i += blockDim.x) order[i] = i;
    return;
  }
  int n2 = 1;
  while (n2 < ngroups) n2 <<= 1;
  for (int i = t; i < n2; i += blockDim.x) {
    if (i < ngroups) {
      const unsigned c = static_cast<unsigned>(min(max(cost[static_cast<long long>(i) * cost_stride], 0), (1 << 18) - 1));
      keys[i] = ((c ^ 0x3ffffu) << 13) | static_cast<unsigned>(i);
    } else {
      keys[i] = 0xffffffffu;
    }
  }
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = t; i < n2; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned a = keys[i], b = keys[ixj];
          const bool up = ((i & k) == 0);
          if ((a > b) == up) { keys[i] = b; keys[ixj] = a; }
        }
      }
      __syncthreads();
    }
  }
  for (int i = t; i < ngroups; i += blockDim.x) order[i] = static_cast<int>(keys[i] & 0x1fffu);
}

}  // namespace cpthd
