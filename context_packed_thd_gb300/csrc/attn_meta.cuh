// Per-row and per-tile metadata of the causal packed-THD attention.
//
// Document isolation and causality (TransformerEngine PR #3221, "Scope and
// constraints": causal, window_size = (-1, 0); "What changed": logical
// document boundaries kept through THD metadata) reduce, for a query row with
// physical index p in document j, to one contiguous interval of allowed key
// slots: [cu_seqlens_padded[j], p]. Pad keys of document j lie beyond every
// real query of j, so they never fall inside an interval. A pad query row
// gets the empty interval.
//
// For every tile of kBlockM consecutive local rows the metadata kernel
// stores the union of its rows' intervals (one interval per document present
// in the tile, sorted by document), the number of kBlockN-key blocks that
// covers them (the tile's cost), and the largest interval start / smallest
// interval end over its real rows: a key block inside [maxLo, minHi] needs no
// mask. A second kernel orders the tiles by decreasing cost, so that a grid
// launched in that order hands the longest work to the SMs first.
#pragma once

#include "common.cuh"

namespace cpthd {

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // keys per key block
constexpr int kMaxSortTiles = 8192;

struct TileInfo {
  int n_intervals;
  int n_blocks;
  int max_lo;  // over real rows; INT_MIN when the tile has none
  int min_hi;  // over real rows; INT_MAX when the tile has none
};

struct AttnWorkspace {
  int32_t* row_lo;      // [ntiles * kBlockM]
  int32_t* row_hi;      // [ntiles * kBlockM]
  TileInfo* tile_info;  // [ntiles]
  int2* intervals;      // [ntiles * kBlockM] (start, end) inclusive
  int32_t* order;       // [ntiles]
};

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

inline size_t attn_workspace_bytes(long long ntiles) {
  size_t b = 0;
  b += align256(sizeof(int32_t) * ntiles * kBlockM);
  b += align256(sizeof(int32_t) * ntiles * kBlockM);
  b += align256(sizeof(TileInfo) * ntiles);
  b += align256(sizeof(int2) * ntiles * kBlockM);
  b += align256(sizeof(int32_t) * ntiles);
  return b;
}

inline AttnWorkspace carve_workspace(void* base, long long ntiles) {
  char* p = static_cast<char*>(base);
  AttnWorkspace w;
  w.row_lo = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * ntiles * kBlockM);
  w.row_hi = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * ntiles * kBlockM);
  w.tile_info = reinterpret_cast<TileInfo*>(p); p += align256(sizeof(TileInfo) * ntiles);
  w.intervals = reinterpret_cast<int2*>(p); p += align256(sizeof(int2) * ntiles * kBlockM);
  w.order = reinterpret_cast<int32_t*>(p);
  return w;
}

// Document table checks: offsets start at 0, never decrease, padded offsets
// end at T, and L_j <= P_j.
__global__ void attn_validate_docs_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ cup,
                                          int num_docs, long long T, int32_t* err) {
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j <= num_docs; j += gridDim.x * blockDim.x) {
    if (j == 0 && (cu[0] != 0 || cup[0] != 0)) record_error(err, CPTHD_ERR_BAD_OFFSETS, 0);
    if (j == num_docs && cup[j] != T) record_error(err, CPTHD_ERR_BAD_OFFSETS, j);
    if (j < num_docs) {
      const int L = cu[j + 1] - cu[j];
      const int P = cup[j + 1] - cup[j];
      if (L < 0 || P < 0) record_error(err, CPTHD_ERR_BAD_OFFSETS, j);
      else if (L > P) record_error(err, CPTHD_ERR_PAD_LENGTH, j);
    }
  }
}

// One block of kBlockM threads per tile; thread t owns local row tile*kBlockM + t.
__global__ void __launch_bounds__(kBlockM) attn_tile_meta_kernel(
    const int32_t* __restrict__ idx, long long t_local, const int32_t* __restrict__ cu,
    const int32_t* __restrict__ cup, int num_docs, long long T, AttnWorkspace ws, int32_t* err) {
  __shared__ unsigned long long keys[kBlockM];
  __shared__ int warp_sum[kBlockM / 32];
  __shared__ int red_blocks[kBlockM / 32];
  __shared__ int red_lo[kBlockM / 32];
  __shared__ int red_hi[kBlockM / 32];
  const int t = threadIdx.x;
  const int lane = t & 31, wid = t >> 5;
  const long long tile = blockIdx.x;
  const long long row = tile * kBlockM + t;

  int lo = 1, hi = 0;  // empty interval
  bool valid = false;
  int doc = 0;
  if (row < t_local) {
    const int p = idx[row];
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
  keys[t] = valid ? ((static_cast<unsigned long long>(doc) << 32) | static_cast<unsigned>(hi))
                  : ~0ull;
  __syncthreads();
  // bitonic sort of the (document, end) keys, ascending
  for (int k = 2; k <= kBlockM; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      const int ixj = t ^ j;
      if (ixj > t) {
        const unsigned long long a = keys[t], b = keys[ixj];
        const bool up = ((t & k) == 0);
        if ((a > b) == up) { keys[t] = b; keys[ixj] = a; }
      }
      __syncthreads();
    }
  }
  const unsigned long long key = keys[t];
  const unsigned long long nxt = (t + 1 < kBlockM) ? keys[t + 1] : ~0ull;
  const bool last = (key != ~0ull) && ((nxt >> 32) != (key >> 32));
  int my_lo = 0, my_hi = -1, my_blocks = 0;
  if (last) {
    const int d = static_cast<int>(key >> 32);
    my_lo = max(cup[d], 0);
    my_hi = static_cast<int>(key & 0xffffffffu);
    my_blocks = (my_hi - my_lo + kBlockN) / kBlockN;
  }
  // compact the interval ends in document order
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
    ws.intervals[tile * kBlockM + slot] = make_int2(my_lo, my_hi);
  }
  if (t == 0) {
    TileInfo ti;
    ti.n_intervals = 0; ti.n_blocks = 0; ti.max_lo = INT_MIN; ti.min_hi = INT_MAX;
    for (int w = 0; w < kBlockM / 32; ++w) {
      ti.n_intervals += warp_sum[w];
      ti.n_blocks += red_blocks[w];
      ti.max_lo = max(ti.max_lo, red_lo[w]);
      ti.min_hi = min(ti.min_hi, red_hi[w]);
    }
    ws.tile_info[tile] = ti;
  }
}

// One block of 1024 threads: order[] = tiles by decreasing block count
// (ties by tile index). Larger tile counts keep the natural order.
__global__ void __launch_bounds__(1024) attn_tile_order_kernel(int ntiles, AttnWorkspace ws) {
  __shared__ unsigned keys[kMaxSortTiles];
  const int t = threadIdx.x;
  if (ntiles > kMaxSortTiles) {
    for (int i = t; i < ntiles; i += blockDim.x) ws.order[i] = i;
    return;
  }
  int n2 = 1;
  while (n2 < ntiles) n2 <<= 1;
  for (int i = t; i < n2; i += blockDim.x) {
    if (i < ntiles) {
      const unsigned cost = static_cast<unsigned>(min(max(ws.tile_info[i].n_blocks, 0), (1 << 18) - 1));
      keys[i] = ((cost ^ 0x3ffffu) << 13) | static_cast<unsigned>(i);
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
  for (int i = t; i < ntiles; i += blockDim.x) ws.order[i] = static_cast<int>(keys[i] & 0x1fffu);
}

}  // namespace cpthd
