// The forward attention's plan: variable-height query tiles cut at document
// boundaries, their key intervals, and the order the attention kernel takes
// them in.
//
// A query row with physical slot p in document j may attend exactly the key
// slots [cu_seqlens_padded[j], p] (TransformerEngine PR #3221, "Scope and
// constraints": causal, window_size = (-1, 0); "What changed": document
// boundaries kept through THD metadata). The tensor cores work on 128-row
// query tiles, and a tile pays for the union of its rows' key intervals, so
// the plan cuts the slice's rows where the document changes: every run of
// consecutive rows of one document (a DualChunkSwap rank holds each document
// as one run, chunk r then chunk 2*cp_size-1-r; a NO_LOAD_BALANCE rank as a
// contiguous piece) is cut into 128-row tiles aligned to the run's end, with
// the remainder as the run's first tile, which holds its earliest positions
// and therefore its cheapest rows. Runs shorter than a tile are packed
// together, in order, while they fit in 128 rows (a packed tile pays each
// document's keys once, as separate tiles would). Any two consecutive tiles
// then hold more than 128 rows together, so a slice of n rows has at most
// 2 * ceil(n / 128) + 1 tiles; buffers and grids are sized by that bound.
//
// Kernels, in stream order (both launched by thd_causal_attn_plan):
//  1. attn_rows_kernel: per local row, its document and key interval, and
//     whether it starts a run; also checks the offset table.
//  2. attn_fwd_group_kernel: each block finds its own group's tiles (the run
//     starts in order, then the greedy cut, walked until they are known;
//     block 0 walks to the end and publishes the counts), then, per group
//     (one tile under two query heads when
//     the GQA group size is even, else two consecutive tiles under one head)
//     the union of its rows' intervals, one per document, sorted; its cost
//     in 128-key blocks; and per tile the bounds inside which a key block
//     needs no mask. The block that finishes last writes the attention
//     kernel's schedule: when there are more work items than SMs, the
//     groups' order by decreasing cost; always, the running total of the
//     work (128-key blocks, at least one per item, plus a fixed cost per
//     item) over the items in that order, and for every attention CTA the
//     first and last item of its equal share of the total (see the
//     attention kernel for how a share that cuts an item is handled).
#pragma once

#include "attn_meta.cuh"

namespace cpthd {

struct FwdGroup {
  int n_intervals;
  int n_blocks;   // cost: 128-key blocks over the group's intervals
  int max_lo[2];  // per tile, over real rows; INT_MIN when the tile has none
  int min_hi[2];  // per tile, over real rows; INT_MAX when the tile has none
  int row0[2];    // first local row of each tile
  int h[2];       // rows of each tile (0: no tile)
};

// Attention CTAs the schedule is made for (at most; the grid is the smaller
// of this and the SM count), and the least work a CTA is given.
constexpr int kMaxCtas = 160;
constexpr int kMinCtaBlocks = 4;
// The fixed cost of a work item in key blocks (its Q load, first scores and
// epilogue take about as long as three key blocks): the schedule counts an
// item as max(blocks, 1) + kItemCost, its blocks first.
constexpr int kItemCost = 3;
// Equal shares pay off when items are long: below this mean number of key
// blocks per item, the CTAs instead take whole items from a counter in the
// plan's order (their fixed costs and cache reuse then balance better than
// cut pieces do).
constexpr int kSharesMinMeanBlocks = 64;

// Device arrays of a plan, carved from the caller's workspace.
struct FwdPlan {
  int32_t* row_lo;     // [n] first allowed key slot of each local row (empty: lo > hi)
  int32_t* row_hi;     // [n] last allowed key slot
  int32_t* row_doc;    // [n] document of the row's slot, -1 when the slot is out of range
  int32_t* seg;        // [n] run starts past the group blocks' shared copy (scratch)
  uint32_t* run_bits;  // [ceil(n / 32)] bit r of word w: row 32 w + r starts a run
  int32_t* ctrl;       // [0] tiles, [1] groups, [2] next work item (taken from a counter), [3] attention
                       // CTAs finished, [4] group blocks finished (cleared by the rows kernel), [5]
                       // attention CTAs with work, [6] 1: equal shares, 0: items from the counter
  FwdGroup* groups;    // [max_groups]
  int2* intervals;     // [max_groups * group_rows] (start, end) inclusive, per group
  int32_t* order;      // [max_groups]
  long long* cum;      // [max_groups + 1] work before each position of the order (blocks x head units)
  long long* work;     // [1] the total
  int32_t* cta_first;  // [kMaxCtas] first work item of each CTA's share
  int32_t* cta_last;   // [kMaxCtas] last work item of each CTA's share
  int32_t* flags;      // [2 * kMaxCtas] hand-off flags of the pieces of cut items (cleared by the rows
                       // kernel and by the attention kernel's last CTA)
};

struct FwdShape {
  long long n;           // query rows of the slice
  long long max_tiles;   // 2 * ceil(n / 128) + 1
  long long max_groups;  // tiles (head pairs) or ceil(tiles / 2) (tile pairs)
  int group_rows;        // 128 (head pairs) or 256 (tile pairs): interval slots per group
  int head_pairs;        // 1: a group is one tile under two query heads of one KV head
};

inline FwdShape fwd_shape(long long n, int Hq, int Hkv) {
  FwdShape s;
  s.n = n;
  s.head_pairs = ((Hq / Hkv) % 2 == 0) ? 1 : 0;
  s.max_tiles = 2 * ((n + kBlockM - 1) / kBlockM) + 1;
  s.max_groups = s.head_pairs ? s.max_tiles : (s.max_tiles + 1) / 2;
  s.group_rows = s.head_pairs ? kBlockM : 2 * kBlockM;
  return s;
}

inline size_t fwd_plan_bytes(const FwdShape& s) {
  size_t b = 0;
  b += 4 * align256(sizeof(int32_t) * s.n);
  b += align256(sizeof(uint32_t) * ((s.n + 31) / 32));
  b += align256(sizeof(int32_t) * 8);
  b += align256(sizeof(FwdGroup) * s.max_groups);
  b += align256(sizeof(int2) * s.max_groups * s.group_rows);
  b += align256(sizeof(int32_t) * s.max_groups);
  b += align256(sizeof(long long) * (s.max_groups + 1));
  b += align256(sizeof(long long));
  b += 3 * align256(sizeof(int32_t) * 2 * kMaxCtas);
  return b;
}

inline FwdPlan carve_fwd_plan(void* base, const FwdShape& s) {
  char* p = static_cast<char*>(base);
  FwdPlan w;
  w.row_lo = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * s.n);
  w.row_hi = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * s.n);
  w.row_doc = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * s.n);
  w.seg = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * s.n);
  w.run_bits = reinterpret_cast<uint32_t*>(p); p += align256(sizeof(uint32_t) * ((s.n + 31) / 32));
  w.ctrl = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * 8);
  w.groups = reinterpret_cast<FwdGroup*>(p); p += align256(sizeof(FwdGroup) * s.max_groups);
  w.intervals = reinterpret_cast<int2*>(p); p += align256(sizeof(int2) * s.max_groups * s.group_rows);
  w.order = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * s.max_groups);
  w.cum = reinterpret_cast<long long*>(p); p += align256(sizeof(long long) * (s.max_groups + 1));
  w.work = reinterpret_cast<long long*>(p); p += align256(sizeof(long long));
  w.cta_first = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * 2 * kMaxCtas);
  w.cta_last = reinterpret_cast<int32_t*>(p); p += align256(sizeof(int32_t) * 2 * kMaxCtas);
  w.flags = reinterpret_cast<int32_t*>(p);
  return w;
}

// 1. One thread per local row: the row's physical slot (from the slice's
// index list or the partition formulas), its document and its key interval,
// and whether the row starts a run of equal documents (its document differs
// from the row before it); each warp writes those 32 flags as one word. The
// blocks also check the document table (offsets start at 0 and never
// decrease, padded offsets end at T, L_j <= P_j, and under a computed
// DualChunkSwap slice every padded length is a multiple of 2*cp_size) in a
// grid-stride loop over documents.
static __device__ __forceinline__ int row_document(const IndexGen& slots, long long row, const int32_t* cup,
                                                   int num_docs, long long T) {
  const int p = slots.at(row);
  return (p < 0 || p >= T) ? -1 : upper_bound_doc(cup, num_docs, p);
}

static __global__ void __launch_bounds__(256) attn_rows_kernel(IndexGen slots, long long n,
                                                               const int32_t* __restrict__ cu,
                                                               const int32_t* __restrict__ cup, int num_docs,
                                                               long long T, FwdPlan plan, int32_t* err) {
  __shared__ int warp_last_doc[8];
  grid_dependency_wait();
  grid_dependents_launch();
  const long long i = blockIdx.x * 256LL + threadIdx.x;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const bool in = i < n;
  const int p = in ? slots.at(i) : 0;  // issued before the checks below
  // the document of the row before this block's first row (a run may go on
  // across the block boundary)
  int doc_before_block = -2;
  if (threadIdx.x == 0 && i > 0 && in) doc_before_block = row_document(slots, i - 1, cup, num_docs, T);
  for (long long j = i; j <= num_docs; j += static_cast<long long>(gridDim.x) * 256) {
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
  // the group kernel's completion count starts at zero (it counts blocks
  // only after this kernel has finished), and so do the attention kernel's
  // hand-off flags
  if (i == 0) plan.ctrl[4] = 0;
  for (long long j = i; j < 2 * kMaxCtas; j += static_cast<long long>(gridDim.x) * 256) plan.flags[j] = 0;
  int lo = 1, hi = 0, doc = -1;  // empty interval
  if (in) {
    if (p < 0 || p >= T) {
      record_error(err, CPTHD_ERR_INDEX_RANGE, i);
    } else {
      doc = upper_bound_doc(cup, num_docs, p);
      const int start = cup[doc];
      const int L = cu[doc + 1] - cu[doc];
      const int pos = p - start;
      // start >= 0 is re-checked so that malformed offsets can never widen
      // an interval beyond [0, T)
      if (pos >= 0 && pos < L && start >= 0) { lo = start; hi = p; }
    }
    plan.row_lo[i] = lo;
    plan.row_hi[i] = hi;
    plan.row_doc[i] = doc;
  }
  // run starts: compare with the row before (same warp: a shuffle; the
  // previous warp's last row: shared memory; the previous block: the
  // document computed above)
  int before = __shfl_up_sync(0xffffffffu, doc, 1);
  if (lane == 31) warp_last_doc[wid] = doc;
  __syncthreads();
  if (lane == 0) before = (wid > 0) ? warp_last_doc[wid - 1] : doc_before_block;
  const bool starts = in && (i == 0 || doc != before);
  const unsigned bits = __ballot_sync(0xffffffffu, starts);
  if (lane == 0 && i < n) plan.run_bits[i >> 5] = bits;
}

// 3. One block of ROWS threads per group (grid: max_groups): thread t owns
// row t of tile A (t < 128) or row t - 128 of tile B. Groups past the
// count get an empty record. The rows' intervals are sorted by (document,
// end) with a bitonic sort (partners closer than 32 rows exchange through
// warp shuffles, the rest through shared memory), and the last row of each
// document gives that document's interval [cup[j], its largest slot].
// The intervals and record of real group g (the body of attn_fwd_group_kernel).
template <int ROWS>
static __device__ __forceinline__ void group_intervals(const int32_t* __restrict__ cup, const FwdPlan& plan, int g,
                                                       int2 A, int2 B, unsigned long long (&xbuf)[2][ROWS],
                                                       int* warp_sum, int* red_blocks, int* red_lo, int* red_hi) {
  constexpr int kWarps = ROWS / 32;
  const int t = threadIdx.x;
  const int lane = t & 31, wid = t >> 5;
  const int x = (ROWS == 2 * kBlockM) ? (t >> 7) : 0;
  const int r = t & (kBlockM - 1);
  const int2 tile = x ? B : A;
  const bool in_tile = r < tile.y;
  const long long row = static_cast<long long>(tile.x) + r;
  int lo = 1, hi = 0, doc = 0;
  if (in_tile) {
    lo = plan.row_lo[row];
    hi = plan.row_hi[row];
    doc = plan.row_doc[row];
  }
  const bool valid = in_tile && lo <= hi && doc >= 0;
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
    plan.intervals[static_cast<long long>(g) * ROWS + slot] = make_int2(my_lo, my_hi);
  }
  if (t == 0) {
    FwdGroup gi;
    gi.n_intervals = 0;
    gi.n_blocks = 0;
    for (int y = 0; y < 2; ++y) { gi.max_lo[y] = INT_MIN; gi.min_hi[y] = INT_MAX; }
    for (int w = 0; w < kWarps; ++w) {
      gi.n_intervals += warp_sum[w];
      gi.n_blocks += red_blocks[w];
      const int y = (w * 32) / kBlockM;  // tile of this warp's rows
      gi.max_lo[y] = max(gi.max_lo[y], red_lo[w]);
      gi.min_hi[y] = min(gi.min_hi[y], red_hi[w]);
    }
    gi.row0[0] = A.x;
    gi.h[0] = A.y;
    if (ROWS == kBlockM) {
      gi.max_lo[1] = gi.max_lo[0];
      gi.min_hi[1] = gi.min_hi[0];
      gi.row0[1] = A.x;
      gi.h[1] = A.y;
    } else {
      gi.row0[1] = B.x;
      gi.h[1] = B.y;
    }
    plan.groups[g] = gi;
  }
}


// The block that finishes last then writes the attention kernel's schedule.
// When sort_n > 0: the LPT order of the groups (decreasing cost, ties by
// index, so unused groups come last) by a bitonic sort of sort_n (a power of
// two >= the grid) keys in dynamic shared memory. Always: the running total
// of the work over the positions of the order (each group's blocks, at least
// one, plus kItemCost, times the head units), and for each of the G attention
// CTAs (G: the
// grid, fewer when the work is small) the first and last work item of its
// share [c W / G, (c + 1) W / G). cum_sh (cum_cap entries) keeps the running
// totals for the searches when they fit.
template <int ROWS>
static __device__ void schedule_last_block(const FwdPlan& plan, int ngroups_total, int sort_n, int units, int grid,
                                           long long* cum_sh, int cum_cap, long long* scan_sh) {
  extern __shared__ unsigned sort_keys[];
  const int t = threadIdx.x;
  if (sort_n > 0) {
    for (int i = t; i < sort_n; i += ROWS) {
      if (i < ngroups_total) {
        const int c = __ldcg(&plan.groups[i].n_blocks);  // written by other blocks: read past L1
        const unsigned cost = static_cast<unsigned>(min(max(c, 0), (1 << 18) - 1));
        sort_keys[i] = ((cost ^ 0x3ffffu) << 13) | static_cast<unsigned>(i);
      } else {
        sort_keys[i] = 0xffffffffu;
      }
    }
    __syncthreads();
    for (int k = 2; k <= sort_n; k <<= 1) {
      for (int j = k >> 1; j > 0; j >>= 1) {
        for (int i = t; i < sort_n; i += ROWS) {
          const int ixj = i ^ j;
          if (ixj > i) {
            const unsigned a = sort_keys[i], b = sort_keys[ixj];
            const bool up = ((i & k) == 0);
            if ((a > b) == up) { sort_keys[i] = b; sort_keys[ixj] = a; }
          }
        }
        __syncthreads();
      }
    }
    for (int i = t; i < ngroups_total; i += ROWS) plan.order[i] = static_cast<int>(sort_keys[i] & 0x1fffu);
  }
  // running totals: each thread sums a contiguous run of positions (keeping
  // the terms in cum_sh when they fit), a shuffle scan over the threads
  // places the runs
  const int P = min(max(__ldcg(plan.ctrl + 1), 0), ngroups_total);
  const int per = (P + ROWS - 1) / ROWS;
  const int a = min(P, t * per);
  const int b = min(P, a + per);
  const bool in_shared = (P < cum_cap);
  auto work_at = [&](int pos) -> long long {
    const int g = (sort_n > 0) ? static_cast<int>(sort_keys[pos] & 0x1fffu) : pos;
    return static_cast<long long>(max(__ldcg(&plan.groups[g].n_blocks), 1) + kItemCost) * units;
  };
  long long sum = 0;
  for (int i = a; i < b; ++i) {
    const long long w = work_at(i);
    if (in_shared) cum_sh[i] = w;
    sum += w;
  }
  // inclusive scan of the per-thread sums: within each warp by shuffles,
  // then over the warp totals
  constexpr int kWarps = ROWS / 32;
  const int lane = t & 31, wid = t >> 5;
  long long incl = sum;
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) scan_sh[wid] = incl;
  __syncthreads();
  long long warp_base = 0, W = 0;
  for (int w = 0; w < kWarps; ++w) {
    const long long x = scan_sh[w];
    if (w < wid) warp_base += x;
    W += x;
  }
  // Each position counts max(blocks, 1) + kItemCost per head unit, so the
  // blocks alone are the total less the fixed costs; their mean per item
  // decides between equal shares and the counter.
  const long long blocks = W - static_cast<long long>(kItemCost) * units * P;
  const bool shares = (P > 0) && blocks >= static_cast<long long>(kSharesMinMeanBlocks) * P * units;
  const long long G = max(1LL, min(static_cast<long long>(grid), W / kMinCtaBlocks));
  if (t == 0) {
    plan.work[0] = W;
    plan.ctrl[5] = static_cast<int>(G);
    plan.ctrl[6] = shares ? 1 : 0;
  }
  if (!shares) return;  // the counter needs neither the totals nor the shares
  long long run = warp_base + incl - sum;
  for (int i = a; i < b; ++i) {
    const long long w = in_shared ? cum_sh[i] : work_at(i);
    plan.cum[i] = run;
    if (in_shared) cum_sh[i] = run;
    run += w;
  }
  if (t == 0) {
    plan.cum[P] = W;
    if (in_shared) cum_sh[P] = W;
  }
  __syncthreads();
  // the work item holding work index w: the last position whose running total
  // is <= w, then the head unit inside it
  auto cum_at = [&](int pos) -> long long { return in_shared ? cum_sh[pos] : __ldcg(plan.cum + pos); };
  auto item_at = [&](long long w) -> int {
    int lo = 0, hi = P - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum_at(mid) <= w) lo = mid; else hi = mid - 1;
    }
    const long long per_unit = (cum_at(lo + 1) - cum_at(lo)) / units;
    const long long u = per_unit > 0 ? (w - cum_at(lo)) / per_unit : 0;
    return lo * units + static_cast<int>(min(u, static_cast<long long>(units - 1)));
  };
  for (int c = t; c < G; c += ROWS) {
    const long long r0 = c * W / G, r1 = (c + 1) * W / G;
    plan.cta_first[c] = item_at(r0);
    plan.cta_last[c] = item_at(r1 - 1);
  }
}

constexpr int kRunsInShared = 4096;  // run starts a group block keeps in shared memory for the greedy walk

// The tiles of group g (tile indices ta and tb), found by the group's own
// block: the run starts (the set bits of the rows kernel's flag words) in
// row order, each thread taking a contiguous share of the words and a
// block-wide scan placing them, then the greedy cut described at the top of
// this file, walked by thread 0 only until the group's tiles are known
// (block 0 walks to the end and publishes the tile and group counts). Runs
// past kRunsInShared also go to the global run list; every block writes the
// same values there.
template <int ROWS>
static __device__ void find_group_tiles(long long n, long long max_tiles, int head_pairs, const FwdPlan& plan,
                                        int g, int* run_start, int* warp_total, int* sh, int2* tiles_out,
                                        int32_t* err) {
  constexpr int kWarps = ROWS / 32;
  const int t = threadIdx.x;
  const int lane = t & 31, wid = t >> 5;
  const long long words = (n + 31) / 32;
  const long long per = (words + ROWS - 1) / ROWS;
  const long long a = min(words, t * per);
  const long long b = min(words, a + per);
  int count = 0;
  for (long long w = a; w < b; ++w) count += __popc(plan.run_bits[w]);
  int incl = count;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_total[wid] = incl;
  __syncthreads();
  if (t == 0) {
    int acc = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int x = warp_total[w];
      warp_total[w] = acc;
      acc += x;
    }
    sh[0] = acc;  // runs
  }
  __syncthreads();
  const int runs = sh[0];
  int pos = warp_total[wid] + incl - count;
  for (long long w = a; w < b; ++w) {
    unsigned bits = plan.run_bits[w];
    while (bits) {
      const int row = static_cast<int>(w * 32) + __ffs(bits) - 1;
      bits &= bits - 1;
      if (pos < kRunsInShared) run_start[pos] = row;
      else plan.seg[pos] = row;
      ++pos;
    }
  }
  __syncthreads();  // the run starts above are visible to thread 0
  if (t == 0) {
    auto run_at = [&](int k) -> long long { return k < kRunsInShared ? run_start[k] : plan.seg[k]; };
    const long long ta = head_pairs ? g : 2LL * g;
    const long long tb = head_pairs ? g : 2LL * g + 1;
    int2 A = make_int2(0, 0), B = make_int2(0, 0);
    long long nt = 0;
    auto emit = [&](long long r0, int h) {
      if (nt == ta) A = make_int2(static_cast<int>(r0), h);
      if (nt == tb) B = make_int2(static_cast<int>(r0), h);
      ++nt;
    };
    long long cur0 = 0;
    int curh = 0;
    for (int k = 0; k < runs; ++k) {
      const long long st = run_at(k);
      const long long e = (k + 1 < runs) ? run_at(k + 1) : n;
      const long long len = e - st;
      const int head = static_cast<int>(len % kBlockM);
      const long long full = len / kBlockM;
      if (head > 0) {
        if (curh > 0 && curh + head <= kBlockM) {
          curh += head;  // packed with the short runs before it (rows are contiguous)
        } else {
          if (curh > 0) emit(cur0, curh);
          cur0 = st;
          curh = head;
        }
      }
      if (full > 0) {
        if (curh > 0) {
          emit(cur0, curh);
          curh = 0;
        }
        // the run's full tiles are nt .. nt + full - 1; only this group's
        // (ta, tb) are written
        for (long long x = (ta > nt ? ta : nt); x <= tb && x < nt + full; ++x) {
          const int2 tile = make_int2(static_cast<int>(st + head + kBlockM * (x - nt)), kBlockM);
          if (x == ta) A = tile;
          if (x == tb) B = tile;
        }
        nt += full;
      }
      if (g != 0 && nt > tb) break;  // this group's tiles are known
    }
    if (curh > 0 && (g == 0 || nt <= tb)) emit(cur0, curh);
    if (g == 0) {
      // The bound holds for every input (any two consecutive tiles hold more
      // than 128 rows); were it ever exceeded, the groups past it are lost
      // and that is reported.
      if (nt > max_tiles) {
        record_error(err, CPTHD_ERR_INDEX_RANGE, nt);
        nt = max_tiles;
      }
      plan.ctrl[0] = static_cast<int>(nt);
      plan.ctrl[1] = static_cast<int>(head_pairs ? nt : (nt + 1) / 2);
      plan.ctrl[2] = 0;
      plan.ctrl[3] = 0;
    }
    const bool real = ta < nt;
    if (tb >= nt) B = make_int2(A.x + A.y, 0);  // no second tile
    tiles_out[0] = A;
    tiles_out[1] = B;
    sh[1] = real ? 1 : 0;
  }
  __syncthreads();
}

template <int ROWS>
static __global__ void __launch_bounds__(ROWS) attn_fwd_group_kernel(long long n, long long max_tiles, int head_pairs,
                                                                     const int32_t* __restrict__ cup, FwdPlan plan,
                                                                     int sort_n, int units, int grid, int32_t* err) {
  __shared__ unsigned long long xbuf[2][ROWS];
  __shared__ int warp_sum[ROWS / 32];
  __shared__ int red_blocks[ROWS / 32];
  __shared__ int red_lo[ROWS / 32];
  __shared__ int red_hi[ROWS / 32];
  __shared__ __align__(8) int run_start[kRunsInShared];  // later the running totals (kRunsInShared / 2 of them)
  __shared__ long long scan_sh[ROWS / 32];
  __shared__ int2 tiles[2];
  __shared__ int sh[2];
  __shared__ int is_last;
  grid_dependency_wait();
  grid_dependents_launch();
  const int t = threadIdx.x;
  const int g = blockIdx.x;
  find_group_tiles<ROWS>(n, max_tiles, head_pairs, plan, g, run_start, warp_sum, sh, tiles, err);
  if (sh[1] == 0) {
    if (t == 0) {
      FwdGroup e;
      e.n_intervals = 0;
      e.n_blocks = 0;
      for (int x = 0; x < 2; ++x) { e.max_lo[x] = INT_MIN; e.min_hi[x] = INT_MAX; e.row0[x] = 0; e.h[x] = 0; }
      plan.groups[g] = e;
    }
  } else {
    group_intervals<ROWS>(cup, plan, g, tiles[0], tiles[1], xbuf, warp_sum, red_blocks, red_lo, red_hi);
  }
  // every block counts itself done; the last one writes the schedule
  __syncthreads();
  if (t == 0) {
    __threadfence();
    is_last = (atomicAdd(plan.ctrl + 4, 1) == static_cast<int>(gridDim.x) - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  schedule_last_block<ROWS>(plan, static_cast<int>(gridDim.x), sort_n, units, grid,
                            reinterpret_cast<long long*>(run_start), kRunsInShared / 2, scan_sh);
}

}  // namespace cpthd
