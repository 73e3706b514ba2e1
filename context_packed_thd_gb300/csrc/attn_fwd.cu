// Causal packed-THD attention forward on tcgen05 tensor cores (sm_103a).
//
// What is computed (TransformerEngine PR #3221, "Scope and constraints" and
// "What changed"): causal THD self-attention without a sliding window, one
// context-parallel rank's query slice against the full (all-gathered) K/V
// buffer, documents isolated through cu_seqlens / cu_seqlens_padded. Output
// O in bf16 and the natural-log LSE in fp32 ([Hq, t_local]).
//
// Kernel design. A CTA owns two 128-row query tiles A and B that read the
// same K/V blocks: one row tile under two query heads that share a KV head
// (GQA group sizes divisible by 2), or two consecutive row tiles under one
// head. Twelve warps in three warpgroups; warpgroup 0 gives registers to the
// softmax warpgroups (setmaxnreg: 96 vs 192 per thread; 96*128 + 192*256 stays
// within the 168 * 384 the launch allocates):
//  * warp 0      TMA producer: both Q tiles once per item, then K and V
//                128-key blocks into a two-stage shared-memory ring (128-byte
//                swizzle, the layout the UMMA shared-memory descriptors
//                read). A stage is refilled once tile B's score barrier
//                reports that the MMAs reading it are done. A Q tile is
//                replaced by the next item's as soon as the item's last
//                scores are done (the issuer commits to q_free after the
//                last S), so the next item's Q loads while this one ends.
//  * warp 1      one lane issues all tcgen05 MMAs: S_A(0), S_B(0), then per
//                block j and tile x = A, B: O_x += P_x(j) V_j in two halves
//                of 64 keys (the first as soon as the softmax has stored
//                P_x for those keys, so that it runs while the softmax
//                computes the other 64), then S_x(j+1).
//                Issuing tile A's batch before tile B's from one thread keeps
//                the two tiles half a period apart, so that each tile's
//                softmax runs while the tensor pipe works on the other tile.
//                The issue is fully unrolled with descriptors precomputed
//                (an issue loop with address arithmetic per MMA halves the
//                rate). Warp 1 also owns the 512-column TMEM allocation (S_A,
//                S_B, O_A, O_B). P_x(j) is written by the softmax into the
//                first 64 columns of S_x (bf16 pairs) and is read from TMEM
//                by the MMA. Because one thread's MMAs complete in issue
//                order, the commit that reports S_x(j+1) also reports that
//                O_x += P_x(j) V_j is done, so the softmax may then rescale
//                O_x and overwrite P_x without further waits.
//  * warp 2      data relay: per block j, waits until V_j has landed and
//                arrives on both tiles' first-half barriers (p_half), then
//                until K_{j+1} has landed and arrives on both tiles' P-ready
//                barriers (p_full), so that the issuer waits once per half
//                of P V.
//  * warp 3      idle.
//  * warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: each thread
//                owns one query row (its TMEM lane). It reads S with one
//                tcgen05.ld, masks by the row's key interval [document
//                start, own position] clipped to the end of the block's
//                interval (only on blocks the tile's bounds do not cover
//                fully), keeps the fp32 running max / sum in base 2, rescales
//                O in TMEM only when the max grows by more than 2^8 (exact
//                either way; before the block's first half of P is
//                released), and writes P back into TMEM, 64 keys at a time. At the end each
//                thread normalises its row of O and writes it (bf16, 16-byte
//                stores) straight to the output, and its LSE.
// Key blocks start at the group's interval starts (document starts), so
// documents the group does not see are never loaded or multiplied.
//
// Schedule. A work item is a group under one head unit; its work is the
// group's key blocks. The plan lays the items out in order (costliest groups
// first when there are more items than SMs). When items are short (fewer
// than kSharesMinMeanBlocks blocks on average) the CTAs (one per SM) take
// whole items from a counter in that order, each claiming its next item as
// the current one's last blocks are loaded: a greedy costliest-first
// schedule, under which the items running together start together and share
// their K/V blocks in L2. When items are long, a whole item per CTA leaves
// SMs idle at the end (256 items on 152 SMs finish in two item lengths, not
// 1.7), so each CTA instead takes an equal share of the total work (each
// item's blocks plus a fixed cost per item). An item that crosses a share
// boundary runs in pieces, one per
// CTA whose share it touches, each over its own key blocks. The online
// softmax of a piece is a partial result: its unnormalised O (fp32), the
// row maxima m and the sums l. Every piece but the last stores those to a
// slot of the workspace (one per share boundary and tile) and raises a flag;
// the last piece, which the CTA runs after the rest of its share, waits for
// the flags and combines all pieces in piece order (the standard rescaling
// by 2^(m_i - max m)), so that results do not depend on timing. That wait
// only ever points at CTAs of lower index whose pieces end or fill their
// shares, and those pieces wait for nothing, so the waits cannot form a
// cycle. Every wait is bounded; a wait that times out makes the CTA drain its
// copies and MMAs, free TMEM, record CPTHD_ERR_TIMEOUT and return.
#include <cuda_bf16.h>

#include "attn_common.cuh"
#include "attn_plan.cuh"

namespace cpthd {

using namespace sm100;

constexpr int kAttnThreads = 384;
constexpr int kRegsControl = 96;   // warpgroup 0: producer, MMA issuer, data relay
constexpr int kRegsSoftmax = 192;  // warpgroups 1 and 2
static_assert(kRegsControl * 128 + kRegsSoftmax * 256 <= 168 * kAttnThreads, "register split exceeds the launch");
constexpr int kStages = 2;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 256x
constexpr float kMaskShift = 1.2676506e30f;  // 2^100: subtracted from masked scores

template <int D>
struct AttnSmem {
  static constexpr int kChunk = kBlockM * 64 * 2;  // one 128-row x 64-column bf16 swizzle panel
  static constexpr int kChunks = D / 64;
  static constexpr int kQ = kChunks * kChunk;      // one Q tile
  static constexpr int kKV = kChunks * kChunk;     // one K or V block
  static constexpr int kQOff = 0;                  // Q_A, Q_B
  static constexpr int kKOff = 2 * kQ;
  static constexpr int kVOff = kKOff + kStages * kKV;
  // per softmax warp: its 32 rows x 64 output columns, staged for a TMA store
  static constexpr int kOutSlice = 32 * 128;
  static constexpr int kOutOff = kVOff + kStages * kKV;
  static constexpr int kBytes = kOutOff + 8 * kOutSlice;
  // request at least this much so that one CTA holds an SM (TMEM is taken whole)
  static constexpr int kLaunchBytes = (kBytes + 1024 > 120 * 1024) ? kBytes + 1024 : 120 * 1024;
};

struct AttnParams {
  const int32_t* row_lo;
  const int32_t* row_hi;
  const FwdGroup* groups;
  const int2* intervals;
  const int32_t* order;  // groups by decreasing cost; null: natural order
  int32_t* ctrl;         // plan counters: [1] groups, [3] CTAs finished, [5] CTAs with a share of the work
  const long long* cum;  // work before each position of the order (blocks x head units)
  const long long* work; // [0]: the total
  const int32_t* cta_first;  // first and last work item of each CTA's share
  const int32_t* cta_last;
  int32_t* flags;        // [2 * (boundary) + tile]: that piece's partial result is stored
  float* partial;        // the pieces' partial results, one slot per share boundary and tile
  float* lse;
  uint8_t* out;          // bf16 [t_local, Hq, D]: tiles of fewer than 128 rows are stored through it
  long long t_local;
  int Hq;
  int Hkv;
  int head_pairs;  // 1: tiles A/B = heads 2u, 2u+1 of one row tile; 0: two consecutive row tiles of one head
  int group_rows;  // interval slots per group: 128 with head pairs, 256 with tile pairs
  int max_groups;  // groups the plan can hold (guards a malformed count)
  int max_blocks;  // upper bound on blocks per group, guards malformed metadata
  float scale_log2;
  int32_t* err;
};

constexpr int kItemConsumers = 4;  // MMA issuer, data relay, one warp of each softmax warpgroup

#ifdef CPTHD_WAIT_TEST
// Test build only: which wait is made to run out. 1: the data relay withholds
// its arrivals for key block 1; 2: the pieces of cut items never raise their
// hand-off flags, so the merging pieces' flag waits run out.
__device__ int g_wait_test_mode = 1;
#endif

// A slot holds one tile's partial result: O as [D / 4][128 rows] float4 (so
// that a warp's 32 rows are 512 contiguous bytes), then m and l per row.
template <int D>
constexpr int slot_floats() { return D * kBlockM + 2 * kBlockM; }

// A work item as the producer hands it to the other roles: the group (a
// position of the plan's order), the head unit, and the piece of the group's
// key blocks this CTA runs: blocks [j0, j0 + nb) of the group's walk, piece
// s of S, the pieces' first share being `first`.
struct ItemDesc {
  int group;  // -1: no item left
  int unit;
  int j0;
  int nb;
  int s;
  int S;
  int first;
  int pad;
};

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const AttnParams p) {
  using L = AttnSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + L::kQOff;
  uint8_t* sK = smem + L::kKOff;
  uint8_t* sV = smem + L::kVOff;
  uint8_t* sOut = smem + L::kOutOff;

  __shared__ uint64_t q_full[2], q_free[2], k_full[kStages], v_full[kStages];
  // p_half[x]: P_x of the block's first 64 keys is in TMEM (and V_b has
  // landed); p_full[x]: all of P_x (and K_{b+1} has landed)
  __shared__ uint64_t s_full[2][kStages], p_half[2], p_full[2], o_final[2], o_free[2];
  __shared__ uint64_t item_full[2], item_empty[2], drain[1];
  __shared__ ItemDesc item_desc[2];
  __shared__ ItemDesc wg_desc[2];
  __shared__ int wg_abort[2];
  __shared__ int wg_flag_ok[2];
  __shared__ int wg_bounds[2][2];  // per tile: the bounds inside which a key block needs no mask
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Barriers and TMEM are set up before waiting on the kernel this launch
  // depends on: none of it touches global memory.
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int x = 0; x < 2; ++x) {
      mbar_init(&q_full[x], 1);
      mbar_init(&q_free[x], 1);   // the commit after the item's last S_x
      for (int s = 0; s < kStages; ++s) mbar_init(&s_full[x][s], 1);  // scores of tile x, key blocks of stage s
      mbar_init(&p_half[x], 5);   // four softmax warps and the data relay
      mbar_init(&p_full[x], 5);   // four softmax warps and the data relay
      mbar_init(&o_final[x], 1);
      mbar_init(&o_free[x], 4);   // the four softmax warps of tile x
      mbar_init(&item_full[x], 1);
      mbar_init(&item_empty[x], kItemConsumers);
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
    }
    mbar_init(&drain[0], 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  // columns: S_A [0,128), S_B [128,256), O_A [256, 256+D), O_B [256+D, 256+2D)

  grid_dependency_wait();
  grid_dependents_launch();
  const int units = p.head_pairs ? (p.Hq >> 1) : p.Hq;
  const int gqa = p.Hq / p.Hkv;
  // The k-th item of this CTA, as the producer published it (false: none
  // left, or the CTA aborted). Reading the slot and releasing it are one step.
  auto take_item = [&](int k, ItemDesc& d) -> bool {
    d.group = -1;
    if (!mbar_wait(&item_full[k & 1], (k >> 1) & 1, &abort_flag)) return false;
    d = item_desc[k & 1];
    mbar_arrive(&item_empty[k & 1]);
    return d.group >= 0;
  };

  if (warp < 4) {
   setmaxnreg_dec<kRegsControl>();
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Walks the CTA's share of the work, publishes each item (or piece) in a
    // two-slot ring, and loads its Q tiles and K/V blocks. Key blocks are
    // numbered across items (b), so the stage ring and its release through
    // tile B's score barrier run on without a break between items.
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int P = min(max(p.ctrl[1], 0), p.max_groups);
      const int G = min(max(p.ctrl[5], 0), static_cast<int>(gridDim.x));
      // equal shares, or whole items from the plan's counter (taken only
      // once the previous item's loads are issued, so that items go to the
      // CTAs about to be free and the costliest-first order balances the SMs
      // as a greedy schedule does)
      const bool shares = (p.ctrl[6] != 0);
      int next = static_cast<int>(blockIdx.x);
      const long long W = p.work[0];
      const int bx = static_cast<int>(blockIdx.x);
      const int f_share = p.cta_first[bx];
      const int l_share = p.cta_last[bx];
      const long long n_total = static_cast<long long>(P) * units;
      long long R0 = 0, R1 = 0;  // this CTA's share of the work
      int i_first = 0, n_it = 0;
      if (shares && bx < G && W > 0) {
        R0 = bx * W / G;
        R1 = (bx + 1) * W / G;
        if (R0 < R1 && f_share >= 0 && l_share >= f_share && l_share < n_total) {
          i_first = f_share;
          n_it = l_share - f_share + 1;
        }
      }
      // Item i spans the work [st, st + w) of the running totals: its key
      // blocks (at least one counted), then its fixed cost; nb_of: the
      // blocks counted for it.
      auto item_range = [&](int i, long long& st, long long& nb_of) {
        const int pos = i / units;
        const long long c0 = p.cum[pos], c1 = p.cum[pos + 1];
        const long long w = max(c1 - c0, 0LL) / units;
        st = c0 + (i - pos * units) * w;
        nb_of = max(w - kItemCost, 1LL);
      };
      // the share holding work index w
      auto share_of = [&](long long w) -> int { return static_cast<int>(((w + 1) * G - 1) / W); };
      // whether item i has a block in this share (a share may begin or end
      // inside an item's fixed cost)
      auto in_share = [&](int i) {
        long long st, nb_of;
        item_range(i, st, nb_of);
        return st < R1 && st + nb_of > R0;
      };
      // An item begun in the share before (this CTA finishes it and combines
      // its pieces) runs last, after the rest of the share.
      bool head_last = false;
      if (n_it > 1) {
        long long st, nb_of;
        item_range(i_first, st, nb_of);
        head_last = (st < R0) && (st + nb_of > R0);
      }
      int cand = head_last ? i_first + 1 : i_first;  // next candidate item
      const int i_end = i_first + n_it;
      int b = 0;       // key blocks of all items so far
      int issued = 0;  // K/V loads issued, in block order: 2b + 1 after K_b, 2b + 2 after V_b
      int nq[2] = {0, 0};
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (k >= 2 && !mbar_wait(&item_empty[k & 1], ((k >> 1) - 1) & 1, &abort_flag)) break;
        int i = -1;
        if (!shares) {
          if (next < n_total) i = next;
        } else {
          while (cand < i_end && i < 0) {
            if (in_share(cand)) i = cand;
            ++cand;
          }
          if (i < 0 && head_last) {
            i = i_first;
            head_last = false;
          }
        }
        ItemDesc d;
        d.group = -1;
        d.unit = d.j0 = d.nb = d.s = d.first = d.pad = 0;
        d.S = 1;
        if (i >= 0) {
          const int pos = i / units;
          d.unit = i - pos * units;
          d.group = min(max(p.order ? __ldg(p.order + pos) : pos, 0), p.max_groups - 1);
          const long long n = min(max(p.groups[d.group].n_blocks, 0), p.max_blocks);
          if (!shares) {
            d.nb = static_cast<int>(n);
          } else {
            long long st, nb_of;
            item_range(i, st, nb_of);
            const long long j0 = max(R0, st) - st, j1 = min(R1, st + nb_of) - st;
            d.j0 = static_cast<int>(j0);
            d.nb = static_cast<int>(max(0LL, min(j1, n) - j0));
            d.first = share_of(st);
            d.S = share_of(st + nb_of - 1) - d.first + 1;
            d.s = bx - d.first;
          }
        }
        item_desc[k & 1] = d;
        mbar_arrive(&item_full[k & 1]);
        if (d.group < 0) break;
        if (d.nb == 0) {  // no key block here: nothing to load
          if (!shares) next = static_cast<int>(gridDim.x) + atomicAdd(p.ctrl + 2, 1);
          continue;
        }
        const int head0 = p.head_pairs ? 2 * d.unit : d.unit;
        const int kvh = head0 / gqa;
        const FwdGroup* gi = p.groups + d.group;
        const int n_blocks = d.nb;
        const int2* group_iv = p.intervals + static_cast<long long>(d.group) * p.group_rows;
        const int n_iv = min(max(gi->n_intervals, 0), p.group_rows);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          // the previous item's last S_x has read tile x's buffer
          if (nq[x] > 0 && !mbar_wait(&q_free[x], (nq[x] - 1) & 1, &abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&q_full[x], L::kQ);
          const int qh = p.head_pairs ? head0 + x : head0;
          const int qrow = gi->row0[x];
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sQ + x * L::kQ + c * L::kChunk, &tm_q, &q_full[x], c * 64, qh, qrow);
          ++nq[x];
        }
        if (!ok) break;
        BlockCursor cur;
        cur.init(group_iv, n_iv);
        cur.skip(d.j0);
        for (int i = 0; i < n_blocks; ++i, ++b) {
          const int st = b & 1;
          // Stages are released through tile B's score barriers, one per
          // stage: the commit after S_B(c) goes to s_full[1][c & 1] and
          // reports every MMA issued up to it (one thread issues them all,
          // tile B last). So S_B(b - 2) done frees K_{b-2} (same stage) and
          // S_B(b - 1) done frees V_{b-2} (P V of block b - 2 is issued before
          // S(b - 1)). The phase after the one waited for is S_B(b) for K and
          // S_B(b + 1) for V, which need K_b and K_{b+1}: loads this thread
          // has not issued yet. So no barrier is ever two phases past a wait,
          // however long the producer stalls between items, and the parity
          // is unambiguous.
          if (b >= kStages && !mbar_wait(&s_full[1][st], ((b - 2) >> 1) & 1, &abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&k_full[st], L::kKV);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sK + st * L::kKV + c * L::kChunk, &tm_k, &k_full[st], c * 64, kvh, cur.start);
          issued = 2 * b + 1;
          if (b >= kStages && !mbar_wait(&s_full[1][st ^ 1], ((b - 1) >> 1) & 1, &abort_flag)) { ok = false; break; }
          mbar_arrive_expect_tx(&v_full[st], L::kKV);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sV + st * L::kKV + c * L::kChunk, &tm_v, &v_full[st], c * 64, kvh, cur.start);
          issued = 2 * b + 2;
          cur.next();
        }
        if (!shares) next = static_cast<int>(gridDim.x) + atomicAdd(p.ctrl + 2, 1);
      }
      if (abort_flag) {
        // let every copy still in flight land before the CTA exits
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (nq[x] > 0) mbar_wait_drain(&q_full[x], (nq[x] - 1) & 1);
        for (int y = (issued > 4 ? issued - 4 : 0); y < issued; ++y) {
          const int i = y >> 1, st = i & 1;
          mbar_wait_drain((y & 1) ? &v_full[st] : &k_full[st], (i >> 1) & 1);
        }
      }
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues both tiles' MMAs, tile A's batch before tile B's, so
    // that tile B's scores arrive a batch after tile A's and one tile's
    // softmax runs under the other tile's MMAs (two issuing threads started
    // together interleave on the tensor pipe and fall into lockstep). An
    // item's first scores are issued as soon as its Q and first K block are
    // in, while the softmax warps may still be storing the previous item; its
    // first P V waits until they have read that item's O.
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
      constexpr uint32_t kIdescO = idesc_bf16_f32(kBlockM, D, 0, 1);
      // A descriptor's low word holds the start address (>> 4) and the
      // leading-byte offset; its high word (stride offset, version, swizzle)
      // is the same for every block of one operand. Addresses stay below
      // 256 KB, so adding an offset to the low word never carries.
      const uint64_t dq = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv = smem_desc_sw128(smem_u32(sV), L::kChunk, 1024);
      const uint32_t q_lo = static_cast<uint32_t>(dq), q_hi = static_cast<uint32_t>(dq >> 32);
      const uint32_t k_lo = static_cast<uint32_t>(dk), k_hi = static_cast<uint32_t>(dk >> 32);
      const uint32_t v_lo = static_cast<uint32_t>(dv), v_hi = static_cast<uint32_t>(dv >> 32);
      auto issue_s = [&](int j, int x) {  // S_x = Q_x K_j^T
        const uint32_t t_s = tmem + x * kBlockN;
        const uint32_t qb = q_lo + ((x * L::kQ) >> 4);
        const uint32_t kb = k_lo + (((j & 1) * L::kKV) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kChunk + (kk & 3) * 32) >> 4;
          umma_ss_w(t_s, qb + off, q_hi, kb + off, k_hi, kIdescS, kk > 0);
        }
      };
      // O_x (+)= P_x V_j over keys [64 h, 64 h + 64) of the block, P_x read from TMEM
      auto issue_pv = [&](int j, int x, int h, uint32_t acc0) {
        const uint32_t t_s = tmem + x * kBlockN;
        const uint32_t t_o = tmem + 256 + x * D;
        const uint32_t vb = v_lo + (((j & 1) * L::kKV) >> 4);
#pragma unroll
        for (int kk = 4 * h; kk < 4 * h + kBlockN / 32; ++kk)
          umma_ts_w(t_o, t_s + kk * 8, vb + ((kk * 16 * 128) >> 4), v_hi, kIdescO, kk > 0 ? 1u : acc0);
      };
      int b = 0, nq = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        ItemDesc d;
        if (!take_item(k, d)) break;
        const int n_blocks = d.nb;
        int finals = 0;
        if (n_blocks > 0) {
          ok = mbar_wait(&q_full[0], nq & 1, &abort_flag) && mbar_wait(&q_full[1], nq & 1, &abort_flag) &&
               mbar_wait(&k_full[b & 1], (b >> 1) & 1, &abort_flag);
          ++nq;
          if (ok) {
            tc_fence_after_sync();
            issue_s(b, 0);
            umma_commit(&s_full[0][b & 1]);
            if (n_blocks == 1) umma_commit(&q_free[0]);  // the item's last read of Q_A
            issue_s(b, 1);
            umma_commit(&s_full[1][b & 1]);
            if (n_blocks == 1) umma_commit(&q_free[1]);
          }
          for (int j = 0; ok && j < n_blocks; ++j) {
            const int bb = b + j;
            const bool more = (j + 1 < n_blocks);
#pragma unroll
            for (int x = 0; x < 2; ++x) {
              // the previous item's O_x has been read by its epilogue
              if (j == 0 && k > 0 && !mbar_wait(&o_free[x], (k - 1) & 1, &abort_flag)) { ok = false; break; }
              // P_x(bb) over the first 64 keys is ready (and, through the
              // relay's arrival, V_bb has landed): the first half of P V
              // runs while the softmax warps finish the other 64 keys
              if (!mbar_wait(&p_half[x], bb & 1, &abort_flag)) { ok = false; break; }
              tc_fence_after_sync();
              issue_pv(bb, x, 0, j > 0 ? 1u : 0u);
              // all of P_x(bb) is ready, and K_{bb+1} has landed
              if (!mbar_wait(&p_full[x], bb & 1, &abort_flag)) { ok = false; break; }
              tc_fence_after_sync();
              issue_pv(bb, x, 1, 1u);
              if (more) {
                issue_s(bb + 1, x);
                umma_commit(&s_full[x][(bb + 1) & 1]);  // also reports O_x += P_x(bb) V_bb done
                // the item's last scores: once they are done, Q_x may be
                // replaced by the next item's while this one finishes
                if (j + 2 == n_blocks) umma_commit(&q_free[x]);
              } else {
                umma_commit(&o_final[x]);  // tile x's epilogue need not wait for the other tile
                finals |= 1 << x;
              }
            }
          }
          b += n_blocks;
        } else if (k > 0) {
          // an item without keys (only pad rows): no MMA, but its epilogue
          // must not be signalled before the previous one has read O
          ok = mbar_wait(&o_free[0], (k - 1) & 1, &abort_flag) && mbar_wait(&o_free[1], (k - 1) & 1, &abort_flag);
        }
        // a tile whose final commit did not happen (no key block, or an abort)
        if (!(finals & 1)) umma_commit(&o_final[0]);
        if (!(finals & 2)) umma_commit(&o_final[1]);
      }
      umma_commit(&drain[0]);
      mbar_wait_drain(&drain[0], 0);
    }
   } else if (warp == 2) {
    // ------------------------------------------------------------ data relay
    // Waits, per key block, until V_b has landed and arrives on both tiles'
    // p_half, then until (when the item has a next block) K_{b+1} has landed
    // and arrives on both tiles' p_full, so that the MMA issuer (the busiest
    // thread of the CTA) waits on one barrier per half of P V. Before
    // arriving for block b it waits for both p_full phases of block b - 1 to
    // complete (which implies the p_half phases: the softmax warps arrive on
    // p_half first), so that an early arrival never counts toward the
    // previous phase.
    if (lane == 0) {
      int b = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        ItemDesc d;
        if (!take_item(k, d)) break;
        const int n_blocks = d.nb;
        for (int j = 0; j < n_blocks; ++j) {
          const int bb = b + j;
          if (bb > 0 && !(mbar_wait(&p_full[0], (bb - 1) & 1, &abort_flag) &&
                          mbar_wait(&p_full[1], (bb - 1) & 1, &abort_flag))) { ok = false; break; }
          if (!mbar_wait(&v_full[bb & 1], (bb >> 1) & 1, &abort_flag)) { ok = false; break; }
#ifdef CPTHD_WAIT_TEST
          // Test build only: key block 1's arrivals are withheld, so the waits
          // for P(1) can never complete and must run out into the abort path.
          if (g_wait_test_mode == 1 && bb == 1) continue;
#endif
          mbar_arrive(&p_half[0]);
          mbar_arrive(&p_half[1]);
          if (j + 1 < n_blocks && !mbar_wait(&k_full[(bb + 1) & 1], ((bb + 1) >> 1) & 1, &abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive(&p_full[0]);
          mbar_arrive(&p_full[1]);
        }
        b += n_blocks;
      }
    }
   }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) >> 2;  // tile of this warpgroup
    const int quarter = warp & 3;   // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;
    const int bar_id = 1 + x;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + x * kBlockN;
    const uint32_t t_o = tmem + lane_off + 256 + x * D;
    const float sl2 = p.scale_log2;
    int b = 0;
    for (int k = 0;; ++k) {
      // One warp takes the item for the warpgroup, so that its four warps
      // always agree on the item and on stopping.
      if (quarter == 0 && lane == 0) {
        ItemDesc d;
        take_item(k, d);
        wg_desc[x] = d;
        wg_abort[x] = 0;
        // kept in shared memory: the block loop has no registers to spare
        if (d.group >= 0) {
          wg_bounds[x][0] = p.groups[d.group].max_lo[x];
          wg_bounds[x][1] = p.groups[d.group].min_hi[x];
        }
      }
      named_bar_sync(bar_id, 128);
      int n_blocks, lo = 1, hi = 0;
      BlockCursor cur;
      {
        const int group = wg_desc[x].group;
        if (group < 0) break;
        const FwdGroup* gi = p.groups + group;
        n_blocks = wg_desc[x].nb;
        cur.init(p.intervals + static_cast<long long>(group) * p.group_rows,
                 min(max(gi->n_intervals, 0), p.group_rows));
        cur.skip(wg_desc[x].j0);
        if (r < min(max(gi->h[x], 0), kBlockM)) {
          lo = p.row_lo[static_cast<long long>(gi->row0[x]) + r];
          hi = p.row_hi[static_cast<long long>(gi->row0[x]) + r];
        }
      }
      float m = -INFINITY;  // running max of scale*log2(e)*s
      float l = 0.f;
      bool ok = true;
      for (int j = 0; j < n_blocks; ++j) {
        const int bb = b + j;
        // a block never reaches past its interval's end: the next interval may
        // start inside it, and its keys must be counted there only
        const int kstart = cur.start;
        const int kend = cur.end;
        cur.next();
        if (!warp_wait(&s_full[x][bb & 1], (bb >> 1) & 1, &abort_flag)) { ok = false; break; }
        tc_fence_after_sync();
        uint32_t sr[kBlockN];
        tmem_ld128(t_s, sr);
        tmem_ld_wait128(sr);
        const bool full = (kstart >= wg_bounds[x][0]) && (kstart + kBlockN - 1 <= min(wg_bounds[x][1], kend));
        // 16-column groups of this block that no row of the warp may use
        uint32_t dead_groups = 0;
        bool row_dead = false;  // this row has no key in this block
        if (!full) {
          // allowed columns of this row: [c_lo, c_hi] (empty when c_lo > c_hi)
          const int c_lo = min(max(lo - kstart, 0), kBlockN);
          int c_hi = max(min(min(hi, kend) - kstart, kBlockN - 1), -1);
          // Blocks start at document starts, so with monotone offsets a row
          // either starts at or before the block (c_lo = 0) or has no key in
          // it (c_lo > c_hi). Anything else can only come from offsets the
          // plan has already reported; such a row uses no key of the block,
          // so it never reaches a key before its own start.
          if (c_lo > 0 && c_lo <= c_hi) record_error(p.err, CPTHD_ERR_BAD_OFFSETS, kstart);
          row_dead = (c_lo > 0) || (c_hi < 0);
          if (row_dead) c_hi = -1;
          // bounds over the warp's live rows (a warp whose rows straddle a
          // document boundary still skips the mask where its live rows may use
          // every column); dead rows are zeroed below whatever their scores
          const int w_min = __reduce_min_sync(0xffffffffu, row_dead ? kBlockN - 1 : c_hi);
          const int w_max = __reduce_max_sync(0xffffffffu, c_hi);
          dead_groups = (w_max < 0) ? 0xffu : ((0xffu << ((w_max >> 4) + 1)) & 0xffu);
          if (w_max >= 0) {
            // The mask runs on the FMA pipe: u = saturate(c - c_hi) is 1
            // exactly for columns past the row's last key (c is an integer),
            // and s - u * 2^100 pushes them far below any real score. A row
            // left with no key in this block is caught after the max (below),
            // so no two huge values are ever subtracted from each other.
            // Groups every live row may use are left alone.
            const float f_hi = static_cast<float>(c_hi);
#pragma unroll
            for (int g = 0; g < kBlockN / 16; ++g) {
              if (16 * g + 15 > w_min) {
#pragma unroll
                for (int c = 16 * g; c < 16 * g + 16; c += 2) {
                  float s0, s1;
                  fma2(s0, s1, __saturatef(static_cast<float>(c) - f_hi),
                       __saturatef(static_cast<float>(c + 1) - f_hi), -kMaskShift, __uint_as_float(sr[c]),
                       __uint_as_float(sr[c + 1]));
                  sr[c] = __float_as_uint(s0);
                  sr[c + 1] = __float_as_uint(s1);
                }
              }
            }
          }
        }
        // row max of the raw scores: four chains of three-input max
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kBlockN; c += 8) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            mx[u] = max3f(mx[u], __uint_as_float(sr[c + 2 * u]), __uint_as_float(sr[c + 2 * u + 1]));
        }
        float mx_row = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3]));
        // no key of this row in this block
        if (row_dead || mx_row < -0.5f * kMaskShift) mx_row = -INFINITY;
        const float m_new = fmaxf(m, mx_row * sl2);
        const bool grow_o = (m != -INFINITY) && (m_new > m + kRescaleThreshold);
        float alpha = 1.f;
        if (m == -INFINITY) {
          m = m_new;  // nothing accumulated yet: O and l are exactly zero
        } else if (grow_o) {
          alpha = ex2(m - m_new);
          l *= alpha;
          m = m_new;
        }
        // a dead row subtracts 2^100 from every exponent, so all its p are 0
        const float mref = row_dead ? kMaskShift : ((m == -INFINITY) ? 0.f : m);
        // p = 2^(scale*log2(e)*s - m): one packed FMA per pair, ex2 per element,
        // row sum in two packed accumulators. A 64-column half no row may use
        // stores zeros without exponentials; elsewhere masked columns give 0.
        // Each half is released to the MMA issuer as soon as it is stored, so
        // that P V over the first 64 keys runs during the second half.
        float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t pk[32];
          if (((dead_groups >> (4 * h2)) & 0xfu) == 0xfu) {
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = 0u;
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              float a0, a1;
              fma2(a0, a1, __uint_as_float(sr[64 * h2 + 2 * c]), __uint_as_float(sr[64 * h2 + 2 * c + 1]), sl2,
                   -mref);
              const float e0 = ex2(a0);
              const float e1 = ex2(a1);
              add2(rs[2 * (c & 1)], rs[2 * (c & 1) + 1], e0, e1);
              pk[c] = pack_bf16x2(e0, e1);
            }
          }
          tmem_st32(t_s + 32 * h2, pk);
          if (h2 == 0 && __any_sync(0xffffffffu, grow_o)) {
            // O_x holds P_x V up to the previous block (complete before S_x(bb)
            // was reported) and nothing newer: rescale it before this block's
            // first half of P V, which p_half releases (here, once the first
            // half's scores no longer hold registers)
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t orr[32];
              tmem_ld32(t_o + c * 32, orr);
              tmem_ld_wait(orr);
#pragma unroll
              for (int q = 0; q < 32; ++q) orr[q] = __float_as_uint(__uint_as_float(orr[q]) * alpha);
              tmem_st32(t_o + c * 32, orr);
            }
          }
          tmem_st_wait();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(h2 == 0 ? &p_half[x] : &p_full[x]);
        }
        l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      }
      b += n_blocks;
      // The tile's rows and head are read again here rather than kept
      // through the block loop, whose registers the scores fill.
      const int d_s = wg_desc[x].s, d_S = wg_desc[x].S;
      const FwdGroup* gi = p.groups + wg_desc[x].group;
      const int qh = p.head_pairs ? 2 * wg_desc[x].unit + x : wg_desc[x].unit;
      const int row0 = gi->row0[x];
      const int h = min(max(gi->h[x], 0), kBlockM);
      const bool in_tile = r < h;
      const long long grow = static_cast<long long>(row0) + r;
      const bool valid = in_tile && (lo <= hi);
      // a piece of an item cut at share boundaries: every piece but the last
      // publishes its partial result, the last combines them all
      const bool split = d_S > 1;
      const bool publisher = split && d_s != d_S - 1;
      const bool combiner = split && !publisher;
      constexpr int kSlot = slot_floats<D>();
      // piece t (< S - 1) of this tile: the slot of the boundary it ends at,
      // and its flag
      const int slot0 = 2 * wg_desc[x].first + x;
      float* const slot_base = p.partial + static_cast<long long>(slot0) * kSlot;
      auto slot_of = [slot_base](int t) { return slot_base + static_cast<long long>(2 * t) * kSlot; };
      // ---------------------------------------------------------- epilogue
      // Once o_final[x] reports the last P V done, each thread reads its row
      // of O from TMEM, merges or publishes pieces of a cut item, and writes
      // O / l in bf16 straight to the output (no staging: the Q buffer is
      // already the next item's). Every warp reaches the barriers of every
      // item it took; an aborted one only marks the tile.
      if (ok) ok = warp_wait(&o_final[x], k & 1, &abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after_sync();
      if (publisher) {
        // O (unnormalised), m and l of this row into the piece's slot; the
        // flag goes up after the warpgroup's barrier below
        float* so = slot_of(d_s);
        if (ok) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t rr[32];
            if (n_blocks > 0) {
              tmem_ld32(t_o + c * 32, rr);
              tmem_ld_wait(rr);
            } else {
#pragma unroll
              for (int q = 0; q < 32; ++q) rr[q] = 0u;
            }
            float4* dst = reinterpret_cast<float4*>(so) + (c * 8) * kBlockM + r;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q * kBlockM] = make_float4(__uint_as_float(rr[4 * q]), __uint_as_float(rr[4 * q + 1]),
                                             __uint_as_float(rr[4 * q + 2]), __uint_as_float(rr[4 * q + 3]));
          }
          so[D * kBlockM + r] = (n_blocks > 0) ? m : -INFINITY;
          so[D * kBlockM + kBlockM + r] = (n_blocks > 0) ? l : 0.f;
        }
        __threadfence();
      }
      if (combiner) {
        // every other piece of this tile has published (their CTAs have lower
        // indices and their pieces wait for nothing)
        bool got = ok && n_blocks > 0;
        if (ok && n_blocks == 0) record_error(p.err, CPTHD_ERR_INDEX_RANGE, wg_desc[x].group);
        if (got && r == 0)
          for (int t = 0; t < d_S - 1 && got; ++t) got = flag_wait(p.flags + slot0 + 2 * t, &abort_flag);
        if (r == 0) wg_flag_ok[x] = got ? 1 : 0;
        named_bar_sync(bar_id, 128);
        ok = ok && (wg_flag_ok[x] != 0);
        fence_acq_rel_gpu();
        if (ok) {
          // the combined maximum and sum, pieces in order (own piece last)
          float ms = m;
          for (int t = 0; t < d_S - 1; ++t) ms = fmaxf(ms, __ldcg(slot_of(t) + D * kBlockM + r));
          float ls = 0.f;
          for (int t = 0; t < d_S - 1; ++t) {
            const float mt = __ldcg(slot_of(t) + D * kBlockM + r);
            if (mt != -INFINITY) ls += ex2(mt - ms) * __ldcg(slot_of(t) + D * kBlockM + kBlockM + r);
          }
          const float w_own = (m != -INFINITY) ? ex2(m - ms) : 0.f;
          ls += w_own * l;
          m = ms;
          l = ls;
          // O of all pieces, in piece order (own piece last), back into TMEM
          for (int c = 0; c < D / 32; ++c) {
            float acc[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) acc[q] = 0.f;
            for (int t = 0; t < d_S - 1; ++t) {
              const float* so = slot_of(t);
              const float mt = __ldcg(so + D * kBlockM + r);
              const float wt = (mt != -INFINITY) ? ex2(mt - m) : 0.f;
              const float4* src = reinterpret_cast<const float4*>(so) + (c * 8) * kBlockM + r;
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 v = __ldcg(src + q * kBlockM);
                acc[4 * q] += wt * v.x;
                acc[4 * q + 1] += wt * v.y;
                acc[4 * q + 2] += wt * v.z;
                acc[4 * q + 3] += wt * v.w;
              }
            }
            uint32_t rr[32];
            tmem_ld32(t_o + c * 32, rr);
            tmem_ld_wait(rr);
#pragma unroll
            for (int q = 0; q < 32; ++q) rr[q] = __float_as_uint(acc[q] + w_own * __uint_as_float(rr[q]));
            tmem_st32(t_o + c * 32, rr);
          }
          tmem_st_wait();
        }
      }
      // O / l in bf16, 64 columns at a time: each warp packs its 32 rows into
      // its slice of shared memory (128-byte swizzle) and one lane stores the
      // slice with TMA; a warp whose rows cross the end of a short tile
      // stores its rows directly instead (a TMA box would write the next
      // tile's rows). O_x is released to the next item's first P V right
      // after the warp's last TMEM read, before the stores.
      bool freed = false;
      if (ok && n_blocks > 0 && !publisher) {
        const float inv = (valid && l > 0.f) ? 1.f / l : 0.f;
        const int wrow = quarter * 32;  // the warp's first row in the tile
        const bool tma_rows = (wrow + 32 <= h);
        uint8_t* slice = sOut + (warp - 4) * L::kOutSlice;
        uint4* dst = reinterpret_cast<uint4*>(p.out + (grow * p.Hq + qh) * static_cast<long long>(D) * 2);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          uint32_t ob[32];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t rr[32];
            tmem_ld32(t_o + (2 * hh + cc) * 32, rr);
            tmem_ld_wait(rr);
#pragma unroll
            for (int q = 0; q < 16; ++q)
              ob[16 * cc + q] =
                  valid ? pack_bf16x2(__uint_as_float(rr[2 * q]) * inv, __uint_as_float(rr[2 * q + 1]) * inv) : 0u;
          }
          if (hh == D / 64 - 1) {
            // O_x is read: the next item's first P V may overwrite it
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_free[x]);
            freed = true;
          }
          if (tma_rows) {
            // the slice's previous store (this item's last round, or the
            // previous item's) has been read
            if (lane == 0) bulk_wait_group_read_all();
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(slice + lane * 128 + ((u ^ (lane & 7)) << 4)) =
                  make_uint4(ob[4 * u], ob[4 * u + 1], ob[4 * u + 2], ob[4 * u + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tm_o, slice, hh * 64, qh, row0 + wrow);
              bulk_commit_group();
            }
          } else if (in_tile) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              dst[8 * hh + u] = make_uint4(ob[4 * u], ob[4 * u + 1], ob[4 * u + 2], ob[4 * u + 3]);
          }
        }
      }
      if (!freed) {
        // O_x is read: the next item's first P V may overwrite it
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_free[x]);
      }
      if (ok && in_tile && !publisher) {
        p.lse[static_cast<long long>(qh) * p.t_local + grow] =
            (valid && l > 0.f) ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        if (n_blocks == 0 && !split) {
          // no key in the whole group (only pad rows): zeros, stored directly
          uint4* dst = reinterpret_cast<uint4*>(p.out + (grow * p.Hq + qh) * static_cast<long long>(D) * 2);
#pragma unroll
          for (int u = 0; u < D / 8; ++u) dst[u] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (!ok) wg_abort[x] = 1;
      named_bar_sync(bar_id, 128);
      // read once, between the two barriers: the warpgroup's first warp
      // clears the flag for the next item only after the second one
      const bool stop = (wg_abort[x] != 0);
      // every thread's partial is written and fenced: raise the piece's flag
#ifdef CPTHD_WAIT_TEST
      const bool raise_flag = (g_wait_test_mode != 2);  // test build: mode 2 withholds the flags
#else
      const bool raise_flag = true;
#endif
      if (publisher && !stop && r == 0 && raise_flag) st_release_gpu(p.flags + slot0 + 2 * d_s, 1);
      named_bar_sync(bar_id, 128);
      if (stop) break;
    }
    if (lane == 0) bulk_wait_group_all();  // this warp's last output store has landed
  }

  tc_fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (abort_flag) record_error(p.err, CPTHD_ERR_TIMEOUT, blockIdx.x);
    // The last CTA to finish returns the work counters to zero for the next
    // launch on this plan.
    __threadfence();
    if (atomicAdd(p.ctrl + 3, 1) == static_cast<int>(gridDim.x) - 1) {
      // every CTA is done with the hand-off flags: lower them for the next launch
      if (p.ctrl[6] != 0)
        for (int f = 0; f < 2 * static_cast<int>(gridDim.x); ++f) p.flags[f] = 0;
      atomicExch(p.ctrl + 2, 0);
      atomicExch(p.ctrl + 3, 0);
    }
  }
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// The attention grid, which the plan's schedule is made for: one CTA per SM,
// at most kMaxCtas.
static int attn_grid() {
  const int sms = sm_count();
  return sms < kMaxCtas ? sms : kMaxCtas;
}

template <int D>
static int launch_attn(const void* q, const void* k, const void* v, long long t_local, long long T, int Hq, int Hkv,
                       float scale_log2, const FwdPlan& plan, const FwdShape& shape, bool ordered, float* partial,
                       void* out, float* lse, int32_t* err, cudaStream_t s) {
  EncodeTiledFn enc = get_encode_tiled();
  if (enc == nullptr) return CPTHD_ERR_CUDA;
  CUtensorMap mq, mk, mv, mo;
  if (!make_rows_heads_map(enc, &mq, q, t_local, Hq, D) || !make_rows_heads_map(enc, &mk, k, T, Hkv, D) ||
      !make_rows_heads_map(enc, &mv, v, T, Hkv, D) || !make_rows_heads_map(enc, &mo, out, t_local, Hq, D, 32))
    return CPTHD_ERR_UNSUPPORTED;
  AttnParams p;
  p.row_lo = plan.row_lo;
  p.row_hi = plan.row_hi;
  p.groups = plan.groups;
  p.intervals = plan.intervals;
  p.order = ordered ? plan.order : nullptr;
  p.ctrl = plan.ctrl;
  p.cum = plan.cum;
  p.work = plan.work;
  p.cta_first = plan.cta_first;
  p.cta_last = plan.cta_last;
  p.flags = plan.flags;
  p.partial = partial;
  p.lse = lse;
  p.out = static_cast<uint8_t*>(out);
  p.t_local = t_local;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.head_pairs = shape.head_pairs;
  p.group_rows = shape.group_rows;
  p.max_groups = static_cast<int>(shape.max_groups);
  p.max_blocks = static_cast<int>((T + kBlockN - 1) / kBlockN + shape.group_rows);
  p.scale_log2 = scale_log2;
  p.err = err;
  const int smem = AttnSmem<D>::kLaunchBytes;
  CPTHD_TRY_CUDA(cudaFuncSetAttribute(attn_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  const long long items = shape.max_groups * (shape.head_pairs ? Hq / 2 : Hq);
  if (items > INT32_MAX) return CPTHD_ERR_UNSUPPORTED;
  // one CTA per SM (one fits: shared memory and TMEM are taken whole), each
  // running its share of the plan's work; the plan was made for this grid
  const int grid = attn_grid();
  if (grid < 1) return CPTHD_ERR_CUDA;
  CPTHD_TRY_CUDA(launch_pdl(attn_fwd_tc_kernel<D>, dim3(static_cast<unsigned>(grid)), dim3(kAttnThreads), smem, s,
                            mq, mk, mv, mo, p));
  return CPTHD_OK;
}

// Whether the plan orders the groups (costliest first): when there are more
// work items than SMs and the groups fit the sort.
static bool plan_ordered(const FwdShape& shape, int Hq) {
  const long long items = shape.max_groups * (shape.head_pairs ? Hq / 2 : Hq);
  return items > sm_count() && shape.max_groups <= kMaxSortGroups;
}

// The partial results of cut items: one slot per share boundary and tile,
// after the plan in the workspace.
static size_t split_bytes(int d) {
  return align256(sizeof(float) * static_cast<size_t>(2 * (kMaxCtas - 1)) * (d == 64 ? slot_floats<64>()
                                                                                       : slot_floats<128>()));
}

}  // namespace cpthd

extern "C" int thd_causal_attn_workspace_size(int64_t t_local, int Hq, int Hkv, int d, size_t* bytes_host) {
  if (bytes_host == nullptr || t_local < 0 || Hq < 1 || Hkv < 1) return CPTHD_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return CPTHD_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return CPTHD_ERR_UNSUPPORTED;
  *bytes_host = cpthd::fwd_plan_bytes(cpthd::fwd_shape(t_local, Hq, Hkv)) + cpthd::split_bytes(d);
  return CPTHD_OK;
}

namespace cpthd {

// d = 0: the plan alone (thd_causal_attn_plan, which does not know d)
static int check_workspace(int64_t t_local, int Hq, int Hkv, int d, const void* workspace_dev,
                           size_t workspace_bytes) {
  const size_t need = fwd_plan_bytes(fwd_shape(t_local, Hq, Hkv)) + (d > 0 ? split_bytes(d) : 0);
  if (workspace_dev == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace_dev) & 255))
    return CPTHD_ERR_WORKSPACE;
  return CPTHD_OK;
}

// The plan of the slice (rows, then the groups: their tiles, intervals and,
// past one wave of work items, their order) into the workspace; shape and
// workspace already checked.
static int launch_plan(const IndexGen& slots, long long t_local, long long T, const int32_t* cu,
                       const int32_t* cup, int num_docs, int Hq, int Hkv, void* workspace, int32_t* err,
                       cudaStream_t s) {
  const FwdShape shape = fwd_shape(t_local, Hq, Hkv);
  FwdPlan plan = carve_fwd_plan(workspace, shape);
  const int sms = sm_count();
  if (sms < 1) return CPTHD_ERR_CUDA;
  if (shape.max_groups > INT32_MAX / 2) return CPTHD_ERR_UNSUPPORTED;
  CPTHD_TRY_CUDA(launch_pdl(attn_rows_kernel, dim3(static_cast<unsigned>((t_local + 255) / 256)), dim3(256), 0, s,
                            slots, t_local, cu, cup, num_docs, T, plan, err));
  // The costliest groups go first when there are more work items than SMs:
  // the group kernel's last block sorts them (a power-of-two key buffer in
  // dynamic shared memory); plans too large for the sort keep index order.
  int sort_n = 0;
  if (plan_ordered(shape, Hq) && shape.max_groups <= kMaxSortGroups) {
    sort_n = 1;
    while (sort_n < shape.max_groups) sort_n <<= 1;
  }
  const size_t sort_bytes = sizeof(unsigned) * static_cast<size_t>(sort_n);
  const int units = shape.head_pairs ? Hq / 2 : Hq;
  const int grid = attn_grid();
  if (grid < 1) return CPTHD_ERR_CUDA;
  if (shape.head_pairs) {
    CPTHD_TRY_CUDA(launch_pdl(attn_fwd_group_kernel<kBlockM>, dim3(static_cast<unsigned>(shape.max_groups)),
                              dim3(kBlockM), sort_bytes, s, t_local, shape.max_tiles, 1, cup, plan, sort_n, units,
                              grid, err));
  } else {
    CPTHD_TRY_CUDA(launch_pdl(attn_fwd_group_kernel<2 * kBlockM>, dim3(static_cast<unsigned>(shape.max_groups)),
                              dim3(2 * kBlockM), sort_bytes, s, t_local, shape.max_tiles, 0, cup, plan, sort_n,
                              units, grid, err));
  }
  return CPTHD_OK;
}

}  // namespace cpthd

extern "C" int thd_causal_attn_plan(const int32_t* q_slice_idx_dev, int64_t t_local, int64_t T,
                                    const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_padded_dev,
                                    int num_docs, int Hq, int Hkv, void* workspace_dev, size_t workspace_bytes,
                                    int32_t* err_dev, cpthd_stream_t stream) {
  using namespace cpthd;
  int st = check_attn_shape(t_local, T, num_docs, Hq, Hkv);
  if (st != CPTHD_OK) return st;
  if (t_local == 0) return CPTHD_OK;
  if (q_slice_idx_dev == nullptr || cu_seqlens_dev == nullptr || num_docs < 1 || T < 1) return CPTHD_ERR_INVALID_ARG;
  st = check_workspace(t_local, Hq, Hkv, 0, workspace_dev, workspace_bytes);
  if (st != CPTHD_OK) return st;
  const int32_t* cup = cu_seqlens_padded_dev ? cu_seqlens_padded_dev : cu_seqlens_dev;
  return launch_plan(index_list(q_slice_idx_dev), t_local, T, cu_seqlens_dev, cup, num_docs, Hq, Hkv, workspace_dev,
                     err_dev, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int thd_causal_attn_plan_partition(int strategy, int64_t T, const int32_t* cu_seqlens_dev,
                                              const int32_t* cu_seqlens_padded_dev, int num_docs, int cp_size,
                                              int rank, int Hq, int Hkv, void* workspace_dev,
                                              size_t workspace_bytes, int32_t* err_dev, cpthd_stream_t stream) {
  using namespace cpthd;
  int64_t t_local = 0;
  int st = cp_local_tokens(strategy, T, cp_size, &t_local);
  if (st != CPTHD_OK) return st;
  if (rank < 0 || rank >= cp_size) return CPTHD_ERR_INVALID_ARG;
  st = check_attn_shape(t_local, T, num_docs, Hq, Hkv);
  if (st != CPTHD_OK) return st;
  if (t_local == 0) return CPTHD_OK;
  if (cu_seqlens_dev == nullptr || num_docs < 1) return CPTHD_ERR_INVALID_ARG;
  st = check_workspace(t_local, Hq, Hkv, 0, workspace_dev, workspace_bytes);
  if (st != CPTHD_OK) return st;
  const int32_t* cup = cu_seqlens_padded_dev ? cu_seqlens_padded_dev : cu_seqlens_dev;
  return launch_plan(index_formula(strategy, cup, num_docs, T, cp_size, rank, t_local), t_local, T, cu_seqlens_dev,
                     cup, num_docs, Hq, Hkv, workspace_dev, err_dev, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int thd_causal_attn_fwd_planned(int64_t t_local, const void* q_dev, const void* k_dev, const void* v_dev,
                                           int64_t T, int Hq, int Hkv, int d, float softmax_scale, void* out_dev,
                                           float* lse_dev, const void* workspace_dev, size_t workspace_bytes,
                                           int32_t* err_dev, cpthd_stream_t stream) {
  using namespace cpthd;
  int st = check_attn_shape(t_local, T, 0, Hq, Hkv);
  if (st != CPTHD_OK) return st;
  if (d != 64 && d != 128) return CPTHD_ERR_UNSUPPORTED;
  if (t_local == 0) return CPTHD_OK;
  if (q_dev == nullptr || k_dev == nullptr || v_dev == nullptr || out_dev == nullptr || lse_dev == nullptr || T < 1)
    return CPTHD_ERR_INVALID_ARG;
  const uintptr_t align = reinterpret_cast<uintptr_t>(q_dev) | reinterpret_cast<uintptr_t>(k_dev) |
                          reinterpret_cast<uintptr_t>(v_dev) | reinterpret_cast<uintptr_t>(out_dev);
  if (align & 15) return CPTHD_ERR_UNSUPPORTED;
  st = check_workspace(t_local, Hq, Hkv, d, workspace_dev, workspace_bytes);
  if (st != CPTHD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(d));
  const float scale_log2 = scale * 1.4426950408889634f;
  const FwdShape shape = fwd_shape(t_local, Hq, Hkv);
  const FwdPlan plan = carve_fwd_plan(const_cast<void*>(workspace_dev), shape);
  float* partial = reinterpret_cast<float*>(static_cast<char*>(const_cast<void*>(workspace_dev)) +
                                            fwd_plan_bytes(shape));
  // the plan ordered its groups exactly when there are more items than SMs
  const bool ordered = plan_ordered(shape, Hq);
  if (d == 128)
    return launch_attn<128>(q_dev, k_dev, v_dev, t_local, T, Hq, Hkv, scale_log2, plan, shape, ordered, partial,
                            out_dev, lse_dev, err_dev, s);
  return launch_attn<64>(q_dev, k_dev, v_dev, t_local, T, Hq, Hkv, scale_log2, plan, shape, ordered, partial,
                         out_dev, lse_dev, err_dev, s);
}

extern "C" int thd_causal_attn_fwd(const int32_t* q_slice_idx_dev, int64_t t_local, const void* q_dev,
                                   const void* k_dev, const void* v_dev, int64_t T,
                                   const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_padded_dev,
                                   int num_docs, int Hq, int Hkv, int d, float softmax_scale, void* out_dev,
                                   float* lse_dev, void* workspace_dev, size_t workspace_bytes,
                                   int32_t* err_dev, cpthd_stream_t stream) {
  using namespace cpthd;
  int st = check_attn_shape(t_local, T, num_docs, Hq, Hkv);
  if (st != CPTHD_OK) return st;
  if (d != 64 && d != 128) return CPTHD_ERR_UNSUPPORTED;
  if (t_local == 0) return CPTHD_OK;
  if (q_slice_idx_dev == nullptr || q_dev == nullptr || k_dev == nullptr || v_dev == nullptr ||
      cu_seqlens_dev == nullptr || out_dev == nullptr || lse_dev == nullptr || num_docs < 1 || T < 1)
    return CPTHD_ERR_INVALID_ARG;
  const uintptr_t align = reinterpret_cast<uintptr_t>(q_dev) | reinterpret_cast<uintptr_t>(k_dev) |
                          reinterpret_cast<uintptr_t>(v_dev) | reinterpret_cast<uintptr_t>(out_dev);
  if (align & 15) return CPTHD_ERR_UNSUPPORTED;
  st = check_workspace(t_local, Hq, Hkv, d, workspace_dev, workspace_bytes);
  if (st != CPTHD_OK) return st;
  st = thd_causal_attn_plan(q_slice_idx_dev, t_local, T, cu_seqlens_dev, cu_seqlens_padded_dev, num_docs, Hq, Hkv,
                            workspace_dev, workspace_bytes, err_dev, stream);
  if (st != CPTHD_OK) return st;
  return thd_causal_attn_fwd_planned(t_local, q_dev, k_dev, v_dev, T, Hq, Hkv, d, softmax_scale, out_dev, lse_dev,
                                     workspace_dev, workspace_bytes, err_dev, stream);
}

#ifdef CPTHD_WAIT_TEST
// Test build only: selects the wait the kernel makes run out (see g_wait_test_mode).
extern "C" CPTHD_API int cpthd_wait_test_mode(int mode) {
  return cudaMemcpyToSymbol(cpthd::g_wait_test_mode, &mode, sizeof(int)) == cudaSuccess ? CPTHD_OK : CPTHD_ERR_CUDA;
}
#endif
