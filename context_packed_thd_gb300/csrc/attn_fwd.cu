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
//  * warp 0      TMA producer: both Q tiles once, then K and V 128-key blocks
//                into a two-stage shared-memory ring (128-byte swizzle, the
//                layout the UMMA shared-memory descriptors read). A stage is
//                refilled once tile B's score barrier reports that the MMAs
//                reading it are done, so the issuer commits only to the two
//                score barriers inside its loop.
//  * warp 1      one lane issues all tcgen05 MMAs: S_A(0), S_B(0), then per
//                block j and tile x = A, B: O_x += P_x(j) V_j, S_x(j+1).
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
//  * warp 2      data relay: per block j, waits until V_j and K_{j+1} have
//                landed and arrives on both tiles' P-ready barriers, so that
//                the issuer waits once per tile and block.
//  * warp 3      idle.
//  * warps 4-7   softmax of tile A, warps 8-11 softmax of tile B: each thread
//                owns one query row (its TMEM lane). It reads S with one
//                tcgen05.ld, masks by the row's key interval [document
//                start, own position] clipped to the end of the block's
//                interval (only on blocks the tile's bounds do not cover
//                fully), keeps the fp32 running max / sum in base 2, rescales
//                O in TMEM only when the max grows by more than 2^8 (exact
//                either way), and writes P back into TMEM. At the end it
//                normalises O into the tile's Q buffer in shared memory and
//                one thread stores the tile with TMA; LSE per row.
// Key blocks start at the group's interval starts (document starts), so
// documents the group does not see are never loaded or multiplied. The grid
// runs the groups in decreasing-cost order. Every wait is bounded; a wait
// that times out makes the CTA drain its copies and MMAs, free TMEM, record
// CPTHD_ERR_TIMEOUT and return.
#include <cuda_bf16.h>

#include "attn_common.cuh"

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
  static constexpr int kBytes = kVOff + kStages * kKV;
  // request at least this much so that one CTA holds an SM (TMEM is taken whole)
  static constexpr int kLaunchBytes = (kBytes + 1024 > 120 * 1024) ? kBytes + 1024 : 120 * 1024;
};

struct AttnParams {
  const int32_t* row_lo;
  const int32_t* row_hi;
  const GroupInfo* group_info;
  const int2* intervals;
  const int32_t* order;
  float* lse;
  long long t_local;
  int Hq;
  int Hkv;
  int head_pairs;  // 1: tiles A/B = heads 2u, 2u+1 of one row tile; 0: row tiles 2g, 2g+1 of one head
  int group_rows;  // 128 with head pairs, 256 with tile pairs
  int max_blocks;  // upper bound on blocks per group, guards malformed metadata
  float scale_log2;
  int32_t* err;
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

  __shared__ uint64_t q_full, k_full[kStages], v_full[kStages];
  __shared__ uint64_t s_full[2], p_full[2], o_final[2], drain[1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;
  __shared__ int epi_abort[2];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Barriers and TMEM are set up before waiting on the kernel this launch
  // depends on: none of it touches global memory.
  if (threadIdx.x == 0) {
    abort_flag = 0;
    epi_abort[0] = epi_abort[1] = 0;
    mbar_init(&q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s_full[x], 1);
      mbar_init(&p_full[x], 5);  // four softmax warps and the data relay
      mbar_init(&o_final[x], 1);
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
  const int item = blockIdx.x;
  // without an order (a grid of one wave) the groups run in index order
  const int group = p.order ? __ldg(p.order + item / units) : item / units;
  const int unit = item % units;
  const int head0 = p.head_pairs ? 2 * unit : unit;
  const int kvh = head0 / (p.Hq / p.Hkv);
  const GroupInfo gi = p.group_info[group];
  const int n_blocks = min(max(gi.n_blocks, 0), p.max_blocks);
  const int2* group_iv = p.intervals + static_cast<long long>(group) * p.group_rows;
  const int n_iv = min(max(gi.n_intervals, 0), p.group_rows);
  const long long group_row0 = static_cast<long long>(group) * p.group_rows;

  if (warp < 4) {
   setmaxnreg_dec<kRegsControl>();
   if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_blocks > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&q_full, 2 * L::kQ);
      for (int x = 0; x < 2; ++x) {
        const int qh = p.head_pairs ? head0 + x : head0;
        const int qrow = static_cast<int>(group_row0) + (p.head_pairs ? 0 : x * kBlockM);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sQ + x * L::kQ + c * L::kChunk, &tm_q, &q_full, c * 64, qh, qrow);
      }
      BlockCursor cur;
      cur.init(group_iv, n_iv);
      int issued = 0;
      for (int i = 0; i < n_blocks; ++i) {
        const int st = i & 1;
        // Stages are released through tile B's score barrier: its phase k
        // completes when every MMA issued up to S_B(k) is done (one thread
        // issues them all, tile B last), so phase i - 2 frees K_{i-2} and
        // phase i - 1 frees V_{i-2}. Each phase is waited for once, in order
        // (phase 0 before K_2, then phase i - 1 before V_i; K_i for i >= 3
        // needs phase i - 2, already seen before V_{i-1}). A phase can only
        // complete after loads this thread issues just before waiting for
        // the phase ahead of it, so the barrier is never two phases ahead
        // of a wait and the parity is unambiguous.
        if (i == kStages && !mbar_wait(&s_full[1], 0, &abort_flag)) break;
        mbar_arrive_expect_tx(&k_full[st], L::kKV);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sK + st * L::kKV + c * L::kChunk, &tm_k, &k_full[st], c * 64, kvh, cur.start);
        issued = 2 * i + 1;
        if (i >= kStages && !mbar_wait(&s_full[1], (i - 1) & 1, &abort_flag)) break;
        mbar_arrive_expect_tx(&v_full[st], L::kKV);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sV + st * L::kKV + c * L::kChunk, &tm_v, &v_full[st], c * 64, kvh, cur.start);
        issued = 2 * i + 2;
        cur.next();
      }
      if (abort_flag) {
        // let every copy still in flight land before the CTA exits
        mbar_wait_drain(&q_full, 0);
        for (int x = (issued > 4 ? issued - 4 : 0); x < issued; ++x) {
          const int i = x >> 1, st = i & 1;
          mbar_wait_drain((x & 1) ? &v_full[st] : &k_full[st], (i >> 1) & 1);
        }
      }
    }
   } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // One thread issues both tiles' MMAs, tile A's batch before tile B's.
    // Issued from one thread they run in that order, so tile B's scores
    // arrive a batch after tile A's and the two tiles settle into a
    // staggered schedule: one tile's softmax runs under the other tile's
    // MMAs. (Two issuing threads started together interleave their MMAs on
    // the tensor pipe, both tiles finish together, and their softmaxes then
    // leave the tensor pipe idle: a lockstep that a single issuer avoids.)
    if (lane == 0 && n_blocks > 0) {
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
      auto issue_pv = [&](int j, int x) {  // O_x += P_x V_j, P_x read from TMEM
        const uint32_t t_s = tmem + x * kBlockN;
        const uint32_t t_o = tmem + 256 + x * D;
        const uint32_t vb = v_lo + (((j & 1) * L::kKV) >> 4);
        const uint32_t acc0 = (j > 0) ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          umma_ts_w(t_o, t_s + kk * 8, vb + ((kk * 16 * 128) >> 4), v_hi, kIdescO, kk > 0 ? 1u : acc0);
      };
      int finals = 0;
      bool ok = mbar_wait(&q_full, 0, &abort_flag) && mbar_wait(&k_full[0], 0, &abort_flag);
      if (ok) {
        tc_fence_after_sync();
        issue_s(0, 0);
        umma_commit(&s_full[0]);
        issue_s(0, 1);
        umma_commit(&s_full[1]);
      }
      for (int j = 0; ok && j < n_blocks; ++j) {
        const bool more = (j + 1 < n_blocks);
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          // P_x(j) is ready, and (through the relay's arrival) V_j and K_{j+1}
          // have landed
          if (!mbar_wait(&p_full[x], j & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after_sync();
          issue_pv(j, x);
          if (more) {
            issue_s(j + 1, x);
            umma_commit(&s_full[x]);  // also reports O_x += P_x(j) V_j done
          } else {
            umma_commit(&o_final[x]);  // tile x's epilogue need not wait for the other tile
            finals |= 1 << x;
          }
        }
      }
      // a tile whose final commit did not happen (no block, or an abort)
      if (!(finals & 1)) umma_commit(&o_final[0]);
      if (!(finals & 2)) umma_commit(&o_final[1]);
      umma_commit(&drain[0]);
      mbar_wait_drain(&drain[0], 0);
    }
   } else if (warp == 2) {
    // ------------------------------------------------------------ data relay
    // Waits, per block j, until V_j and K_{j+1} have landed and then arrives
    // on both tiles' p_full, so that the MMA issuer (the busiest thread of
    // the CTA) needs a single wait per tile and block. Before arriving for
    // block j it waits for both p_full phases of block j - 1 to complete, so
    // that an early arrival never counts toward the previous phase.
    if (lane == 0) {
      for (int j = 0; j < n_blocks; ++j) {
        if (j > 0 && !(mbar_wait(&p_full[0], (j - 1) & 1, &abort_flag) &&
                       mbar_wait(&p_full[1], (j - 1) & 1, &abort_flag)))
          break;
        if (!mbar_wait(&v_full[j & 1], (j >> 1) & 1, &abort_flag)) break;
        if (j + 1 < n_blocks && !mbar_wait(&k_full[(j + 1) & 1], ((j + 1) >> 1) & 1, &abort_flag)) break;
#ifdef CPTHD_WAIT_TEST
        // Test build only: block 1's arrivals are withheld, so the waits for
        // P(1) can never complete and must run out into the abort path.
        if (j == 1) continue;
#endif
        mbar_arrive(&p_full[0]);
        mbar_arrive(&p_full[1]);
      }
    }
   }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int x = (warp - 4) >> 2;  // tile of this warpgroup
    const int quarter = warp & 3;   // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;
    const long long grow = group_row0 + (p.head_pairs ? 0 : x * kBlockM) + r;
    const int qh = p.head_pairs ? head0 + x : head0;
    const int lo = p.row_lo[grow];
    const int hi = p.row_hi[grow];
    const bool valid = (grow < p.t_local) && (lo <= hi);
    const int tmax_lo = gi.max_lo[x], tmin_hi = gi.min_hi[x];
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + x * kBlockN;
    const uint32_t t_o = tmem + lane_off + 256 + x * D;
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // running max of scale*log2(e)*s
    float l = 0.f;
    BlockCursor cur;
    cur.init(group_iv, n_iv);
    bool ok = true;
    for (int j = 0; j < n_blocks; ++j) {
      // a block never reaches past its interval's end: the next interval may
      // start inside it, and its keys must be counted there only
      const int kstart = cur.start;
      const int kend = cur.end;
      cur.next();
      if (!warp_wait(&s_full[x], j & 1, &abort_flag)) { ok = false; break; }
      tc_fence_after_sync();
      uint32_t sr[kBlockN];
      tmem_ld128(t_s, sr);
      tmem_ld_wait128(sr);
      const bool full = (kstart >= tmax_lo) && (kstart + kBlockN - 1 <= min(tmin_hi, kend));
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
        // metadata kernel has already reported; such a row uses no key of
        // the block, so it never reaches a key before its own start.
        if (c_lo > 0 && c_lo <= c_hi) record_error(p.err, CPTHD_ERR_BAD_OFFSETS, grow);
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
            fma2(a0, a1, __uint_as_float(sr[64 * h2 + 2 * c]), __uint_as_float(sr[64 * h2 + 2 * c + 1]), sl2, -mref);
            const float e0 = ex2(a0);
            const float e1 = ex2(a1);
            add2(rs[2 * (c & 1)], rs[2 * (c & 1) + 1], e0, e1);
            pk[c] = pack_bf16x2(e0, e1);
          }
        }
        tmem_st32(t_s + 32 * h2, pk);
      }
      l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      if (__any_sync(0xffffffffu, grow_o)) {
        // O_x holds P_x(j-1) V_{j-1} (complete before S_x(j) was reported) and
        // nothing newer: rescale it before O_x += P_x(j) V_j is issued
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
      if (lane == 0) mbar_arrive(&p_full[x]);
    }
    // ---------------------------------------------------------- epilogue
    // O / l in bf16 goes into this tile's Q buffer (free once o_final[x] is
    // reported: the last MMA reading it is done), in the 128-byte swizzle of
    // the output's tensor map, and one thread of the warpgroup stores the
    // tile with TMA (rows past the slice are not written). Every warp of the
    // warpgroup reaches the barrier; an aborted one only marks the tile.
    if (ok && n_blocks > 0) ok = warp_wait(&o_final[x], 0, &abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after_sync();
    uint8_t* stile = sQ + x * L::kQ;
    if (ok) {
      const float inv = (valid && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t rr[32];
        if (n_blocks > 0) {
          tmem_ld32(t_o + c * 32, rr);
          tmem_ld_wait(rr);
        }
        uint32_t ob[16];
#pragma unroll
        for (int q = 0; q < 16; ++q)
          ob[q] = (valid && n_blocks > 0)
                      ? pack_bf16x2(__uint_as_float(rr[2 * q]) * inv, __uint_as_float(rr[2 * q + 1]) * inv)
                      : 0u;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int u = 4 * c + q4;  // 16-byte unit of the row; 8 units per 64-column panel
          uint8_t* dst = stile + (u >> 3) * L::kChunk + r * 128 + (((u & 7) ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = make_uint4(ob[4 * q4], ob[4 * q4 + 1], ob[4 * q4 + 2], ob[4 * q4 + 3]);
        }
      }
      if (grow < p.t_local)
        p.lse[static_cast<long long>(qh) * p.t_local + grow] =
            (valid && l > 0.f) ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
      fence_proxy_async_smem();
    } else {
      epi_abort[x] = 1;
    }
    named_bar_sync(1 + x, 128);
    const long long tile_row0 = group_row0 + (p.head_pairs ? 0 : x * kBlockM);
    if (r == 0 && !epi_abort[x] && tile_row0 < p.t_local) {
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c)
        tma_store_3d(&tm_o, stile + c * L::kChunk, c * 64, qh, static_cast<int>(tile_row0));
      bulk_commit_group();
      bulk_wait_group_read_all();
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (abort_flag && threadIdx.x == 0) record_error(p.err, CPTHD_ERR_TIMEOUT, item);
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <int D>
static int launch_attn(const void* q, const void* k, const void* v, long long t_local, long long T, int Hq, int Hkv,
                       float scale_log2, const AttnWorkspace& ws, long long ngroups, int group_rows, bool ordered,
                       void* out,
                       float* lse, int32_t* err, cudaStream_t s) {
  EncodeTiledFn enc = get_encode_tiled();
  if (enc == nullptr) return CPTHD_ERR_CUDA;
  CUtensorMap mq, mk, mv, mo;
  if (!make_rows_heads_map(enc, &mq, q, t_local, Hq, D) || !make_rows_heads_map(enc, &mk, k, T, Hkv, D) ||
      !make_rows_heads_map(enc, &mv, v, T, Hkv, D) || !make_rows_heads_map(enc, &mo, out, t_local, Hq, D))
    return CPTHD_ERR_UNSUPPORTED;
  AttnParams p;
  p.row_lo = ws.row_lo;
  p.row_hi = ws.row_hi;
  p.group_info = ws.group_info;
  p.intervals = ws.intervals;
  p.order = ordered ? ws.order : nullptr;
  p.lse = lse;
  p.t_local = t_local;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.head_pairs = (group_rows == kBlockM) ? 1 : 0;
  p.group_rows = group_rows;
  p.max_blocks = static_cast<int>((T + kBlockN - 1) / kBlockN + group_rows);
  p.scale_log2 = scale_log2;
  p.err = err;
  const int smem = AttnSmem<D>::kLaunchBytes;
  CPTHD_TRY_CUDA(cudaFuncSetAttribute(attn_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  const long long items = ngroups * (p.head_pairs ? Hq / 2 : Hq);
  if (items > INT32_MAX) return CPTHD_ERR_UNSUPPORTED;
  CPTHD_TRY_CUDA(launch_pdl(attn_fwd_tc_kernel<D>, dim3(static_cast<unsigned>(items)), dim3(kAttnThreads), smem, s,
                            mq, mk, mv, mo, p));
  return CPTHD_OK;
}

}  // namespace cpthd

extern "C" int thd_causal_attn_workspace_size(int64_t t_local, int Hq, int Hkv, int d, size_t* bytes_host) {
  if (bytes_host == nullptr || t_local < 0 || Hq < 1 || Hkv < 1) return CPTHD_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return CPTHD_ERR_UNSUPPORTED;
  (void)d;
  const int rows = cpthd::group_rows_for(Hq, Hkv);
  const long long ngroups = (t_local + rows - 1) / rows;
  *bytes_host = cpthd::attn_workspace_bytes(ngroups, rows);
  return CPTHD_OK;
}

namespace cpthd {

static int check_workspace(int64_t t_local, int Hq, int Hkv, const void* workspace_dev, size_t workspace_bytes) {
  const int rows = group_rows_for(Hq, Hkv);
  const long long ngroups = (t_local + rows - 1) / rows;
  if (workspace_dev == nullptr || workspace_bytes < attn_workspace_bytes(ngroups, rows) ||
      (reinterpret_cast<uintptr_t>(workspace_dev) & 255))
    return CPTHD_ERR_WORKSPACE;
  return CPTHD_OK;
}

}  // namespace cpthd

namespace cpthd {

// Metadata of the slice's row groups (and, past one wave, their order) into
// the workspace; shape and workspace already checked.
static int launch_plan(const IndexGen& slots, long long t_local, long long T, const int32_t* cu,
                       const int32_t* cup, int num_docs, int Hq, int Hkv, void* workspace, int32_t* err,
                       cudaStream_t s) {
  const int rows = group_rows_for(Hq, Hkv);
  const long long ngroups = (t_local + rows - 1) / rows;
  AttnWorkspace ws = carve_workspace(workspace, ngroups, rows);
  if (rows == kBlockM) {
    CPTHD_TRY_CUDA(launch_pdl(attn_group_meta_kernel<kBlockM>, dim3(static_cast<unsigned>(ngroups)), dim3(kBlockM), 0,
                              s, slots, t_local, cu, cup, num_docs, T, ws, err));
  } else {
    CPTHD_TRY_CUDA(launch_pdl(attn_group_meta_kernel<2 * kBlockM>, dim3(static_cast<unsigned>(ngroups)),
                              dim3(2 * kBlockM), 0, s, slots, t_local, cu, cup, num_docs, T, ws, err));
  }
  // The longest groups go first when the grid needs more than one wave (one
  // CTA per SM); within a single wave the order makes no difference and the
  // ordering launch is skipped.
  const long long items = ngroups * ((rows == kBlockM) ? Hq / 2 : Hq);
  if (items > sm_count())
    CPTHD_TRY_CUDA(launch_pdl(attn_group_order_kernel, dim3(1), dim3(1024), 0, s, static_cast<int>(ngroups), ws));
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
  st = check_workspace(t_local, Hq, Hkv, workspace_dev, workspace_bytes);
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
  st = check_workspace(t_local, Hq, Hkv, workspace_dev, workspace_bytes);
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
  st = check_workspace(t_local, Hq, Hkv, workspace_dev, workspace_bytes);
  if (st != CPTHD_OK) return st;
  const int rows = group_rows_for(Hq, Hkv);
  const long long ngroups = (t_local + rows - 1) / rows;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(d));
  const float scale_log2 = scale * 1.4426950408889634f;
  AttnWorkspace ws = carve_workspace(const_cast<void*>(workspace_dev), ngroups, rows);
  // the plan launched the group order exactly when the grid exceeds a wave
  const long long items = ngroups * ((rows == kBlockM) ? Hq / 2 : Hq);
  const bool ordered = items > sm_count();
  if (d == 128)
    return launch_attn<128>(q_dev, k_dev, v_dev, t_local, T, Hq, Hkv, scale_log2, ws, ngroups, rows, ordered, out_dev,
                            lse_dev, err_dev, s);
  return launch_attn<64>(q_dev, k_dev, v_dev, t_local, T, Hq, Hkv, scale_log2, ws, ngroups, rows, ordered, out_dev,
                         lse_dev, err_dev, s);
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
  st = check_workspace(t_local, Hq, Hkv, workspace_dev, workspace_bytes);
  if (st != CPTHD_OK) return st;
  st = thd_causal_attn_plan(q_slice_idx_dev, t_local, T, cu_seqlens_dev, cu_seqlens_padded_dev, num_docs, Hq, Hkv,
                            workspace_dev, workspace_bytes, err_dev, stream);
  if (st != CPTHD_OK) return st;
  return thd_causal_attn_fwd_planned(t_local, q_dev, k_dev, v_dev, T, Hq, Hkv, d, softmax_scale, out_dev, lse_dev,
                                     workspace_dev, workspace_bytes, err_dev, stream);
}
